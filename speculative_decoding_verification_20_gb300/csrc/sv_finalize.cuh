// sv_finalize.cuh -- per-sequence finalisation and unit completion, shared by the
// streaming and dense paths.
#pragma once

#include "sv_internal.cuh"

namespace sv {

// Called by every thread of the block that completed the last unit of
// sequence b.  Implements the truncation of Algorithm 1 (review page of
// "Fast Inference from Transformers via Speculative Decoding", step 3):
// n = index of the first rejected draft token (gamma_b if none), output
// x_1..x_n followed by the token drawn at position n+1.
__device__ __forceinline__ void finalize_sequence(const Args& a, int b) {
    __shared__ int s_n;
    const SeqInfo si = a.seq[b];
    const int G = a.G, gamma = si.gamma;
    const uint32_t st = __ldcg(&a.seq_status[b]);
    if (threadIdx.x == 0) {
        int n = gamma;
        if (!st)
            for (int i = 0; i < gamma; ++i)
                if (__ldcg(&a.unit_acc[(size_t)b * G + i]) == 0) {
                    n = i;
                    break;
                }
        s_n = n;
        a.accepted_len[b] = st ? 0 : n;
        if (a.row_status) a.row_status[b] = st;
    }
    __syncthreads();
    const int n = s_n;
    for (int j = threadIdx.x; j <= G; j += blockDim.x) {
        int tok = -1;
        if (!st) {
            if (j < n)
                tok = a.draft_tokens[(size_t)b * G + j];
            else if (j == n)
                tok = __ldcg(&a.unit_tok[(size_t)b * (G + 1) + n]);
        }
        a.out_tokens[(size_t)b * (G + 1) + j] = tok;
    }
    if (st) {  // a data problem found on the device: the defaults of an invalid sequence
        for (int i = threadIdx.x; i < G; i += blockDim.x) {
            if (a.alpha) a.alpha[(size_t)b * G + i] = 0.0f;
            if (a.pos_accept) a.pos_accept[(size_t)b * G + i] = -1;
        }
        if (a.pos_token)
            for (int j = threadIdx.x; j <= G; j += blockDim.x) a.pos_token[(size_t)b * (G + 1) + j] = -1;
        const size_t V = (size_t)a.V;
        if (a.p_out)
            for (size_t i = threadIdx.x; i < (size_t)(G + 1) * V; i += blockDim.x)
                a.p_out[(size_t)b * (G + 1) * V + i] = 0.0f;
        if (a.q_out)
            for (size_t i = threadIdx.x; i < (size_t)G * V; i += blockDim.x) a.q_out[(size_t)b * G * V + i] = 0.0f;
    }
}

// Count one finished unit of sequence b; the block that finishes the last
// unit finalises the sequence.  Every thread of the block calls this after
// the unit's results are written.
__device__ __forceinline__ void unit_finished(const Args& a, int b) {
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const int units = a.seq[b].gamma + 1;
        s_last = (atomicAdd(&a.seq_done[b], 1u) == (uint32_t)(units - 1));
    }
    __syncthreads();
    if (s_last) {
        __threadfence();
        finalize_sequence(a, b);
    }
    __syncthreads();
}

// Warp versions of the two functions above, for kernels where one warp owns
// a unit.  The first rejection is found with a ballot over 32 positions at a
// time and the lowest set lane.
static __device__ __noinline__ void finalize_sequence_warp(const Args& a, int b, int lane) {
    const SeqInfo si = a.seq[b];
    const int G = a.G, gamma = si.gamma;
    const uint32_t st = __ldcg(&a.seq_status[b]);
    int n = gamma;
    if (!st) {
        for (int i0 = 0; i0 < gamma; i0 += 32) {
            const int i = i0 + lane;
            const bool rejected = i < gamma && __ldcg(&a.unit_acc[(size_t)b * G + i]) == 0;
            const unsigned m = __ballot_sync(0xFFFFFFFFu, rejected);
            if (m) {
                n = i0 + __ffs(m) - 1;
                break;
            }
        }
    }
    if (lane == 0) {
        a.accepted_len[b] = st ? 0 : n;
        if (a.row_status) a.row_status[b] = st;
    }
    for (int j = lane; j <= G; j += 32) {
        int tok = -1;
        if (!st) {
            if (j < n)
                tok = a.draft_tokens[(size_t)b * G + j];
            else if (j == n)
                tok = __ldcg(&a.unit_tok[(size_t)b * (G + 1) + n]);
        }
        a.out_tokens[(size_t)b * (G + 1) + j] = tok;
    }
    if (st) {
        for (int i = lane; i < G; i += 32) {
            if (a.alpha) a.alpha[(size_t)b * G + i] = 0.0f;
            if (a.pos_accept) a.pos_accept[(size_t)b * G + i] = -1;
        }
        if (a.pos_token)
            for (int j = lane; j <= G; j += 32) a.pos_token[(size_t)b * (G + 1) + j] = -1;
        const size_t V = (size_t)a.V;
        if (a.p_out)
            for (size_t i = lane; i < (size_t)(G + 1) * V; i += 32) a.p_out[(size_t)b * (G + 1) * V + i] = 0.0f;
        if (a.q_out)
            for (size_t i = lane; i < (size_t)G * V; i += 32) a.q_out[(size_t)b * G * V + i] = 0.0f;
    }
}

__device__ __forceinline__ void unit_finished_warp(const Args& a, int b, int lane) {
    __threadfence();
    __syncwarp();
    int last = 0;
    if (lane == 0) last = atomicAdd(&a.seq_done[b], 1u) == (uint32_t)a.seq[b].gamma;  // gamma + 1 units
    if (__shfl_sync(0xFFFFFFFFu, last, 0)) {
        __threadfence();
        finalize_sequence_warp(a, b, lane);
    }
    __syncwarp();
}

}  // namespace sv
