// sv_stream.cu -- streaming top-k path (greedy and 1 <= top_k <= 256 sequences).
//
// Normalisation with top-k ("Fast Inference from Transformers via Speculative
// Decoding" review page, section "Method: Speculative Decoding": top-k and
// argmax are standard sampling from an adjusted distribution) only ever needs
// the k largest logits of a row: the softmax normaliser of the whole
// vocabulary cancels when the kept set is renormalised.  So a row is streamed
// from HBM exactly once, in 64 KB pieces, and each piece hands at most
// kCandCap (logit key, token id) candidates to its unit; no exponential is
// evaluated on the bulk of the vocabulary.
//
// Piece (one CTA, 256 threads x 16 loads of 16 bytes, all in flight at once):
//   1. ordered integer keys of the logits, per-thread maximum;
//   2. theta = k-th largest per-thread maximum (bitwise search with
//      __syncthreads_count): at least k elements of the piece are >= theta,
//      so every element of the piece's top-k is >= theta;
//   3. elements >= theta are appended to the piece's candidate list
//      (warp-aggregated atomics); rare overflow falls back to an exact
//      k-th-key search with lowest-id tie breaking.
// The last piece of a unit (atomic counter) merges the candidate lists of the
// unit's target and draft rows (exact top-k by (logit desc, id asc)), then one
// warp does in fp64: softmax over the kept logits, top-p, alpha, the
// acceptance test and the residual / bonus draw (inverse CDF by token id).
#include <cooperative_groups.h>

#include "sv_finalize.cuh"

namespace sv {

template <typename TIn>
struct StreamCfg {
    static constexpr int NT = kStreamThreads;
    static constexpr int L = kStreamLoads;
    static constexpr int VEC = 16 / (int)sizeof(TIn);
    static constexpr int EPT = L * VEC;
    static constexpr int PE = NT * EPT;
    static constexpr int KB = 8 * (int)sizeof(TIn);  // key bits
};

// key of element j of a 16-byte vector
template <typename TIn>
__device__ __forceinline__ uint32_t elem_bits(const uint4& v, int j) {
    const uint32_t w = (j / (int)(4 / sizeof(TIn)) == 0) ? v.x : (j / (int)(4 / sizeof(TIn)) == 1) ? v.y
                       : (j / (int)(4 / sizeof(TIn)) == 2) ? v.z : v.w;
    if (sizeof(TIn) == 4) return w;
    return (j & 1) ? (w >> 16) : (w & 0xFFFFu);
}
template <typename TIn>
__device__ __forceinline__ uint32_t to_key(uint32_t bits) {
    return sizeof(TIn) == 4 ? okey32(bits) : okey16(bits);
}
template <typename TIn>
__device__ __forceinline__ bool is_bad(uint32_t bits) {
    return sizeof(TIn) == 4 ? bad32(bits) : bad16(bits);
}
template <typename TIn>
__device__ __forceinline__ double key_to_value(uint32_t k) {
    return sizeof(TIn) == 4 ? (double)key_value32(k) : (double)key_value16(k);
}

__device__ __forceinline__ int block_sum_int(int v, int* s_red) {
    v = warp_sum(v);
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) s_red[wid] = v;
    __syncthreads();
    int tot = 0;
#pragma unroll
    for (int w = 0; w < kStreamThreads / 32; ++w) tot += s_red[w];
    return tot;
}

// exclusive scan of an int over the block (thread order); returns the prefix and the total
__device__ __forceinline__ int block_excl_scan_int(int v, int* s_red, int* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
    }
    __syncthreads();
    if (lane == 31) s_red[wid] = x;
    __syncthreads();
    int before = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kStreamThreads / 32; ++w) {
        const int t = s_red[w];
        before += (w < wid) ? t : 0;
        tot += t;
    }
    *total = tot;
    return before + x - v;
}

// Bitonic sort, descending, of n (power of two) 64-bit keys in shared memory.
__device__ __forceinline__ void block_sort_desc(unsigned long long* s, int n) {
    for (int k2 = 2; k2 <= n; k2 <<= 1) {
        for (int j = k2 >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < n; i += blockDim.x) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const unsigned long long x = s[i], y = s[ixj];
                    const bool desc = ((i & k2) == 0);
                    if (desc ? (x < y) : (x > y)) {
                        s[i] = y;
                        s[ixj] = x;
                    }
                }
            }
            __syncthreads();
        }
    }
}

__device__ __forceinline__ int next_pow2(int n) {
    int p = 1;
    while (p < n) p <<= 1;
    return p;
}

// composite sort key: logit key descending, then token id ascending
__device__ __forceinline__ unsigned long long composite(uint32_t key, uint32_t id) {
    return ((unsigned long long)key << 32) | (unsigned long long)(~id);
}
__device__ __forceinline__ uint32_t comp_key(unsigned long long c) { return (uint32_t)(c >> 32); }
__device__ __forceinline__ int comp_id(unsigned long long c) { return (int)(~(uint32_t)c); }

struct StreamSmem {
    unsigned long long sort[kSortCap];
    unsigned long long top[2][kStreamMaxK];  // exact top-k of target (0) and draft (1) rows
    double prob[2][kStreamMaxK];
    double resid[kStreamMaxK];
    int rid[kStreamMaxK];
    int red[32];
    int cnt;
    int last;
};

// Exact top-k (sorted) of one row from its pieces' candidate lists.
template <typename TIn>
__device__ void merge_row_topk(const Args& a, uint32_t row_slot, int k, unsigned long long* out, StreamSmem& sm) {
    const int ppr = a.ppr;
    int total = 0;
    for (int j = 0; j < ppr; ++j) total += (int)__ldcg(&a.cand_cnt[(size_t)row_slot * ppr + j]);
    if (total <= kSortCap) {
        const int n2 = next_pow2(total < 2 ? 2 : total);
        int off = 0;
        for (int j = 0; j < ppr; ++j) {
            const size_t piece = (size_t)row_slot * ppr + j;
            const int c = (int)__ldcg(&a.cand_cnt[piece]);
            for (int i = threadIdx.x; i < c; i += blockDim.x) {
                const uint2 e = __ldcg(&a.cand[piece * kCandCap + i]);
                sm.sort[off + i] = composite(e.x, e.y);
            }
            off += c;
        }
        for (int i = total + threadIdx.x; i < n2; i += blockDim.x) sm.sort[i] = 0ull;
        __syncthreads();
        block_sort_desc(sm.sort, n2);
        for (int i = threadIdx.x; i < k; i += blockDim.x) out[i] = sm.sort[i];
        __syncthreads();
        return;
    }
    // Many candidates (adversarial inputs): k-th largest composite by a bitwise
    // search over the candidates in global memory, then sort the k survivors.
    unsigned long long theta = 0ull;
    for (int bit = 63; bit >= 0; --bit) {
        const unsigned long long c = theta | (1ull << bit);
        int cnt = 0;
        for (int j = 0; j < ppr; ++j) {
            const size_t piece = (size_t)row_slot * ppr + j;
            const int n = (int)__ldcg(&a.cand_cnt[piece]);
            for (int i = threadIdx.x; i < n; i += blockDim.x) {
                const uint2 e = __ldcg(&a.cand[piece * kCandCap + i]);
                cnt += composite(e.x, e.y) >= c;
            }
        }
        if (block_sum_int(cnt, sm.red) >= k) theta = c;
    }
    if (threadIdx.x == 0) sm.cnt = 0;
    __syncthreads();
    for (int j = 0; j < ppr; ++j) {
        const size_t piece = (size_t)row_slot * ppr + j;
        const int n = (int)__ldcg(&a.cand_cnt[piece]);
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            const uint2 e = __ldcg(&a.cand[piece * kCandCap + i]);
            const unsigned long long c = composite(e.x, e.y);
            if (c >= theta) sm.sort[atomicAdd(&sm.cnt, 1)] = c;
        }
    }
    __syncthreads();
    const int n2 = next_pow2(k < 2 ? 2 : k);
    for (int i = k + threadIdx.x; i < n2; i += blockDim.x) sm.sort[i] = 0ull;
    __syncthreads();
    block_sort_desc(sm.sort, n2);
    for (int i = threadIdx.x; i < k; i += blockDim.x) out[i] = sm.sort[i];
    __syncthreads();
}

// fp64 normalisation of one sorted kept list by warp 0: softmax over the kept
// logits at temperature T (one-hot if T == 0), then top-p.  prob[j] for j < k.
template <typename TIn>
__device__ void normalise_kept(const unsigned long long* top, int k, float Tf, float Pf, double* prob) {
    const int lane = threadIdx.x & 31;
    const double T = (double)Tf, P = (double)Pf;
    if (Tf == 0.0f) {
        for (int j = lane; j < k; j += 32) prob[j] = (j == 0) ? 1.0 : 0.0;
        __syncwarp();
        return;
    }
    const double vmax = key_to_value<TIn>(comp_key(top[0]));
    double s = 0.0;
    for (int j = lane; j < k; j += 32) {
        const double v = key_to_value<TIn>(comp_key(top[j]));
        const double w = exp((v - vmax) / T);
        prob[j] = w;
        s += w;
    }
    s = warp_sum(s);
    for (int j = lane; j < k; j += 32) prob[j] /= s;
    __syncwarp();
    if (P < 1.0) {  // shortest prefix (prob desc, id asc) whose mass reaches P, crossing token kept
        double carry = 0.0;
        int keep = k;
        for (int c0 = 0; c0 < k; c0 += 32) {
            const int j = c0 + lane;
            double x = (j < k) ? prob[j] : 0.0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double y = __shfl_up_sync(0xFFFFFFFFu, x, o);
                if (lane >= o) x += y;
            }
            const double cum = carry + x;
            const unsigned hit = __ballot_sync(0xFFFFFFFFu, j < k && cum >= P);
            if (hit) {
                keep = c0 + __ffs(hit);  // index of the crossing token + 1
                break;
            }
            carry += __shfl_sync(0xFFFFFFFFu, x, 31);
        }
        double s2 = 0.0;
        for (int j = lane; j < k; j += 32) {
            if (j >= keep) prob[j] = 0.0;
            s2 += prob[j];
        }
        s2 = warp_sum(s2);
        __syncwarp();
        for (int j = lane; j < keep; j += 32) prob[j] /= s2;
    }
    __syncwarp();
}

template <typename TIn>
__device__ __noinline__ void combine_unit(const Args& a, int b, int unit, const SeqInfo& si, StreamSmem& sm) {
    const int G = a.G, k = si.k;
    const bool pair = unit < si.gamma;
    const uint32_t slot_t = si.row_off + (uint32_t)unit;
    const uint32_t slot_d = si.row_off + (uint32_t)si.gamma + 1u + (uint32_t)unit;
    merge_row_topk<TIn>(a, slot_t, k, sm.top[0], sm);
    if (pair) merge_row_topk<TIn>(a, slot_d, k, sm.top[1], sm);

    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        normalise_kept<TIn>(sm.top[0], k, si.T, si.P, sm.prob[0]);
        if (pair) normalise_kept<TIn>(sm.top[1], k, si.T, si.P, sm.prob[1]);
        // No finite logit in a row: its maximum key is the key of -inf.
        const uint32_t ninf_key = (sizeof(TIn) == 4) ? okey32(0xFF800000u) : okey16(0xFF80u);
        const bool dead = comp_key(sm.top[0][0]) <= ninf_key || (pair && comp_key(sm.top[1][0]) <= ninf_key);
        if (dead && lane == 0) atomicOr(&a.seq_status[b], SV_ROW_NONFINITE);

        // q at each kept target id (0 when the id is not kept in the draft row);
        // alpha_i = sum_x min(p, q) over the ids kept in both rows
        double alpha = 0.0;
        for (int j = lane; j < k; j += 32) {
            const int id = comp_id(sm.top[0][j]);
            double q = 0.0;
            if (pair)
                for (int e = 0; e < k; ++e)
                    if (comp_id(sm.top[1][e]) == id) q = sm.prob[1][e];
            const double p = sm.prob[0][j];
            alpha += fmin(p, q);
            sm.resid[j] = pair ? fmax(p - q, 0.0) : p;  // bonus: q_{gamma+1} := 0
        }
        alpha = warp_sum(alpha);
        __syncwarp();

        // acceptance test u * q(x) < p(x) at this position
        int accept = 0;
        if (pair) {
            const int x = a.draft_tokens[(size_t)b * G + unit];
            double px = 0.0, qx = 0.0;
            for (int j = lane; j < k; j += 32) {
                if (comp_id(sm.top[0][j]) == x) px = sm.prob[0][j];
                if (comp_id(sm.top[1][j]) == x) qx = sm.prob[1][j];
            }
            px = warp_sum(px);
            qx = warp_sum(qx);
            const double u = uniform01(a.seed, (uint32_t)b, (uint32_t)(unit + 1), 0u);
            accept = (u * qx < px) ? 1 : 0;
        }

        // residual (or bonus) draw: inverse CDF in ascending token id
        double Z = 0.0;
        for (int j = lane; j < k; j += 32) Z += sm.resid[j];
        Z = warp_sum(Z);
        if (!(Z > 0.0)) {  // p <= q everywhere: fall back to p
            Z = 0.0;
            for (int j = lane; j < k; j += 32) {
                sm.resid[j] = sm.prob[0][j];
                Z += sm.resid[j];
            }
            Z = warp_sum(Z);
        }
        __syncwarp();
        // rank every kept target entry by token id (ids are distinct in a row)
        double rr[kStreamMaxK / 32];
        int rank[kStreamMaxK / 32];
#pragma unroll
        for (int m = 0; m < kStreamMaxK / 32; ++m) {
            const int j = lane + 32 * m;
            rank[m] = -1;
            if (j < k) {
                const int id = comp_id(sm.top[0][j]);
                int r = 0;
                for (int e = 0; e < k; ++e) r += comp_id(sm.top[0][e]) < id;
                rank[m] = r;
                rr[m] = sm.resid[j];
            }
        }
        __syncwarp();
#pragma unroll
        for (int m = 0; m < kStreamMaxK / 32; ++m) {
            const int j = lane + 32 * m;
            if (j < k) {
                sm.resid[rank[m]] = rr[m];
                sm.rid[rank[m]] = comp_id(sm.top[0][j]);
            }
        }
        __syncwarp();
        const double v = uniform01(a.seed, (uint32_t)b, (uint32_t)(unit + 1), 1u) * Z;
        int token = -1, last_pos = -1;
        double carry = 0.0;
        for (int c0 = 0; c0 < k && token < 0; c0 += 32) {
            const int j = c0 + lane;
            const double r = (j < k) ? sm.resid[j] : 0.0;
            double x = r;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const double y = __shfl_up_sync(0xFFFFFFFFu, x, o);
                if (lane >= o) x += y;
            }
            const unsigned pos = __ballot_sync(0xFFFFFFFFu, j < k && r > 0.0);
            if (pos) last_pos = c0 + 31 - __clz(pos);
            const unsigned hit = __ballot_sync(0xFFFFFFFFu, j < k && r > 0.0 && carry + x > v);
            if (hit) token = sm.rid[c0 + __ffs(hit) - 1];
            carry += __shfl_sync(0xFFFFFFFFu, x, 31);
        }
        if (token < 0 && last_pos >= 0) token = sm.rid[last_pos];

        if (lane == 0) {
            if (pair) {
                a.alpha[(size_t)b * G + unit] = (float)alpha;
                a.unit_acc[(size_t)b * G + unit] = accept;
                if (a.pos_accept) a.pos_accept[(size_t)b * G + unit] = accept;
            }
            a.unit_tok[(size_t)b * (G + 1) + unit] = token;
            if (a.pos_token) a.pos_token[(size_t)b * (G + 1) + unit] = token;
        }
        if (a.p_out)
            for (int j = lane; j < k; j += 32)
                a.p_out[((size_t)b * (G + 1) + unit) * a.V + comp_id(sm.top[0][j])] = (float)sm.prob[0][j];
        if (a.q_out && pair)
            for (int j = lane; j < k; j += 32)
                a.q_out[((size_t)b * G + unit) * a.V + comp_id(sm.top[1][j])] = (float)sm.prob[1][j];
    }
    unit_finished(a, b);
}

template <typename TIn, bool VECTOR>
__global__ void __launch_bounds__(kStreamThreads, 2) stream_kernel(Args a) {
    using C = StreamCfg<TIn>;
    __shared__ StreamSmem sm;
    const int t = threadIdx.x;
    const int V = a.V, G = a.G, ppr = a.ppr;
    const uint32_t n_pieces = a.counts[0] * (uint32_t)ppr;

    for (uint32_t w = blockIdx.x; w < n_pieces; w += gridDim.x) {
        const uint32_t row_slot = w / (uint32_t)ppr;
        const int piece = (int)(w - row_slot * (uint32_t)ppr);
        const uint32_t item = a.stream_rows[row_slot];
        const int b = (int)(item >> 8), r = (int)(item & 0xFFu);
        const SeqInfo si = a.seq[b];
        const bool is_t = r <= si.gamma;
        const int ridx = is_t ? r : r - si.gamma - 1;
        const TIn* row = is_t ? (const TIn*)a.target + ((size_t)b * (G + 1) + ridx) * (size_t)V
                              : (const TIn*)a.draft + ((size_t)b * G + ridx) * (size_t)V;
        const int col0 = piece * C::PE;

        // 1. load the whole piece: 16 independent 16-byte loads per thread
        uint4 raw[C::L];
#pragma unroll
        for (int l = 0; l < C::L; ++l) {
            const int col = col0 + (l * C::NT + t) * C::VEC;
            if (VECTOR) {
                raw[l] = (col < V) ? ld_stream16(row + col) : make_uint4(0u, 0u, 0u, 0u);
            } else {
                uint32_t wv[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                for (int j = 0; j < C::VEC; ++j) {
                    if (col + j < V) {
                        uint32_t bits;
                        if (sizeof(TIn) == 4)
                            bits = __ldg((const unsigned int*)row + col + j);
                        else
                            bits = __ldg((const unsigned short*)row + col + j);
                        const int word = j / (4 / (int)sizeof(TIn));
                        const int sh = (sizeof(TIn) == 2 && (j & 1)) ? 16 : 0;
                        wv[word] |= bits << sh;
                    }
                }
                raw[l] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
            }
        }
        if (t == 0) sm.cnt = 0;

        // 2. per-thread maximum key and non-finite detection
        uint32_t tmax = 0u;
        bool bad = false;
#pragma unroll
        for (int l = 0; l < C::L; ++l) {
            const int col = col0 + (l * C::NT + t) * C::VEC;
#pragma unroll
            for (int j = 0; j < C::VEC; ++j) {
                if (col + j < V) {
                    const uint32_t bits = elem_bits<TIn>(raw[l], j);
                    bad |= is_bad<TIn>(bits);
                    tmax = max(tmax, to_key<TIn>(bits));
                }
            }
        }
        if (__syncthreads_or(bad) && t == 0) atomicOr(&a.seq_status[b], SV_ROW_NONFINITE);

        // 3. theta = k-th largest per-thread maximum
        const int k = si.k;
        uint32_t theta = 0u;
        for (int bit = C::KB - 1; bit >= 0; --bit) {
            const uint32_t c = theta | (1u << bit);
            if (__syncthreads_count(tmax >= c) >= k) theta = c;
        }

        // 4. candidates >= theta
        uint2* list = a.cand + (size_t)w * kCandCap;
        {
            int mine = 0;
#pragma unroll
            for (int l = 0; l < C::L; ++l) {
                const int col = col0 + (l * C::NT + t) * C::VEC;
#pragma unroll
                for (int j = 0; j < C::VEC; ++j)
                    mine += (col + j < V) && (to_key<TIn>(elem_bits<TIn>(raw[l], j)) >= theta);
            }
            const int lane = t & 31;
            int x = mine;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
                if (lane >= o) x += y;
            }
            int base = 0;
            const int wtot = __shfl_sync(0xFFFFFFFFu, x, 31);
            if (lane == 31 && wtot > 0) base = atomicAdd(&sm.cnt, wtot);
            base = __shfl_sync(0xFFFFFFFFu, base, 31) + x - mine;
            if (mine > 0) {
#pragma unroll
                for (int l = 0; l < C::L; ++l) {
                    const int col = col0 + (l * C::NT + t) * C::VEC;
#pragma unroll
                    for (int j = 0; j < C::VEC; ++j) {
                        if (col + j < V) {
                            const uint32_t key = to_key<TIn>(elem_bits<TIn>(raw[l], j));
                            if (key >= theta) {
                                if (base < kCandCap) list[base] = make_uint2(key, (uint32_t)(col + j));
                                ++base;
                            }
                        }
                    }
                }
            }
        }
        __syncthreads();
        int count = sm.cnt;

        if (count > kCandCap) {
            // exact k-th largest key of the piece, then (key > kth) plus the
            // lowest-id ties at the k-th key
            uint32_t kth = 0u;
            for (int bit = C::KB - 1; bit >= 0; --bit) {
                const uint32_t c = kth | (1u << bit);
                int mine = 0;
#pragma unroll
                for (int l = 0; l < C::L; ++l) {
                    const int col = col0 + (l * C::NT + t) * C::VEC;
#pragma unroll
                    for (int j = 0; j < C::VEC; ++j)
                        mine += (col + j < V) && (to_key<TIn>(elem_bits<TIn>(raw[l], j)) >= c);
                }
                if (block_sum_int(mine, sm.red) >= k) kth = c;
            }
            int gt_mine = 0;
#pragma unroll
            for (int l = 0; l < C::L; ++l) {
                const int col = col0 + (l * C::NT + t) * C::VEC;
#pragma unroll
                for (int j = 0; j < C::VEC; ++j)
                    gt_mine += (col + j < V) && (to_key<TIn>(elem_bits<TIn>(raw[l], j)) > kth);
            }
            int gt_total;
            int pos = block_excl_scan_int(gt_mine, sm.red, &gt_total);
#pragma unroll
            for (int l = 0; l < C::L; ++l) {
                const int col = col0 + (l * C::NT + t) * C::VEC;
#pragma unroll
                for (int j = 0; j < C::VEC; ++j) {
                    if (col + j < V) {
                        const uint32_t key = to_key<TIn>(elem_bits<TIn>(raw[l], j));
                        if (key > kth) list[pos++] = make_uint2(key, (uint32_t)(col + j));
                    }
                }
            }
            // ties in ascending column order: load-group major, then thread, then lane element
            const int need = k - gt_total;
            int tie_base = 0;
#pragma unroll
            for (int l = 0; l < C::L; ++l) {
                const int col = col0 + (l * C::NT + t) * C::VEC;
                int ties = 0;
#pragma unroll
                for (int j = 0; j < C::VEC; ++j)
                    ties += (col + j < V) && (to_key<TIn>(elem_bits<TIn>(raw[l], j)) == kth);
                int ltot;
                int rank = tie_base + block_excl_scan_int(ties, sm.red, &ltot);
#pragma unroll
                for (int j = 0; j < C::VEC; ++j) {
                    if ((col + j < V) && (to_key<TIn>(elem_bits<TIn>(raw[l], j)) == kth)) {
                        if (rank < need) list[gt_total + rank] = make_uint2(kth, (uint32_t)(col + j));
                        ++rank;
                    }
                }
                tie_base += ltot;
            }
            count = k;
        }

        // 5. hand the candidates to the unit; the last piece merges
        const int unit = is_t ? (ridx < si.gamma ? ridx : si.gamma) : ridx;
        const int pieces = (unit < si.gamma ? 2 : 1) * ppr;
        __threadfence();
        __syncthreads();
        if (t == 0) {
            a.cand_cnt[w] = (uint32_t)count;
            __threadfence();
            sm.last = (atomicAdd(&a.unit_done[(size_t)b * (G + 1) + unit], 1u) == (uint32_t)(pieces - 1));
        }
        __syncthreads();
        if (sm.last) {
            __threadfence();
            combine_unit<TIn>(a, b, unit, si, sm);
        }
        __syncthreads();
    }
}

namespace {
template <typename TIn, bool VECTOR>
cudaError_t launch_stream_t(const Args& a, int sms, cudaStream_t s) {
    auto k = stream_kernel<TIn, VECTOR>;
    static int occ = [&] {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kStreamThreads, 0) != cudaSuccess) n = 1;
        return n > 0 ? n : 1;
    }();
    const long long upper = (long long)a.B * (2 * a.G + 1) * a.ppr;
    long long grid = (long long)occ * sms;
    if (grid > upper) grid = upper;
    if (grid < 1) grid = 1;
    k<<<(unsigned)grid, kStreamThreads, 0, s>>>(a);
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_stream_kernel(int dtype, bool vector, const Args& a, int sms, cudaStream_t s) {
    if (dtype == SV_BF16)
        return vector ? launch_stream_t<__nv_bfloat16, true>(a, sms, s) : launch_stream_t<__nv_bfloat16, false>(a, sms, s);
    return vector ? launch_stream_t<float, true>(a, sms, s) : launch_stream_t<float, false>(a, sms, s);
}

}  // namespace sv
