// One-pass shared-noise verification of rows with no filter.
//
// "Speculative decoding: the art of guessing well", section 共享噪声的采样: at
// position k the target's token is t_k = argmax_i (log p_k(i) + g_k,i), the draft
// token x_k is kept iff x_k = t_k, and the round ends at the first difference with
// t_k.  With temperature T > 0 and neither top-k nor top-p, log p_k(i) equals
// l_i / T minus one constant of the row, so t_k = argmax_i (l_i / T + g_k,i): the
// row needs no maximum and no sum, and one read of each target logit is the whole
// data movement.  The draft logits are not read at all.
//
// Work split.  The batch's rows of this kind form one flattened range of
// (unit, token) pairs; CTA c takes the contiguous part [c S, (c + 1) S), S a
// multiple of 8 tokens, so every CTA does the same work whatever the row count
// and V.  A CTA keeps its best (score, id) key per row it touches and merges it
// into the row's key with one 64-bit atomic max (the key orders by score, then by
// the lower id).  The CTAs touching a row are known from S, so the one that
// finishes a row's last part (an atomic counter) reads the row's key, writes the
// position's token and acceptance, and finishes the sequence when this is its
// last position.  No CTA waits for another.
//
// Per token the cost is integer and special-function arithmetic: a quarter of a
// Philox4x32-10 block (the counter (b, k, 2, i >> 2) is constant but for its last
// word, so the first two rounds are hoisted per row), and a test that rejects,
// from two fast exponentials, every token whose noise cannot lift it above the
// best score the CTA has seen; only the rest get their exact noise (two
// logarithms).  The threshold is shared: with only its own best, each thread
// passes about ln(n) of its n tokens, and across a warp that is nearly every
// step, each running the exact noise with a few lanes active.  (Dropping tokens
// before their noise is drawn does not pay: the noise spans 17 units of score,
// more than the spread of l / T over most of a row.)
#include "sv_internal.cuh"
#include "sv_finalize.cuh"

namespace sv {
namespace {

constexpr int kGThreads = 256;
constexpr int kGBlocksPerSM = 4;
constexpr unsigned long long kGMinPart = 2048;  // tokens

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11) for counters (c0, c1, c2, c3)
// whose first three words are fixed: the state after round 2 depends on c3 only
// through one XOR and one 32x32 multiply.
struct PhiloxRow {
    uint32_t x;        // c2 after round 1 is x ^ c3
    uint32_t y, z, w;  // after round 2: c0 = hi(M1 c2') ^ y, c1 = lo(M1 c2'), c2 = z, c3 = w
    uint32_t k0, k1;   // the key of round 3
};

__device__ __forceinline__ PhiloxRow philox_row(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t k0, uint32_t k1) {
    PhiloxRow r;
    // round 1
    const uint32_t a_lo = 0xD2511F53u * c0, a_hi = __umulhi(0xD2511F53u, c0);
    const uint32_t b_lo = 0xCD9E8D57u * c2, b_hi = __umulhi(0xCD9E8D57u, c2);
    const uint32_t d0 = b_hi ^ c1 ^ k0, d1 = b_lo, d3 = a_lo;
    r.x = a_hi ^ k1;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
    // round 2: the product with c0 = d0 is fixed, the one with c2 = x ^ c3 is not
    const uint32_t e_lo = 0xD2511F53u * d0, e_hi = __umulhi(0xD2511F53u, d0);
    r.y = d1 ^ k0;
    r.z = e_hi ^ d3 ^ k1;
    r.w = e_lo;
    r.k0 = k0 + 0x9E3779B9u;
    r.k1 = k1 + 0xBB67AE85u;
    return r;
}

// the four output words for last counter word c3
__device__ __forceinline__ uint4 philox_block(const PhiloxRow& r, uint32_t c3) {
    const uint32_t d2 = r.x ^ c3;
    uint32_t c0 = __umulhi(0xCD9E8D57u, d2) ^ r.y, c1 = 0xCD9E8D57u * d2, c2 = r.z, cc3 = r.w;
    uint32_t k0 = r.k0, k1 = r.k1;
#pragma unroll
    for (int i = 0; i < 8; ++i) {  // rounds 3 to 10; each product as one 32x32->64 multiply
        const unsigned long long pa = (unsigned long long)c0 * 0xD2511F53u;
        const unsigned long long pb = (unsigned long long)c2 * 0xCD9E8D57u;
        c0 = (uint32_t)(pb >> 32) ^ c1 ^ k0;
        c1 = (uint32_t)pb;
        c2 = (uint32_t)(pa >> 32) ^ cc3 ^ k1;
        cc3 = (uint32_t)pa;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return make_uint4(c0, c1, c2, cc3);
}

// 2^x by the PTX approximate base-2 exponential (relative error about 2^-22)
__device__ __forceinline__ float gex2(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// The exact test of one token with score s0 = l / T and noise word w against a
// score thr that some token of the row already reached (the CTA's best at the
// last refresh, or this thread's own best).  g(u) increases with u and no u of
// the 24-bit grid gives g above g(1 - 2^-25) = 25 ln 2 = 17.33 (kGMax adds a
// margin), so a token with D = thr - s0 >= kGMax cannot reach thr; otherwise it
// can only if u >= U(D) = exp(-exp(-D)).  U is formed with fast exponentials
// (error below 1e-6) and a 1e-5 allowance, so a rejected token scores strictly
// below thr and is not the row's argmax.  Tokens that pass get their exact noise
// and update the thread's best (equal scores: the lower id).
constexpr float kGMax = 17.5f;
struct Best {
    float s;
    uint32_t id;
};
__device__ __forceinline__ void consider(Best& bt, float thr, float s0, uint32_t w, uint32_t id) {
    constexpr float kLog2e = 1.44269504088896341f;
    const float D = fmaxf(thr, bt.s) - s0;
    if (!(D < kGMax)) return;
    const float uf = fmaf((float)(w >> 8), 5.9604644775390625e-8f, 2.98023223876953125e-8f);
    if (uf < gex2(-gex2(-D * kLog2e) * kLog2e) - 1e-5f) return;
    const float sc = s0 + gumbel_of_word(w);
    if (sc > bt.s || (sc == bt.s && id < bt.id)) {
        bt.s = sc;
        bt.id = id;
    }
}

// order-preserving 32-bit key of a float score and back (scores are never NaN)
__device__ __forceinline__ uint32_t score_okey(float s) {
    const uint32_t b = __float_as_uint(s);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float okey_score(uint32_t k) {
    return k == 0u ? -INFINITY : __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// NaN-propagating maximum (PTX max.NaN): a NaN or +inf logit anywhere shows in the result
__device__ __forceinline__ float max_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

template <typename TIn, bool VECTOR>
__global__ void __launch_bounds__(kGThreads, kGBlocksPerSM) gumbel_kernel(Args a) {
    constexpr int N = 16 / (int)sizeof(TIn);  // tokens per 16-byte vector (a multiple of 4)
    constexpr int U = 16 / N;                 // vectors in flight per thread: 16 tokens
    grid_dependency_wait();                   // the plan's lists
    grid_dependents_go();
    const uint32_t n_units = a.counts[kCntGumUnits];
    if (n_units == 0) return;
    const int V = a.V, G = a.G;
    const unsigned long long total = (unsigned long long)n_units * (unsigned)V;
    // equal parts, a multiple of 8 tokens and at least kGMinPart (a batch with few
    // such rows leaves the last CTAs idle rather than spreading them thin)
    unsigned long long S = ((total + gridDim.x - 1) / gridDim.x + 7ull) & ~7ull;
    if (S < kGMinPart) S = kGMinPart;
    const unsigned long long r0 = (unsigned long long)blockIdx.x * S;
    if (r0 >= total) return;
    const unsigned long long r1 = r0 + S < total ? r0 + S : total;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const uint32_t k0 = (uint32_t)a.seed, k1 = (uint32_t)(a.seed >> 32);
    __shared__ unsigned long long s_key[kGThreads / 32];
    __shared__ int s_bad[kGThreads / 32];
    __shared__ int s_last;
    __shared__ uint32_t s_thr;  // okey of the best score the CTA's warps have published for the row

    for (uint32_t w = (uint32_t)(r0 / (unsigned)V); (unsigned long long)w * (unsigned)V < r1; ++w) {
        const uint32_t item = a.gum_units[w];
        const int b = (int)(item >> 8), u = (int)(item & 0xFFu);
        const float cg = 1.0f / a.seq[b].T;  // the score is l / T + g
        const unsigned long long base = (unsigned long long)w * (unsigned)V;
        const int lo = r0 > base ? (int)(r0 - base) : 0;
        const int hi = r1 - base < (unsigned long long)V ? (int)(r1 - base) : V;
        const TIn* row = (const TIn*)a.target + ((size_t)b * (G + 1) + u) * (size_t)V;
        const PhiloxRow ph = philox_row((uint32_t)b, (uint32_t)(u + 1), 2u, k0, k1);
        Best bt{-INFINITY, 0u};
        float mx = -INFINITY;  // NaN-propagating maximum of the logits seen
        float thr = -INFINITY;
        if (t == 0) s_thr = 0u;
        __syncthreads();

        // vectors of N tokens overlapping [lo, hi); with VECTOR both ends are multiples of N
        const int v0 = lo / N, v1 = (hi + N - 1) / N;
        for (int vb = v0 + t; vb < v1; vb += U * kGThreads) {
            float x[U][N];
#pragma unroll
            for (int q = 0; q < U; ++q) {
                const int vi = vb + q * kGThreads;
                const int col = vi * N;
                if (VECTOR) {
                    uint4 raw = make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);  // -inf
                    if (vi < v1) raw = ld_stream16(row + col);
                    const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                    for (int j = 0; j < N; ++j) {
                        if (sizeof(TIn) == 2)
                            x[q][j] = __uint_as_float((j & 1) ? (wv[j >> 1] & 0xFFFF0000u) : (wv[j >> 1] << 16));
                        else
                            x[q][j] = (vi < v1) ? __uint_as_float(wv[j]) : -INFINITY;
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < N; ++j) {
                        const int id = col + j;
                        float xv = -INFINITY;
                        if (vi < v1 && id >= lo && id < hi) {
                            if (sizeof(TIn) == 2)
                                xv = __uint_as_float((uint32_t)__ldg((const unsigned short*)row + id) << 16);
                            else
                                xv = __ldg((const float*)row + id);
                        }
                        x[q][j] = xv;
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < U; ++q) {
                const int vi = vb + q * kGThreads;
                if (vi >= v1) continue;
                const uint32_t id0 = (uint32_t)(vi * N);  // a multiple of 4
#pragma unroll
                for (int h = 0; h < N / 4; ++h) {
                    const uint4 wq = philox_block(ph, (id0 >> 2) + (uint32_t)h);
                    const uint32_t ws4[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
                    for (int j4 = 0; j4 < 4; ++j4) {
                        const int j = 4 * h + j4;
                        mx = max_nan(mx, x[q][j]);
                        consider(bt, thr, x[q][j] * cg, ws4[j4], id0 + (uint32_t)j);
                    }
                }
            }
            {  // refresh the threshold: this warp's best, published to and read from the CTA's
                const unsigned am = __activemask();
                const uint32_t wk = __reduce_max_sync(am, score_okey(bt.s));
                if (lane == __ffs(am) - 1) atomicMax(&s_thr, wk);
                thr = fmaxf(thr, fmaxf(okey_score(wk), okey_score(*(volatile uint32_t*)&s_thr)));
            }
        }

        // the CTA's key for this row, and whether it saw a NaN or +inf logit
        unsigned long long key = bt.s > -INFINITY ? score_key(bt.s, bt.id) : 0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long y = __shfl_xor_sync(0xFFFFFFFFu, key, o);
            key = y > key ? y : key;
        }
        const bool bad = __any_sync(0xFFFFFFFFu, (mx != mx) || mx == INFINITY);
        if (lane == 0) {
            s_key[warp] = key;
            s_bad[warp] = bad ? 1 : 0;
        }
        __syncthreads();
        if (t == 0) {
            unsigned long long kb = 0ull;
            int any_bad = 0;
#pragma unroll
            for (int i = 0; i < kGThreads / 32; ++i) {
                kb = s_key[i] > kb ? s_key[i] : kb;
                any_bad |= s_bad[i];
            }
            if (kb) atomicMax(&a.gum_key[w], kb);
            if (any_bad) atomicOr(&a.seq_status[b], SV_ROW_NONFINITE);
            __threadfence();
            // the CTAs whose parts meet this row: first (base / S) to last ((base + V - 1) / S)
            const uint32_t parts = (uint32_t)((base + (unsigned)V - 1) / S - base / S + 1);
            s_last = atomicAdd(&a.gum_cnt[w], 1u) == parts - 1u;
        }
        __syncthreads();
        if (s_last) {  // every part of the row is in its key: this CTA finishes the position
            if (t == 0) {
                __threadfence();
                const unsigned long long kf = atomicAdd(&a.gum_key[w], 0ull);
                if (kf == 0ull) {  // no finite logit
                    atomicOr(&a.seq_status[b], SV_ROW_NONFINITE);
                } else {
                    const int token = score_key_id(kf);
                    if (u < a.seq[b].gamma) {
                        const int acc = a.draft_tokens[(size_t)b * G + u] == token ? 1 : 0;
                        a.unit_acc[(size_t)b * G + u] = acc;
                        if (a.pos_accept) a.pos_accept[(size_t)b * G + u] = acc;
                    }
                    a.unit_tok[(size_t)b * (G + 1) + u] = token;
                    if (a.pos_token) a.pos_token[(size_t)b * (G + 1) + u] = token;
                }
            }
            unit_finished(a, b);  // block-wide; finishes the sequence after its last position
        }
    }
}

template <typename TIn, bool VECTOR>
cudaError_t launch_gumbel_t(const Args& a, int sms, cudaStream_t s, void* const ev[2]) {
    auto k = gumbel_kernel<TIn, VECTOR>;
    static const int occ = [&] {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kGThreads, 0) != cudaSuccess) n = 1;
        return n > 0 ? n : 1;
    }();
    // at most one CTA per 2048 tokens of the largest possible batch of such rows
    const long long most = ((long long)a.B * (a.G + 1) * a.V + 2047) / 2048;
    long long grid = (long long)occ * sms;
    if (grid > most) grid = most;
    if (grid < 1) grid = 1;
    if (ev && ev[0]) cudaEventRecord((cudaEvent_t)ev[0], s);
    const cudaError_t e = launch_pdl(k, dim3((unsigned)grid), dim3(kGThreads), 0, s, a);
    if (e != cudaSuccess) return e;
    if (ev && ev[1]) cudaEventRecord((cudaEvent_t)ev[1], s);
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_gumbel_kernel(int dtype, bool vector, const Args& a, int sms, cudaStream_t s, void* const ev[2]) {
    if (dtype == SV_BF16)
        return vector ? launch_gumbel_t<__nv_bfloat16, true>(a, sms, s, ev)
                      : launch_gumbel_t<__nv_bfloat16, false>(a, sms, s, ev);
    return vector ? launch_gumbel_t<float, true>(a, sms, s, ev) : launch_gumbel_t<float, false>(a, sms, s, ev);
}

}  // namespace sv
