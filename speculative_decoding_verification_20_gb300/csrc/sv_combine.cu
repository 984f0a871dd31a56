// sv_combine.cu -- combine kernel of the streaming top-k path.
//
// A warp pair per unit (target row i with draft row i, or the bonus row
// alone): each warp merges its row's candidate lists from the select kernel
// into the exact top-k (ties to the lower id), normalises it (softmax over the
// kept logits at T, then top-p), and the first warp finishes the unit:
// alpha, the acceptance test and the residual / bonus draw (inverse CDF in
// ascending token id) ("Fast Inference from Transformers via Speculative
// Decoding" review page, Algorithm 1; "Speculative decoding: the art of
// guessing well", section 投机采样).
#include "sv_cf.cuh"
#include "sv_keys.cuh"
#include "sv_warp_sort.cuh"

namespace sv {

constexpr int kCombineThreads = 128;  // 4 warps

// ---------------------------------------------------------------------------
// combine kernel
// ---------------------------------------------------------------------------
constexpr int kCombineWarps = 4;  // two units per CTA, a warp pair per unit
static_assert(kCombineWarps == 4, "pair_sync names two pairs");
constexpr int kSelBuf = 288;      // a warp's scratch for a row's candidates (a top-k plus one load step)
static_assert(kSelBuf >= kStreamMaxK + 32, "the scratch holds a top-k plus one load step");

// shared memory of one unit: row r = 0 (target) is handled by the pair's first
// warp, r = 1 (draft) by the second
struct CombPair {
    unsigned long long buf[2][kSelBuf];       // candidates of the row being selected
    unsigned long long top[2][kStreamMaxK];   // kept entries of the target / draft row, (key desc, id asc)
    float prob[2][kStreamMaxK];               // their normalised probabilities, same order
    unsigned long long byid[2][kStreamMaxK];  // (id << 32 | position in top), ascending
    int kept[2];                              // kept entries per row (-1: no finite logit)
};

// Keep the exact top-k (key descending, then id ascending) of buf[0..m) in
// buf[0..k), unordered; returns the count.  The k-th key is found bit by bit
// below the common prefix of the smallest and largest key (warp reductions),
// ties at it by id (ids < 2^18).  M slots per lane cover m.
template <int KB, int M>
__device__ __noinline__ int warp_keep_topk_m(unsigned long long* buf, int m, int k, int lane) {
    const int used = (m + 31) >> 5;
    unsigned long long e[M];
    uint32_t key[M];
    uint32_t lo = 0xFFFFFFFFu, hi = 0u;
#pragma unroll
    for (int i = 0; i < M; ++i) {
        const int idx = lane + 32 * i;
        e[i] = (i < used && idx < m) ? buf[idx] : 0ull;
        key[i] = comp_key(e[i]);
        if (key[i] != 0u) {
            lo = min(lo, key[i]);
            hi = max(hi, key[i]);
        }
    }
    lo = __reduce_min_sync(0xFFFFFFFFu, lo);
    hi = __reduce_max_sync(0xFFFFFFFFu, hi);
    const uint32_t diff = lo ^ hi;
    const int nb = diff ? 32 - __clz(diff) : 0;
    uint32_t kth = nb >= 32 ? 0u : (lo & ~((1u << nb) - 1u));
#pragma unroll 1
    for (int bit = nb - 1; bit >= 0; --bit) {
        const uint32_t c = kth | (1u << bit);
        unsigned n = 0u;
#pragma unroll
        for (int i = 0; i < M; ++i)
            if (i < used) n += key[i] >= c;
        if (__reduce_add_sync(0xFFFFFFFFu, n) >= (unsigned)k) kth = c;
    }
    unsigned gt = 0u, eq = 0u;
#pragma unroll
    for (int i = 0; i < M; ++i) {
        gt += key[i] > kth;
        eq += key[i] == kth;
    }
    gt = __reduce_add_sync(0xFFFFFFFFu, gt);
    eq = __reduce_add_sync(0xFFFFFFFFu, eq);
    const unsigned need = (unsigned)k - gt;
    uint32_t id_cut = 0xFFFFFFFFu;
    if (eq > need) {
        uint32_t idl = 0u;
#pragma unroll 1
        for (int bit = 17; bit >= 0; --bit) {
            const uint32_t c = idl | (1u << bit);
            unsigned nlt = 0u;
#pragma unroll
            for (int i = 0; i < M; ++i) nlt += key[i] == kth && (uint32_t)comp_id(e[i]) < c;
            if (__reduce_add_sync(0xFFFFFFFFu, nlt) < need) idl = c;
        }
        id_cut = idl;
    }
    __syncwarp();
    const unsigned lt = lanemask_lt();
    int base = 0;
#pragma unroll
    for (int i = 0; i < M; ++i) {
        if (i < used) {
            const bool keep = key[i] > kth || (key[i] == kth && (uint32_t)comp_id(e[i]) <= id_cut);
            const unsigned bal = __ballot_sync(0xFFFFFFFFu, keep);
            if (keep) buf[base + __popc(bal & lt)] = e[i];
            base += __popc(bal);
        }
    }
    __syncwarp();
    return base;
}
template <int KB>
__device__ int warp_keep_topk(unsigned long long* buf, int m, int k, int lane) {
    __syncwarp();
    if (m <= k) return m;
    if (m <= 64) return warp_keep_topk_m<KB, 2>(buf, m, k, lane);
    if (m <= 128) return warp_keep_topk_m<KB, 4>(buf, m, k, lane);
    if (m <= 256) return warp_keep_topk_m<KB, 8>(buf, m, k, lane);
    return warp_keep_topk_m<KB, kSelBuf / 32>(buf, m, k, lane);
}

// Exact top-k of a row, sorted by (logit desc, id asc), from its pieces' candidate
// lists (each a superset of that piece's top-k); returns how many were found (k normally).
template <int KB>
__device__ int row_topk(const Args& a, uint32_t row_slot, int k, unsigned long long* buf, unsigned long long* top,
                        int lane) {
    const int ppr = a.ppr;
    int kept = 0;
    for (int j = 0; j < ppr; ++j) {
        const size_t piece = (size_t)row_slot * ppr + j;
        const int c = (int)__ldcg(&a.cand_cnt[piece]);
        const unsigned long long* src = a.cand + (size_t)row_slot * a.cand_rowcap + (size_t)j * kListCap;
        for (int i0 = 0; i0 < c;) {
            if (kept + 32 > kSelBuf) kept = warp_keep_topk<KB>(buf, kept, k, lane);
            const int take = min(c - i0, kSelBuf - kept);
#pragma unroll 4
            for (int i = lane; i < take; i += 32) buf[kept + i] = __ldcg(&src[i0 + i]);
            kept += take;
            i0 += take;
        }
    }
    kept = warp_keep_topk<KB>(buf, kept, k, lane);
    warp_sort(buf, kept, top, true, 0ull, lane);
    return kept;
}

// (id << 32 | position) of the kept entries, ascending by id
__device__ __forceinline__ void index_by_id(const unsigned long long* top, int n, unsigned long long* buf,
                                            unsigned long long* byid, int lane) {
    for (int j = lane; j < n; j += 32) buf[j] = ((unsigned long long)(uint32_t)comp_id(top[j]) << 32) | (uint32_t)j;
    __syncwarp();
    warp_sort(buf, n, byid, false, ~0ull, lane);
}

// probability of token x in a kept list indexed by id (0 if not kept)
__device__ __forceinline__ float prob_of(const unsigned long long* byid, const float* prob, int n, int x) {
    int lo = 0, hi = n - 1;
    while (lo <= hi) {
        const int mid = (lo + hi) >> 1;
        const int id = (int)(byid[mid] >> 32);
        if (id == x) return prob[(uint32_t)byid[mid]];
        if (id < x)
            lo = mid + 1;
        else
            hi = mid - 1;
    }
    return 0.0f;
}

// Unnormalised weight 2^((l - vmax) * c) of a kept logit l, c = log2(e) / T
// given as a float pair chi + clo, to about fp32 rounding whatever the size
// of the exponent and without fp64 arithmetic: the difference is formed
// exactly (two-sum; exact in fp32 anyway for bf16 logits), its product with
// chi by an FMA two-product, the integer part n is applied exactly and only
// the fraction in [-1/2, 1/2] goes through exp2f.  Below 2^-126 the weight is 0.
__device__ __forceinline__ float kept_weight(float l, float vmax, float chi, float clo) {
    const float d = l - vmax;
    const float p = d * chi;
    const float n = rintf(p);
    if (!(n >= -126.0f)) return 0.0f;
    const float bb = d - l;
    const float dlo = (l - (d - bb)) + (-vmax - bb);  // l - vmax = d + dlo exactly
    const float e = fmaf(d, chi, -p);                  // d * chi = p + e exactly
    const float f = (p - n) + (e + fmaf(d, clo, dlo * chi));
    return exp2f(f) * __int_as_float((int)(n + 127.0f) << 23);
}
template <typename TIn>
__device__ __forceinline__ float key_logit(uint32_t k) {
    return sizeof(TIn) == 2 ? key_value16(k) : key_value32(k);
}

// Normalisation of one sorted kept list by one warp: softmax over the kept
// logits at temperature T (one-hot if T == 0), then top-p.  prob[j] for j < k.
// No fp64: the top-p prefix is found by comparing the running sum of the
// weights with P * S (S their sum) as compensated pairs, with no division, so
// k exactly tied weights cross exactly where j >= P * k, as the fp64
// definition decides for k <= 256 and a float P.
template <typename TIn>
__device__ void normalise_kept(const unsigned long long* top, int k, float Tf, float Pf, float* prob) {
    const int lane = threadIdx.x & 31;
    if (Tf == 0.0f) {
        for (int j = lane; j < k; j += 32) prob[j] = (j == 0) ? 1.0f : 0.0f;
        __syncwarp();
        return;
    }
    const float vmax = key_logit<TIn>(comp_key(top[0]));
    // log2(e) / T = chi + clo: chi rounded, clo from the exact remainder of the division
    constexpr float kL2eHi = 1.44269502162933349609375f;  // fp32(log2 e)
    constexpr float kL2eLo = 1.925963033500011e-08f;       // log2 e - kL2eHi
    const float chi = kL2eHi / Tf;
    const float clo = (fmaf(-chi, Tf, kL2eHi) + kL2eLo) / Tf;
    CF s{0.0f, 0.0f};
    for (int j = lane; j < k; j += 32) {
        const float w = kept_weight(key_logit<TIn>(comp_key(top[j])), vmax, chi, clo);
        prob[j] = w;
        s = cf_add(s, CF{w, 0.0f});
    }
    s = warp_cf_sum(s);
    __syncwarp();
    int keep = k;
    if (Pf < 1.0f) {  // shortest prefix (prob desc, id asc) whose mass reaches P, crossing token kept
        const CF ps = cf_scale(Pf, s);
        CF carry{0.0f, 0.0f};
        for (int c0 = 0; c0 < k; c0 += 32) {
            const int j = c0 + lane;
            const CF x = cf_add(carry, warp_cf_scan(CF{j < k ? prob[j] : 0.0f, 0.0f}, lane));
            const unsigned hit = __ballot_sync(0xFFFFFFFFu, j < k && cf_ge(x, ps));
            if (hit) {
                keep = c0 + __ffs(hit);
                break;
            }
            carry = CF{__shfl_sync(0xFFFFFFFFu, x.s, 31), __shfl_sync(0xFFFFFFFFu, x.c, 31)};
        }
    }
    CF s2 = s;
    if (keep < k) {
        s2 = CF{0.0f, 0.0f};
        for (int j = lane; j < keep; j += 32) s2 = cf_add(s2, CF{prob[j], 0.0f});
        s2 = warp_cf_sum(s2);
    }
    const float inv = cf_recip(s2);
    __syncwarp();
    for (int j = lane; j < k; j += 32) prob[j] = j < keep ? prob[j] * inv : 0.0f;
    __syncwarp();
}

// One row of a unit, by one warp: exact top-k, normalisation (softmax at T,
// then top-p) and the index by token id.
template <typename TIn>
__device__ void combine_row(const Args& a, const SeqInfo& si, int unit, int r, CombPair& sm, int lane) {
    // K-SEQ rows are one target and one draft row per sequence
    const uint32_t slot = si.row_off + (a.kseq ? (uint32_t)r
                                               : r == 0 ? (uint32_t)unit : (uint32_t)si.gamma + 1u + (uint32_t)unit);
    const int kk = row_topk<Elem<TIn>::KB>(a, slot, si.k, sm.buf[r], sm.top[r], lane);  // ties to the lower id
    // a row without a finite logit (non-finite ones are already flagged)
    const uint32_t ninf_key = Elem<TIn>::key(Elem<TIn>::kNegInfBits);
    const bool dead = kk < 1 || comp_key(sm.top[r][0]) <= ninf_key;
    if (!dead) {
        normalise_kept<TIn>(sm.top[r], kk, si.T, si.P, sm.prob[r]);
        index_by_id(sm.top[r], kk, sm.buf[r], sm.byid[r], lane);
    }
    if (lane == 0) sm.kept[r] = dead ? -1 : kk;
    __syncwarp();
}

// The rest of a unit, by the pair's first warp once both rows are done.
template <typename TIn>
__device__ void combine_unit(const Args& a, int b, int unit, const SeqInfo& si, CombPair& sm, int lane, int x) {
    const int G = a.G;
    const bool pair = unit < si.gamma;
    const int kt = sm.kept[0], kd = pair ? sm.kept[1] : 0;
    // the unit's two uniforms (acceptance, residual draw), one per lane, in parallel
    const double uu = lane < 2 ? uniform01(a.seed, (uint32_t)b, (uint32_t)(unit + 1), (uint32_t)lane) : 0.0;
    const double u_acc = __shfl_sync(0xFFFFFFFFu, uu, 0), u_res = __shfl_sync(0xFFFFFFFFu, uu, 1);
    if (kt < 0 || kd < 0) {
        if (lane == 0) atomicOr(&a.seq_status[b], SV_ROW_NONFINITE);
        unit_finished_warp(a, b, lane);
        return;
    }

    // acceptance test u * l * q(x) < p(x) (l = 1: the exact rule)
    int accept = 0;
    if (pair) {
        const double px = (double)prob_of(sm.byid[0], sm.prob[0], kt, x);
        const double qx = (double)prob_of(sm.byid[1], sm.prob[1], kd, x);
        accept = lenient_accept(u_acc, si.L, qx, px) ? 1 : 0;
    }

    // alpha_i = sum_x min(p, q) (under lenience l, sum_x min(q, p / l)) and the
    // residual weights, in ascending token id over the target's kept ids (an id
    // kept only by the draft has p = 0, so it adds nothing to either)
    const float invl = lenience_inv(si.L);
    // the residual weights in id order, kept in the target row's free scratch
    float* rr = reinterpret_cast<float*>(sm.buf[0]);
    CF alpha{0.0f, 0.0f}, Z{0.0f, 0.0f}, Zp{0.0f, 0.0f};
    for (int j = lane; j < kt; j += 32) {
        const unsigned long long e = sm.byid[0][j];
        const float p = sm.prob[0][(uint32_t)e];
        const float q = pair ? prob_of(sm.byid[1], sm.prob[1], kd, (int)(e >> 32)) : 0.0f;
        alpha = cf_add(alpha, CF{accept_mass(p, q, invl), 0.0f});
        const float r = fmaxf(p - q, 0.0f);  // bonus: q_{gamma+1} := 0
        rr[j] = r;
        Z = cf_add(Z, CF{r, 0.0f});
        Zp = cf_add(Zp, CF{p, 0.0f});
    }
    const float alpha_v = cf_val(warp_cf_sum(alpha));
    float Zt = cf_val(warp_cf_sum(Z));
    const bool use_p = !(Zt > 0.0f);  // p <= q everywhere: fall back to p
    if (use_p) {
        Zt = cf_val(warp_cf_sum(Zp));
        for (int j = lane; j < kt; j += 32) rr[j] = sm.prob[0][(uint32_t)sm.byid[0][j]];
    }
    __syncwarp();
    // inverse CDF: the first id whose running sum passes v
    const double v = u_res * (double)Zt;
    int token = -1, last_pos = -1;
    CF carry{0.0f, 0.0f};
    for (int c0 = 0; c0 < kt && token < 0; c0 += 32) {
        const int j = c0 + lane;
        const float r = j < kt ? rr[j] : 0.0f;
        const CF x = cf_add(carry, warp_cf_scan(CF{r, 0.0f}, lane));
        const unsigned pos = __ballot_sync(0xFFFFFFFFu, j < kt && r > 0.0f);
        if (pos) last_pos = c0 + 31 - __clz(pos);
        const unsigned hit =
            __ballot_sync(0xFFFFFFFFu, j < kt && r > 0.0f && (double)x.s - (double)x.c > v);
        if (hit) token = (int)(sm.byid[0][c0 + __ffs(hit) - 1] >> 32);
        carry = CF{__shfl_sync(0xFFFFFFFFu, x.s, 31), __shfl_sync(0xFFFFFFFFu, x.c, 31)};
    }
    if (token < 0 && last_pos >= 0) token = (int)(sm.byid[0][last_pos] >> 32);

    if (lane == 0) {
        if (pair) {
            a.alpha[(size_t)b * G + unit] = alpha_v;
            a.unit_acc[(size_t)b * G + unit] = accept;
            if (a.pos_accept) a.pos_accept[(size_t)b * G + unit] = accept;
        }
        a.unit_tok[(size_t)b * (G + 1) + unit] = token;
        if (a.pos_token) a.pos_token[(size_t)b * (G + 1) + unit] = token;
    }
    if (a.p_out)
        for (int j = lane; j < kt; j += 32)
            a.p_out[((size_t)b * (G + 1) + unit) * a.V + comp_id(sm.top[0][j])] = sm.prob[0][j];
    if (a.q_out && pair)
        for (int j = lane; j < kd; j += 32)
            a.q_out[((size_t)b * G + unit) * a.V + comp_id(sm.top[1][j])] = sm.prob[1][j];
    unit_finished_warp(a, b, lane);
}

// Shared-noise verification of one position ("Speculative decoding: the art
// of guessing well", section 共享噪声的采样): the target's token is the argmax over
// the row's kept set of log p(i) + g(i), which for kept tokens is (l_i - l_max) / T
// + g(i) up to one constant (the renormalisation), with g the Philox noise of
// token i at this position; ties go to the lower id; T = 0 is the argmax itself.
// The draft token passes iff it is that token.  One warp, from the sorted kept
// list of the target row.
template <typename TIn>
__device__ void gumbel_unit(const Args& a, int b, int unit, const SeqInfo& si, CombPair& sm, int lane, int x) {
    const int G = a.G;
    const bool pair = unit < si.gamma;
    const int kt = sm.kept[0];
    if (kt < 0) {
        if (lane == 0) atomicOr(&a.seq_status[b], SV_ROW_NONFINITE);
        unit_finished_warp(a, b, lane);
        return;
    }
    int token;
    if (si.T == 0.0f) {
        token = comp_id(sm.top[0][0]);  // the largest logit, lowest id among equals
    } else {
        const float lmax = key_logit<TIn>(comp_key(sm.top[0][0]));
        const float c = 1.0f / si.T;
        const uint32_t k0 = (uint32_t)a.seed, k1 = (uint32_t)(a.seed >> 32);
        unsigned long long best = 0ull;
        for (int j = lane; j < kt; j += 32) {
            if (!(sm.prob[0][j] > 0.0f)) continue;  // past the nucleus cut
            const unsigned long long e = sm.top[0][j];
            const uint32_t id = (uint32_t)comp_id(e);
            const uint4 w = philox4((uint32_t)b, (uint32_t)(unit + 1), 2u, id >> 2, k0, k1);
            const uint32_t wi = (id & 3u) == 0 ? w.x : (id & 3u) == 1 ? w.y : (id & 3u) == 2 ? w.z : w.w;
            const float sc = fmaf(key_logit<TIn>(comp_key(e)) - lmax, c, gumbel_of_word(wi));
            const unsigned long long kk = score_key(sc, id);
            best = kk > best ? kk : best;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long y = __shfl_xor_sync(0xFFFFFFFFu, best, o);
            best = y > best ? y : best;
        }
        token = score_key_id(best);
    }
    if (lane == 0) {
        if (pair) {
            const int acc = (x == token) ? 1 : 0;
            a.unit_acc[(size_t)b * G + unit] = acc;
            if (a.pos_accept) a.pos_accept[(size_t)b * G + unit] = acc;
        }
        a.unit_tok[(size_t)b * (G + 1) + unit] = token;
        if (a.pos_token) a.pos_token[(size_t)b * (G + 1) + unit] = token;
    }
    if (a.p_out)
        for (int j = lane; j < kt; j += 32)
            a.p_out[((size_t)b * (G + 1) + unit) * a.V + comp_id(sm.top[0][j])] = sm.prob[0][j];
    unit_finished_warp(a, b, lane);
}

// K-SEQ verification of one position ("SpecTr: Fast Speculative Decoding via
// Optimal Transport" page, section K-SEQ, eqs. (4)-(7) and the residual
// distribution; p = target, q = draft here) for rows with top-k <= 256 or
// greedy: both rows are supported on their kept lists, so everything below
// runs on one warp over at most 256 tokens.  With m(x) = min(q(x), p(x) / rho)
// and beta(rho) = sum_x m(x) (only tokens kept by both rows add to it):
//   rho* is the root on [1, k] of f(rho) = 1 - (1 - beta)^k - rho beta, which
//     does not increase with rho: bisection, keeping the end where f <= 0;
//   candidate i (in the given order, uniform U(seed, b, 1, 3 + i)) is accepted
//     iff u_i rho* q(X_i) < p(X_i); the first accepted one is emitted;
//   otherwise the token is drawn from p - A, A = (P_A / beta) m at rho*,
//     P_A = 1 - (1 - beta)^k, by the inverse CDF in ascending token id with
//     U(seed, b, 1, 1) (p itself when the residual has no mass).
template <typename TIn>
__device__ void kseq_list_unit(const Args& a, int b, const SeqInfo& si, CombPair& sm, int lane) {
    const int kt = sm.kept[0], kd = sm.kept[1], k = si.gamma;
    uint32_t st = __ldcg(&a.seq_status[b]);  // a NaN or +inf logit seen by the select kernel
    if (kt < 0 || kd < 0) st |= SV_ROW_NONFINITE;
    if (st) {
        if (lane == 0) {
            a.out_tokens[b] = -1;
            a.accepted_len[b] = -1;
            if (a.row_status) a.row_status[b] = st;
        }
        return;
    }
    // the draft probability of each of the target's kept tokens, and the target
    // probability of each of the draft's (in the draft row's free scratch; 0 where
    // the other row does not keep the token)
    float* qk = reinterpret_cast<float*>(sm.buf[1]);
    float* pk = qk + kStreamMaxK;
    for (int j = lane; j < kt; j += 32)
        qk[j] = sm.prob[0][j] > 0.0f ? prob_of(sm.byid[1], sm.prob[1], kd, comp_id(sm.top[0][j])) : 0.0f;
    for (int j = lane; j < kd; j += 32)
        pk[j] = sm.prob[1][j] > 0.0f ? prob_of(sm.byid[0], sm.prob[0], kt, comp_id(sm.top[1][j])) : 0.0f;
    __syncwarp();
    // compensated fp32 sums over the warp of beta = sum min(q, p / rho),
    // R = sum (p - rho q)+ (= 1 - rho beta) and D = sum (q - p / rho)+ (= 1 - beta)
    auto wsum = [&](CF s) -> float { return cf_val(warp_cf_sum(s)); };
    auto beta_f = [&](float inv) {
        CF s{0.0f, 0.0f};
        for (int j = lane; j < kt; j += 32) s = cf_add(s, CF{fminf(qk[j], sm.prob[0][j] * inv), 0.0f});
        return wsum(s);
    };
    // rho*: bisection on [1, k] with the sign of f taken in fp32 from a form without
    // cancellation (dependent fp64 operations are slow on this GPU): for beta <= 1/2,
    // f = 1 - (1 - beta)^k - rho beta = -expm1(k log1p(-beta)) - rho beta, each term
    // accurate to its own size; above, f = R - D^k, two sums of nonnegative terms.
    // Both are accurate relative to f's terms, so a sign is wrong only within about
    // 1e-7 (relative) of the root; the end where f <= 0 is kept, as the page's
    // bisection does
    double lo = 1.0, hi = (double)k;
    for (int it = 0; it < 40 && k > 1 && hi - lo > 5.9604644775390625e-8 * hi; ++it) {
        const double mid = 0.5 * (lo + hi);
        const float r = (float)mid, inv = 1.0f / r;
        const float be = beta_f(inv);
        float fv;
        if (be <= 0.5f) {
            fv = -expm1f((float)k * log1pf(-be)) - r * be;
        } else {
            CF sr{0.0f, 0.0f}, sd{0.0f, 0.0f};
            for (int j = lane; j < kt; j += 32) sr = cf_add(sr, CF{fmaxf(sm.prob[0][j] - r * qk[j], 0.0f), 0.0f});
            for (int j = lane; j < kd; j += 32) sd = cf_add(sd, CF{fmaxf(sm.prob[1][j] - pk[j] * inv, 0.0f), 0.0f});
            const float R = wsum(sr), D = wsum(sd);
            float pw = 1.0f;
            for (int i = 0; i < k; ++i) pw *= D;
            fv = R - pw;
        }
        if (fv > 0.0f)
            lo = mid;
        else
            hi = mid;
    }
    const double rho = k > 1 ? hi : 1.0;
    auto beta_at = [&](double x) -> double {
        const float inv = (float)(1.0 / x);
        CF s{0.0f, 0.0f};
        for (int j = lane; j < kt; j += 32) s = cf_add(s, CF{fminf(qk[j], sm.prob[0][j] * inv), 0.0f});
        s = warp_cf_sum(s);
        return (double)s.s - (double)s.c;
    };
    const double beta = beta_at(rho);

    // the candidates, one per lane: the lowest index that passes wins
    int idx = -1, token = -1;
    {
        bool pass = false;
        int x = 0;
        if (lane < k) {
            x = a.draft_tokens[(size_t)b * a.G + lane];
            const double px = (double)prob_of(sm.byid[0], sm.prob[0], kt, x);
            const double qx = (double)prob_of(sm.byid[1], sm.prob[1], kd, x);
            const double u = uniform01(a.seed, (uint32_t)b, 1u, 3u + (uint32_t)lane);
            pass = u * rho * qx < px;
        }
        const unsigned m = __ballot_sync(0xFFFFFFFFu, pass);
        if (m) {
            idx = __ffs(m) - 1;
            token = __shfl_sync(0xFFFFFFFFu, x, idx);
        }
    }
    if (idx < 0) {
        // the residual p - A at rho*, in ascending token id over the target's kept set
        double omb_k = 1.0;  // (1 - beta)^k, k <= 13 products, once
        for (int i = 0; i < k; ++i) omb_k *= (1.0 - beta);
        const double PA = beta > 0.0 ? 1.0 - omb_k : 0.0;
        const float As = beta > 0.0 ? (float)(PA / beta) : 0.0f;
        const float inv_rho = (float)(1.0 / rho);
        float* rr = reinterpret_cast<float*>(sm.buf[0]);
        CF Z{0.0f, 0.0f}, Zp{0.0f, 0.0f};
        for (int j = lane; j < kt; j += 32) {
            const unsigned long long e = sm.byid[0][j];
            const float p = sm.prob[0][(uint32_t)e];
            const float q = prob_of(sm.byid[1], sm.prob[1], kd, (int)(e >> 32));
            const float r = fmaxf(p - As * fminf(q, p * inv_rho), 0.0f);
            rr[j] = r;
            Z = cf_add(Z, CF{r, 0.0f});
            Zp = cf_add(Zp, CF{p, 0.0f});
        }
        float Zt = cf_val(warp_cf_sum(Z));
        if (!(Zt > 0.0f)) {  // no residual mass (P_A = 1 up to rounding): draw from p
            Zt = cf_val(warp_cf_sum(Zp));
            for (int j = lane; j < kt; j += 32) rr[j] = sm.prob[0][(uint32_t)sm.byid[0][j]];
        }
        __syncwarp();
        const double v = uniform01(a.seed, (uint32_t)b, 1u, 1u) * (double)Zt;
        int last_pos = -1;
        CF carry{0.0f, 0.0f};
        for (int c0 = 0; c0 < kt && token < 0; c0 += 32) {
            const int j = c0 + lane;
            const float r = j < kt ? rr[j] : 0.0f;
            const CF xs = cf_add(carry, warp_cf_scan(CF{r, 0.0f}, lane));
            const unsigned pos = __ballot_sync(0xFFFFFFFFu, j < kt && r > 0.0f);
            if (pos) last_pos = c0 + 31 - __clz(pos);
            const unsigned hit =
                __ballot_sync(0xFFFFFFFFu, j < kt && r > 0.0f && (double)xs.s - (double)xs.c > v);
            if (hit) token = (int)(sm.byid[0][c0 + __ffs(hit) - 1] >> 32);
            carry = CF{__shfl_sync(0xFFFFFFFFu, xs.s, 31), __shfl_sync(0xFFFFFFFFu, xs.c, 31)};
        }
        if (token < 0 && last_pos >= 0) token = (int)(sm.byid[0][last_pos] >> 32);
    }
    if (lane == 0) {
        a.out_tokens[b] = token;
        a.accepted_len[b] = idx;
        if (a.row_status) a.row_status[b] = 0u;
    }
}

// named barrier of warp pair pr (ids 1 and 2; the ids are constants so the
// kernel holds only the barriers it uses)
__device__ __forceinline__ void pair_sync(int pr) {
    if (pr == 0)
        asm volatile("bar.sync 1, 64;" ::: "memory");
    else
        asm volatile("bar.sync 2, 64;" ::: "memory");
}

// a warp pair per unit (target row i with draft row i, or the bonus row alone):
// the two rows are selected and normalised at the same time
// 7 CTAs (14 units) per SM: the whole unit list of a 256-sequence, 8-unit batch
// in one wave on 152 SMs (shared memory 7 x 29 KB, at most 73 registers)
// KSEQ: the K-SEQ instantiation (a.kseq), kept apart so the sampling path's
// register allocation does not carry it
template <typename TIn, bool KSEQ>
__global__ void __launch_bounds__(kCombineThreads, 7) combine_kernel(Args a) {
    extern __shared__ __align__(16) uint8_t comb_raw[];
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int pr = wid >> 1, r = wid & 1;
    CombPair& sm = reinterpret_cast<CombPair*>(comb_raw)[pr];
    constexpr int kPairs = kCombineWarps / 2;
    // No streaming unit: leave at once, without waiting for the select kernel.  The
    // count is the plan's, final and visible here: this kernel is launched only
    // once every select CTA has passed its own wait, which the plan's completion
    // precedes.
    if (a.counts[kCntStreamUnits] == 0u) return;
    grid_dependency_wait();  // the select kernel's candidate lists
    grid_dependents_go();
    const uint32_t n_units = a.counts[kCntStreamUnits];
    const bool failed = a.counts[kCntError] != 0u;
    // both warps of a pair walk the same units, so they meet at the same barriers
    for (uint32_t w = blockIdx.x * kPairs + pr; w < n_units; w += gridDim.x * kPairs) {
        const uint32_t item = a.stream_units[w];
        const int b = (int)(item >> 8), unit = (int)(item & 0xFFu);
        const SeqInfo si = a.seq[b];
        if (failed) {  // a select CTA gave up waiting: no result of this call can be trusted
            if (r == 0) {
                if (KSEQ) {  // K-SEQ outputs are per row, written here
                    if (lane == 0) {
                        a.out_tokens[b] = -1;
                        a.accepted_len[b] = -1;
                        if (a.row_status) a.row_status[b] = __ldcg(&a.seq_status[b]) | SV_ROW_INTERNAL;
                    }
                } else {
                    if (lane == 0) atomicOr(&a.seq_status[b], SV_ROW_INTERNAL);
                    unit_finished_warp(a, b, lane);
                }
            }
            continue;
        }
        if constexpr (KSEQ) {  // both rows of the position, then the K-SEQ step on the first warp
            combine_row<TIn>(a, si, 0, r, sm, lane);
            pair_sync(pr);
            if (r == 0) kseq_list_unit<TIn>(a, b, si, sm, lane);
            pair_sync(pr);
            continue;
        }
        // the draft token, loaded early: its latency hides behind the row work
        const int x = (r == 0 && unit < si.gamma) ? a.draft_tokens[(size_t)b * a.G + unit] : 0;
        // shared-noise verification reads the target rows only
        if (r == 0 || (unit < si.gamma && !a.gumbel)) combine_row<TIn>(a, si, unit, r, sm, lane);
        pair_sync(pr);
        if (r == 0) {
            if (a.gumbel)
                gumbel_unit<TIn>(a, b, unit, si, sm, lane, x);
            else
                combine_unit<TIn>(a, b, unit, si, sm, lane, x);
        }
        pair_sync(pr);  // the rows may be rebuilt
    }
}

namespace {
template <typename TIn, bool KSEQ>
cudaError_t launch_comb_t(const Args& a, int sms, cudaStream_t s) {
    auto comb = combine_kernel<TIn, KSEQ>;
    const int csmem = (int)((kCombineWarps / 2) * sizeof(CombPair));
    static const bool cattr_ok = cudaFuncSetAttribute(comb, cudaFuncAttributeMaxDynamicSharedMemorySize, csmem) ==
                                 cudaSuccess;
    if (!cattr_ok) return cudaErrorInvalidValue;
    static const int cocc = [&] {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, comb, kCombineThreads, csmem) != cudaSuccess) n = 1;
        return n > 0 ? n : 1;
    }();
    long long cgrid = ((long long)a.B * (a.G + 1) + kCombineWarps / 2 - 1) / (kCombineWarps / 2);
    if (cgrid > (long long)sms * cocc) cgrid = (long long)sms * cocc;
    if (cgrid < 1) cgrid = 1;
    return launch_pdl(comb, dim3((unsigned)cgrid), dim3(kCombineThreads), (size_t)csmem, s, a);
}
}  // namespace

cudaError_t launch_combine_kernel(int dtype, const Args& a, int sms, cudaStream_t s) {
    if (a.kseq)
        return dtype == SV_BF16 ? launch_comb_t<__nv_bfloat16, true>(a, sms, s) : launch_comb_t<float, true>(a, sms, s);
    return dtype == SV_BF16 ? launch_comb_t<__nv_bfloat16, false>(a, sms, s) : launch_comb_t<float, false>(a, sms, s);
}

}  // namespace sv
