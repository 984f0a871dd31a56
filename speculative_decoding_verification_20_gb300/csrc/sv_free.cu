// sv_free.cu -- whole-row path of sequences with no top-k and temperature > 0
// (top-p or no filter at all).
//
// A unit is (target row i, draft row i) for i < gamma_b, or the bonus unit
// (target row gamma_b alone, q := 0).  p and q are softmaxes of the whole
// vocabulary at temperature T, cut to the nucleus when top-p < 1 ("Fast
// Inference from Transformers via Speculative Decoding" review page, section
// "Method: Speculative Decoding"), and each unit needs:
//   - the normaliser of each row (online maximum and sum of exp),
//   - for top-p < 1, the last token of each row's nucleus (the shortest prefix,
//     by probability descending then id ascending, whose mass reaches P),
//   - alpha = sum_x min(p, q) and the residual weights r = max(0, p - q)
//     (p for the bonus row),
//   - the acceptance test u * q(x) < p(x) of the draft token
//     ("Speculative decoding: the art of guessing well", section 投机采样), with
//     q(x) scaled by the sequence's lenience (review page, section Lenience),
//   - the residual / bonus draw: v = u * sum r and the first token id at which
//     the running sum of r passes v.
//
// free_kernel (persistent, 2 CTAs per SM, 7 consumer warps + 1 producer warp)
//   The producer claims units from a global counter and streams each unit's
//   rows through a 3-stage ring (a stage holds a 14 KB segment of each row) by
//   TMA bulk copies: pass 0 for the row statistics, passes 1-3 for the nucleus
//   cut when top-p < 1, and the final pass for alpha and the residual weights.
//   Every pass after the first reads the rows again while they are in L2.
//   Consumer warp w owns the contiguous 2 KB block w of each segment, so its
//   sums of r and of p over that block are sums over consecutive token ids;
//   they go to the unit's record in the workspace with the warp's share of
//   alpha.  Per-thread sums are Kahan-compensated fp32 and warp sums an exact
//   two-sum.  Only the row statistics need a barrier of the consumer warps
//   (and each nucleus pass one or two); a unit ends without one.
// free_tail_kernel (a warp per unit, after free_kernel)
//   Sums the unit's block sums, finds the block where the running sum passes
//   v, re-reads that 2 KB block of each row to find the token inside it, runs
//   the acceptance test from the two logits of the draft token and writes the
//   unit's outputs.
// Every wait of free_kernel (ring and the consumers' own barrier) is bounded
// (2 s); on a timeout the CTA records kCntError and the tail kernel marks every
// sequence of the path as failed.
#include <type_traits>

#include "sv_cf.cuh"
#include "sv_finalize.cuh"
#include "sv_warp_sort.cuh"

namespace sv {
namespace {

constexpr int kFStages = 3;
constexpr int kFVec = kFreeBlockBytes / 16 / 32;  // 16-byte vectors per lane per segment (4)
// W consumer warps and a producer warp; up to 128 registers a thread either way
// (7: 2 CTAs per SM, 15: 1 CTA per SM)
template <int W>
struct FGeo {
    static constexpr int kConsumers = 32 * W;
    static constexpr int kThreads = kConsumers + 32;
    static constexpr int kSegBytes = W * kFreeBlockBytes;
    static constexpr int kCtasPerSm = W == kFreeWarpsNarrow ? 2 : 1;
    static_assert(W < 32 && kFVec * 16 * kConsumers == kSegBytes, "segment geometry");
};
constexpr int kTailWarps = 8;

// nucleus (top-p) cut of a row: probability mass histograms over the distance
// below the row maximum, d = (max - l) * log2(e) / T, in log2 units
constexpr float kNDmax = 64.0f;  // beyond it a logit's mass is below 2^-64 of the maximum's
constexpr int kNB1 = 512;        // coarse bins of 1/8 log2 unit
constexpr int kNB2 = 512;        // fine bins inside the coarse bin where the running mass passes P
constexpr int kNCap = 256;       // elements of the crossing fine bin sorted here (else: cluster kernel)
constexpr float kMassScale = 1099511627776.0f;  // 2^40: masses are summed exactly in fixed point
// A logit's fixed-point mass m <= 2^40 is added to a bin as two 32-bit parts,
// m >> 10 and m & 1023 (native shared-memory atomics; a 64-bit atomic per
// logit serialises on the hot bins).  Neither part can overflow: the high
// parts of a row sum to at most 2^30 (the masses sum to 1), and a bin's low
// parts to at most 1023 * SV_MAX_VOCAB < 2^28.
constexpr int kMassLoBits = 10;
static_assert(1023ull * SV_MAX_VOCAB < (1ull << 32), "low parts of a bin fit 32 bits");
// passes of a unit through the ring: 0 statistics, 1 coarse histogram, 2 fine
// histogram, 3 collect the crossing elements, 4 alpha and residual weights
constexpr int kPassFinal = 4;

template <int W>
struct FreeSmem {
    alignas(128) uint8_t buf[kFStages][2][FGeo<W>::kSegBytes];  // [stage][target, draft segment]
    uint64_t full[kFStages];
    uint64_t empty[kFStages];
    uint64_t gsync;
    int4 hdr[kFStages];               // unit index (-1: no more work), pass, tile, elements
    int4 uhdr[kFStages];              // the unit: list item (b << 8 | u), gamma_b, T and top-p (float bits)
    float red[2][W][8];               // per warp: row statistics (by the parity of the CTA's unit count)
    uint32_t h1[2][2][kNB1];          // per row: coarse mass histogram (2^40 fixed point) as [high, low] parts
    uint32_t h2[2][2][kNB2];          // per row: fine mass histogram, the same way
    unsigned long long list[2][kNCap];  // per row: the elements of the crossing fine bin
    int nb[2][2];                     // per row: crossing coarse bin, crossing fine bin
    unsigned long long nbase[2];      // per row: mass before the crossing fine bin
    int ncnt[2];                      // per row: crossing elements collected
    uint32_t cut_key[2], cut_id[2];   // per row: the last kept element (key, id)
    float kinv[2];                    // per row: 1 / (sum x kept mass); -1: too many ties at the cut
    float lhdr[kFStages];             // the unit's lenience, with uhdr
    unsigned long long wait_ns;       // limit of every wait on another warp or a copy (Args::wait_ns)
};

// 228 KB of shared memory per SM, less 1 KB reserved per CTA
static_assert(sizeof(FreeSmem<kFreeWarpsNarrow>) <= 115712, "the narrow whole-row kernel must fit twice on an SM");
static_assert(sizeof(FreeSmem<kFreeWarpsWide>) <= 232448, "the wide whole-row kernel must fit on an SM");

// ---------------------------------------------------------------------------
// PTX helpers (mbarriers, TMA bulk copies); every wait is bounded
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t fs_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void fbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(fs_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(fs_u32(bar)) : "memory");
}
__device__ __forceinline__ void fbar_expect(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(fs_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool fbar_try(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(fs_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long fs_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// bounded wait: false after about limit_ns (each try sleeps at most min(limit_ns, 1 ms))
__device__ __forceinline__ bool fbar_wait(uint64_t* bar, uint32_t parity, unsigned long long limit_ns) {
    const uint32_t hint = limit_ns < 1000000ull ? (uint32_t)limit_ns : 1000000u;
    if (fbar_try(bar, parity, hint)) return true;
    if (limit_ns < 1000ull) return false;  // below the timer's ~1 us resolution: one try only
    const unsigned long long t0 = fs_ns();
    while (!fbar_try(bar, parity, hint))
        if (fs_ns() - t0 > limit_ns) return false;
    return true;
}
__device__ __forceinline__ void ftma(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     fs_u32(dst)),
                 "l"(src), "r"(bytes), "r"(fs_u32(bar))
                 : "memory");
}
// consumer-warp barrier on an mbarrier (one arrival per warp); false once a wait gave up
struct FSync {
    uint32_t ph;
    bool ok;
};
template <int W>
__device__ __forceinline__ bool fsync(FreeSmem<W>& sm, FSync& g) {
    __syncwarp();
    if (!g.ok) return false;
    if ((threadIdx.x & 31) == 0) fbar_arrive(&sm.gsync);
    g.ok = __all_sync(0xFFFFFFFFu, fbar_wait(&sm.gsync, g.ph, sm.wait_ns));
    g.ph ^= 1u;
    return g.ok;
}

// ---------------------------------------------------------------------------
// arithmetic
// ---------------------------------------------------------------------------
template <typename TIn>
struct FE;
__device__ __forceinline__ float fmax_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}
template <>
struct FE<__nv_bfloat16> {
    static constexpr int VEC = 8;
    __device__ static void unpack(const uint4& v, float (&x)[8]) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
    // NaN-propagating maximum of the vector (packed)
    __device__ static float vmax(const uint4& v) {
        const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&v.x);
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&v.y);
        const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&v.z);
        const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&v.w);
        const __nv_bfloat162 m = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
        return fmax_nan(__low2float(m), __high2float(m));
    }
    __device__ static float at(const uint4& v, int j) {
        const uint32_t w = j < 2 ? v.x : j < 4 ? v.y : j < 6 ? v.z : v.w;
        return __uint_as_float((j & 1) ? (w & 0xFFFF0000u) : (w << 16));
    }
    __device__ static float load(const __nv_bfloat16* p, int i) {
        return __uint_as_float((uint32_t)reinterpret_cast<const unsigned short*>(p)[i] << 16);
    }
    // the vector as float pairs (element 2k, element 2k + 1)
    __device__ static void pairs(const uint4& v, float2 (&x)[4]) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
    }
};
template <>
struct FE<float> {
    static constexpr int VEC = 4;
    __device__ static void unpack(const uint4& v, float (&x)[4]) {
        x[0] = __uint_as_float(v.x);
        x[1] = __uint_as_float(v.y);
        x[2] = __uint_as_float(v.z);
        x[3] = __uint_as_float(v.w);
    }
    __device__ static float vmax(const uint4& v) {
        return fmax_nan(fmax_nan(__uint_as_float(v.x), __uint_as_float(v.y)),
                        fmax_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
    }
    __device__ static float at(const uint4& v, int j) {
        return __uint_as_float(j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w);
    }
    __device__ static float load(const float* p, int i) { return p[i]; }
    __device__ static void pairs(const uint4& v, float2 (&x)[2]) {
        x[0] = make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
        x[1] = make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
    }
};

// fp32 sum with Kahan compensation: the value is s - c
struct KSum {
    float s, c;
    __device__ __forceinline__ void add(float x) {
        const float y = x - c;
        const float t = s + y;
        c = (t - s) - y;
        s = t;
    }
};
// warp sum of compensated values (an exact two-sum at every level), as a float
__device__ __forceinline__ float warp_ksum(KSum k) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float s2 = __shfl_xor_sync(0xFFFFFFFFu, k.s, o);
        const float c2 = __shfl_xor_sync(0xFFFFFFFFu, k.c, o);
        const float t = k.s + s2;
        const float bb = t - k.s;
        const float e = (k.s - (t - bb)) + (s2 - bb);
        k.c = (k.c + c2) - e;
        k.s = t;
    }
    return k.s - k.c;
}
__device__ __forceinline__ float warp_maxf(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xFFFFFFFFu, x, o));
    return x;
}

// 2^x by the PTX approximate base-2 exponential (relative error about 2^-22),
// results below the normal range flushed to zero
__device__ __forceinline__ float fex2(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float2 fex2x2(float2 x) { return make_float2(fex2(x.x), fex2(x.y)); }

// Unnormalised weight of a logit l of a row with maximum M at c = log2(e) / T:
// 2^(l * c - mc) with mc = fp32(M * c), one FMA (nmc = -mc).  The rounding of
// mc shifts every exponent of the row by the same amount, so it cancels
// against the row's sum, which is formed from the same weights; what remains
// is the FMA's single rounding, relative to l * c - mc.  Every pass, and the
// tail kernel's re-read, use this expression, so a weight is the same number
// wherever it is computed.
__device__ __forceinline__ float row_nmc(float M, float c) { return -(M * c); }
__device__ __forceinline__ float prob_f(float l, float c, float nmc, float inv) { return fex2(fmaf(l, c, nmc)) * inv; }
__device__ __forceinline__ float resid_f(float p, float q) { return fmaxf(p - q, 0.0f); }
// the (top-p renormalised) probability of element id with logit l: zero past
// the row's last kept element `cut` (CUT: the row is filtered; else no test at all)
template <bool CUT>
__device__ __forceinline__ float kept_prob(float l, uint32_t id, float c, float nmc, float inv2, unsigned long long cut) {
    if (CUT && ((unsigned long long)okey32(__float_as_uint(l)) << 32 | (unsigned long long)(~id)) < cut) return 0.0f;
    return fex2(fmaf(l, c, nmc)) * inv2;
}
// is (l, id) at or before the cut element (logit lc, id ic) in (logit desc, id asc) order
__device__ __forceinline__ bool kept_at(float l, uint32_t id, float lc, uint32_t ic) {
    return l > lc || (l == lc && id <= ic);
}

// online softmax state of one row for one thread: running maximum logit m,
// nmc = -fp32(m * c), and the compensated sum of the weights 2^(l * c + nmc).
// When the maximum grows the sum is rescaled by 2^(nmc_new - nmc_old), so it
// stays the sum of the weights at the current nmc.
struct Online {
    float m, nmc;
    KSum s;
    __device__ __forceinline__ void init() {
        m = -INFINITY;
        nmc = 0.0f;
        s = KSum{0.0f, 0.0f};
    }
    __device__ __forceinline__ void raise(float vm, float c) {
        const float n2 = row_nmc(vm, c);
        const float f = m == -INFINITY ? 0.0f : fex2(n2 - nmc);
        s.s *= f;
        s.c *= f;
        m = vm;
        nmc = n2;
    }
    // a whole vector; vm is its NaN-propagating maximum (a NaN row is flagged
    // by the caller and its sums are not used)
    template <typename TIn>
    __device__ __forceinline__ void add_full(const uint4& v, float vm, float c) {
        if (!(vm > -INFINITY)) return;  // only -inf here (or NaN)
        if (vm > m) raise(vm, c);
        float x[FE<TIn>::VEC];
        FE<TIn>::unpack(v, x);
        float acc = 0.0f;
#pragma unroll
        for (int j = 0; j < FE<TIn>::VEC; ++j) acc += fex2(fmaf(x[j], c, nmc));
        s.add(acc);
    }
    // all kFVec vectors of a full tile at once: one rescale, then independent
    // weights (packed pairs) summed as a tree; vm is the NaN-propagating
    // maximum of them all
    template <typename TIn>
    __device__ __forceinline__ void add_tile(const uint4 (&v)[kFVec], float vm, float c) {
        constexpr int H = FE<TIn>::VEC / 2;
        if (!(vm > -INFINITY)) return;
        if (vm > m) raise(vm, c);
        const float2 c2 = make_float2(c, c), n2 = make_float2(nmc, nmc);
        float2 acc[kFVec];
#pragma unroll
        for (int i = 0; i < kFVec; ++i) {
            float2 x[H];
            FE<TIn>::pairs(v[i], x);
#pragma unroll
            for (int k = 0; k < H; ++k) x[k] = fex2x2(__ffma2_rn(x[k], c2, n2));
#pragma unroll
            for (int w = H / 2; w > 0; w >>= 1)
#pragma unroll
                for (int k = 0; k < w; ++k) x[k] = __fadd2_rn(x[k], x[k + w]);
            acc[i] = x[0];
        }
#pragma unroll
        for (int w = kFVec / 2; w > 0; w >>= 1)
#pragma unroll
            for (int i = 0; i < w; ++i) acc[i] = __fadd2_rn(acc[i], acc[i + w]);
        s.add(acc[0].x + acc[0].y);
    }
    // the first `valid` elements of a vector (the ragged end of a row)
    template <typename TIn>
    __device__ __forceinline__ void add_part(const uint4& v, int valid, float c) {
        float x[FE<TIn>::VEC];
        FE<TIn>::unpack(v, x);
        float vm = -INFINITY;
#pragma unroll
        for (int j = 0; j < FE<TIn>::VEC; ++j)
            if (j < valid) vm = fmaxf(vm, x[j]);
        if (!(vm > -INFINITY)) return;
        if (vm > m) raise(vm, c);
        float acc = 0.0f;
#pragma unroll
        for (int j = 0; j < FE<TIn>::VEC; ++j)
            if (j < valid) acc += fex2(fmaf(x[j], c, nmc));
        s.add(acc);
    }
};

// maximum and rescaled sum of one row over the lanes of a warp
__device__ __forceinline__ void warp_online(const Online& o, float c, float* wm, float* ws) {
    *wm = warp_maxf(o.m);
    KSum k = o.s;
    if (*wm > -INFINITY) {
        const float f = o.m == -INFINITY ? 0.0f : fex2(row_nmc(*wm, c) - o.nmc);
        k.s *= f;
        k.c *= f;
    } else {
        k = KSum{0.0f, 0.0f};
    }
    *ws = warp_ksum(k);
}

// Statistics of one row over all consumer warps, computed by every warp from
// the seven warps' (maximum, rescaled sum) pairs in red[w][col], [col + 1]:
// lane w rescales warp w's sum to the common maximum, and the warp adds them
// with a compensated sum.  M = -inf when the row has no finite logit.
template <int W>
__device__ __forceinline__ void combine_stats(const float (*red)[8], int col, float c, int lane, float* M, float* S) {
    const float wm = lane < W ? red[lane][col] : -INFINITY;
    const float m = warp_maxf(wm);
    float x = 0.0f;
    if (m > -INFINITY && wm > -INFINITY) x = red[lane][col + 1] * fex2(row_nmc(m, c) - row_nmc(wm, c));
    *M = m;
    *S = cf_val(warp_cf_sum(CF{x, 0.0f}));
}

// The weight 2^(l * chi + nmc) of prob_f / kept_prob, with chi = fp32(c),
// computed to about fp32 rounding of the exact 2^((l - M) * c - delta) for
// any l <= M, where c = chi + clo is log2(e) / T as a float pair and delta =
// fp32(M * chi) - M * chi is the row's common shift (so the weight matches the
// row's sum).  The difference l - M is formed exactly (two-sum), the product
// with c by an FMA two-product, -delta = fma(M, chi, nmc) exactly, the integer
// part n is applied exactly and only the fraction f in [-1/2, 1/2] goes
// through exp2f.  Results below 2^-126 are 0.  Used for the two probabilities
// of the acceptance test.
__device__ __forceinline__ float exp2_prod(float l, float M, float chi, float clo, float nmc) {
    const float d = l - M;
    const float p = d * chi;
    const float n = rintf(p);
    if (!(n >= -126.0f)) return 0.0f;  // also l = -inf
    const float bb = d - l;
    const float dlo = (l - (d - bb)) + (-M - bb);  // l - M = d + dlo exactly
    const float e = fmaf(d, chi, -p);               // d * chi = p + e exactly
    const float f = (p - n) + ((e + fmaf(M, chi, nmc)) + fmaf(d, clo, dlo * chi));
    return exp2f(f) * __int_as_float((int)(n + 127.0f) << 23);
}

// ---------------------------------------------------------------------------
// nucleus cut helpers
// ---------------------------------------------------------------------------
// (key << 32 | ~id): descending order is logit descending, then id ascending
__device__ __forceinline__ unsigned long long ncomp(float x, uint32_t id) {
    return ((unsigned long long)okey32(__float_as_uint(x)) << 32) | (unsigned long long)(~id);
}
// Add the mass of probability p (0 <= p <= 1) to bin `bin` of a split
// histogram h[2][n].  The parts of m = floor(p * 2^40) come from fp32 alone:
// with t = p * 2^30 (exact), hi = trunc(t) and lo = floor((t - hi) * 2^10), where
// t - hi is exact, so hi * 2^10 + lo = m exactly (the same integers as a 64-bit
// conversion, which would run on this GPU's narrow fp64 pipe).
template <int N>
__device__ __forceinline__ void mass_add(uint32_t (&h)[2][N], int bin, float p) {
    static_assert(kMassLoBits == 10, "the split below is for 2^40 = 2^30 * 2^10");
    const float t = p * 1073741824.0f;  // 2^30
    const float hf = truncf(t);
    const uint32_t hi = (uint32_t)hf;
    const uint32_t lo = (uint32_t)((t - hf) * 1024.0f);
    if (hi) atomicAdd(&h[0][bin], hi);
    if (lo) atomicAdd(&h[1][bin], lo);
}
template <int N>
__device__ __forceinline__ unsigned long long mass_of(const uint32_t (&h)[2][N], int bin) {
    return ((unsigned long long)h[0][bin] << kMassLoBits) + h[1][bin];
}

// For the warp: the first bin of h[0..n) (n a multiple of 32) at which the
// running mass reaches target, and the mass before it; if the total falls
// short (rounding), the last bin with mass.  -1 when h is empty.
template <int N>
__device__ int warp_cross(const uint32_t (&h)[2][N], unsigned long long target, unsigned long long* before, int lane) {
    constexpr int per = N / 32;
    const int b0 = lane * per;
    unsigned long long own = 0;
    for (int i = 0; i < per; ++i) own += mass_of(h, b0 + i);
    unsigned long long x = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
    }
    const unsigned long long excl = x - own;
    int bin = -1;
    unsigned long long bef = 0;
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, own > 0 && x >= target);
    const unsigned nz = __ballot_sync(0xFFFFFFFFu, own > 0);
    int src = 0;
    if (hit) {
        src = __ffs(hit) - 1;
        if (lane == src) {
            unsigned long long run = excl;
            for (int i = 0; i < per; ++i) {
                const unsigned long long mi = mass_of(h, b0 + i);
                if (mi > 0 && run + mi >= target) {
                    bin = b0 + i;
                    bef = run;
                    break;
                }
                run += mi;
            }
        }
    } else if (nz) {
        src = 31 - __clz(nz);
        if (lane == src) {
            unsigned long long run = excl;
            for (int i = 0; i < per; ++i) {
                const unsigned long long mi = mass_of(h, b0 + i);
                if (mi > 0) {
                    bin = b0 + i;
                    bef = run;
                }
                run += mi;
            }
        }
    }
    bin = __shfl_sync(0xFFFFFFFFu, bin, src);
    *before = __shfl_sync(0xFFFFFFFFu, bef, src);
    return bin;
}

// For the warp: sort the n collected crossing elements of a row (key desc,
// id asc) and walk them from the mass before their fine bin to the first one
// whose running mass reaches P (the nucleus' last token).  Returns false if
// there are too many (or none) to decide here.
__device__ bool warp_cut(unsigned long long* list, int n, unsigned long long base, double P, float c, float nmc,
                         float inv, uint32_t* cut_key, uint32_t* cut_id, double* kept, int lane) {
    if (n < 1 || n > kNCap) return false;
    warp_sort(list, n, list, true, 0ull, lane);
    double cum = (double)base / (double)kMassScale;
    int idx = -1;
    double K = 0.0;
    for (int c0 = 0; c0 < n && idx < 0; c0 += 32) {
        const int j = c0 + lane;
        const double p = j < n ? (double)prob_f(key_value32((uint32_t)(list[j] >> 32)), c, nmc, inv) : 0.0;
        double x = p;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const double y = __shfl_up_sync(0xFFFFFFFFu, x, o);
            if (lane >= o) x += y;
        }
        const unsigned hit = __ballot_sync(0xFFFFFFFFu, j < n && cum + x >= P);
        if (hit) {
            const int l = __ffs(hit) - 1;
            idx = c0 + l;
            K = cum + __shfl_sync(0xFFFFFFFFu, x, l);
        }
        cum += __shfl_sync(0xFFFFFFFFu, x, 31);
    }
    if (idx < 0) {  // rounding: the running mass stops just short of P
        idx = n - 1;
        K = cum;
    }
    *cut_key = (uint32_t)(list[idx] >> 32);
    *cut_id = ~(uint32_t)list[idx];
    *kept = K;
    return true;
}

// Bin coordinate of a logit: t = -8 * (l * c + nmc), the distance below the row
// maximum in 1/8 log2 units, from the weight's own exponent (the scaling by 8
// is exact).  It is the same number in every pass, and monotone in l, so the
// bins partition the row in (logit desc) order consistently.  Coarse bin
// (int)t for t < 512 (t may be a rounding below 0 at the maximum: bin 0);
// fine bin (int)((t - b1) * 512) inside coarse bin b1.
//
// One tile of a nucleus pass for row r (c, nmc = row_nmc(M, c), 1/sum inv);
// the thread holds the vectors vbase + 32 i of the segment (FULL: all whole).
// Pass 1 adds the masses to the coarse histogram, pass 2 those of the
// crossing coarse bin to the fine histogram, pass 3 collects the elements of
// the crossing fine bin.  Passes 2 and 3 test a bin by two compares on t and
// convert only the few logits inside it.
template <typename TIn, bool FULL, int W>
__device__ __forceinline__ void nucleus_tile(FreeSmem<W>& sm, const uint4 (&v)[kFVec], int n, int vbase, int col,
                                             int pass, int r, float c, float nmc, float inv) {
    using F = FE<TIn>;
    constexpr float kTMax = (float)kNB1;  // t >= 512: more than kNDmax below the maximum
    static_assert(kNB1 * 8 == (int)(kNDmax * 64), "coarse bins are 1/8 log2 unit");
    const int b1 = pass >= 2 ? sm.nb[r][0] : -1;
    const int b2 = pass >= 3 ? sm.nb[r][1] : -1;
    const float lo1 = b1 <= 0 ? -INFINITY : (float)b1;            // coarse bin b1 is [lo1, hi1)
    const float hi1 = b1 >= kNB1 - 1 ? kTMax : (float)(b1 + 1);
    const float base1 = (float)max(b1, 0);
#pragma unroll
    for (int i = 0; i < kFVec; ++i) {
        const int e0 = (vbase + 32 * i) * F::VEC;
        const int valid = FULL ? F::VEC : min(F::VEC, n - e0);
        if (!FULL && valid <= 0) continue;
        float x[F::VEC];
        F::unpack(v[i], x);
#pragma unroll
        for (int j = 0; j < F::VEC; ++j) {
            if (!FULL && j >= valid) continue;
            const float e = fmaf(x[j], c, nmc);  // the weight's exponent
            const float t = -8.0f * e;
            if (pass == 1) {
                if (t < kTMax) mass_add(sm.h1[r], (int)t, fex2(e) * inv);
            } else if (t >= lo1 && t < hi1) {
                const int sb = min(kNB2 - 1, max(0, (int)((t - base1) * (float)kNB2)));
                if (pass == 2) {
                    mass_add(sm.h2[r], sb, fex2(e) * inv);
                } else if (sb == b2) {
                    const int slot = atomicAdd(&sm.ncnt[r], 1);
                    if (slot < kNCap) sm.list[r][slot] = ncomp(x[j], (uint32_t)(col + e0 + j));
                }
            }
        }
    }
}

template <typename TIn, bool TMA, int W>
__global__ void __launch_bounds__(FGeo<W>::kThreads, FGeo<W>::kCtasPerSm) free_kernel(Args a) {
    using F = FE<TIn>;
    constexpr int kFWarps = W;
    constexpr int kFConsumers = FGeo<W>::kConsumers;
    constexpr int TS = FGeo<W>::kSegBytes / (int)sizeof(TIn);  // elements per segment (tile)
    extern __shared__ __align__(128) uint8_t fsm_raw[];
    FreeSmem<W>& sm = *reinterpret_cast<FreeSmem<W>*>(fsm_raw);
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int V = a.V, G = a.G;
    const int ntiles = (V + TS - 1) / TS;
    // No unit on this path: leave at once, without waiting for the kernels before
    // this one.  The count is the plan's, final and visible here: this kernel is
    // launched only once every CTA of the previous one has passed its own wait,
    // which the plan's completion precedes.  Nothing here reads their results.
    if (a.counts[kCntFreeUnits] == 0u) return;

    if (t == 0) {
        for (int s = 0; s < kFStages; ++s) {
            fbar_init(&sm.full[s], 1);
            fbar_init(&sm.empty[s], kFWarps);
        }
        fbar_init(&sm.gsync, kFWarps);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        sm.wait_ns = a.wait_ns;
    }
    __syncthreads();
    grid_dependency_wait();  // the previous kernels of the call (the plan's lists)
    grid_dependents_go();
    const uint32_t n_units = a.counts[kCntFreeUnits];
    if (n_units == 0) return;  // no sequence takes this path (the same value for every thread)

    if (warp == kFWarps) {
        // ------------------------------ producer ------------------------------
        if (!TMA || lane == 0) {
            int stage = 0;
            uint32_t ph = 1;  // fresh empty barriers count as released
            int issued[kFStages];
#pragma unroll
            for (int s = 0; s < kFStages; ++s) issued[s] = -1;
            bool ok = true;
            while (ok) {
                uint32_t w = 0;
                if (lane == 0) w = atomicAdd(&a.counts[kCntFreeNext], 1u);
                if (!TMA) w = __shfl_sync(0xFFFFFFFFu, w, 0);
                if (w >= n_units) break;
                const uint32_t item = a.free_units[w];
                const int b = (int)(item >> 8), u = (int)(item & 0xFFu);
                const SeqInfo si = a.seq[b];
                const bool pair = !a.gumbel && u < si.gamma;  // shared noise reads the target row only
                const bool nucleus = si.P < 1.0f;
                const TIn* trow = (const TIn*)a.target + ((size_t)b * (G + 1) + u) * (size_t)V;
                const TIn* drow = (const TIn*)a.draft + ((size_t)b * G + u) * (size_t)V;
                // passes: the statistics (not needed by shared noise without top-p), the
                // nucleus passes when top-p < 1, the final pass
                const int npass = nucleus ? 5 : (a.gumbel ? 1 : 2);
                for (int pi = 0; pi < npass && ok; ++pi) {
                    const int pass = nucleus ? pi : (pi + 1 == npass ? kPassFinal : 0);
                    for (int tile = 0; tile < ntiles && ok; ++tile) {
                        const int col = tile * TS, n = min(TS, V - col);
                        if (!fbar_wait(&sm.empty[stage], ph, sm.wait_ns)) {
                            ok = false;
                            break;
                        }
                        if (lane == 0) {
                            sm.hdr[stage] = make_int4((int)w, pass, tile, n);
                            sm.uhdr[stage] = make_int4((int)item, si.gamma, __float_as_int(si.T), __float_as_int(si.P));
                            sm.lhdr[stage] = si.L;
                        }
                        if (TMA) {
                            const uint32_t bytes = (uint32_t)(n * sizeof(TIn));
                            fbar_expect(&sm.full[stage], pair ? 2u * bytes : bytes);
                            ftma(sm.buf[stage][0], trow + col, bytes, &sm.full[stage]);
                            if (pair) ftma(sm.buf[stage][1], drow + col, bytes, &sm.full[stage]);
                            issued[stage] = (int)(ph ^ 1u);
                        } else {
                            TIn* d0 = reinterpret_cast<TIn*>(sm.buf[stage][0]);
                            TIn* d1 = reinterpret_cast<TIn*>(sm.buf[stage][1]);
                            for (int i = lane; i < n; i += 32) {
                                d0[i] = trow[col + i];
                                if (pair) d1[i] = drow[col + i];
                            }
                            __syncwarp();
                            if (lane == 0) fbar_arrive(&sm.full[stage]);
                        }
                        if (++stage == kFStages) {
                            stage = 0;
                            ph ^= 1u;
                        }
                    }
                }
            }
            if (ok && fbar_wait(&sm.empty[stage], ph, sm.wait_ns)) {
                if (lane == 0) {
                    sm.hdr[stage] = make_int4(-1, 0, 0, 0);
                    fbar_arrive(&sm.full[stage]);
                }
            } else if (lane == 0) {
                atomicOr(&a.counts[kCntError], 1u);
                // let every copy already issued land (with the full limit: a copy in
                // flight must not outlive the CTA)
                for (int s = 0; s < kFStages; ++s)
                    if (issued[s] >= 0) (void)fbar_wait(&sm.full[s], (uint32_t)issued[s], kWaitLimitNs);
            }
        }
        return;
    }


    // ------------------------------ consumers ------------------------------
    int stage = 0;
    uint32_t ph = 0;
    FSync g{0u, true};
    const int vbase = warp * (32 * kFVec) + lane;  // this thread's vectors of a segment: vbase + 32 i
    const size_t nblk = (size_t)a.free_nblk;
    int b = 0, u = 0, par = 1, cur_w = -1;
    float cg = 1.0f;                // 1 / T (shared noise: the score is l / T + g)
    unsigned long long gbest = 0ull;  // shared noise: this thread's best (score, id) key of the unit
    float gbs = -INFINITY;            // and its score
    bool pair = false, nf = false, dead = false;
    bool nuc = false, fall = false;  // top-p < 1; the unit goes to the cluster kernel
    float c = 1.0f, Pf = 1.0f, invl = 1.0f;  // invl: 1 / lenience (alpha = sum_x min(q, p * invl))
    Online op, oq;
    float Mp = 0.0f, Mq = 0.0f, Sp = 0.0f, Sq = 0.0f, invp = 0.0f, invq = 0.0f, invp2 = 0.0f, invq2 = 0.0f;
    float nmcp = 0.0f, nmcq = 0.0f;  // row_nmc of each row's maximum
    unsigned long long cutp = 0ull, cutq = 0ull;  // last kept element of each row (0: keep all)
    KSum alpha{0.0f, 0.0f};
    // the unit's record for the tail kernel (one thread writes it)
    auto write_rec = [&](int w, uint32_t flags) {
        FreeRec& R = a.free_rec[w];
        R.Mp = Mp;
        R.Mq = Mq;
        R.invp = invp2;
        R.invq = invq2;
        R.cutp = cutp;
        R.cutq = cutq;
        R.flags = flags;
        for (int i = kFWarps; i < kFreeWarpsWide; ++i) R.alpha[i] = 0.0f;
    };
    while (true) {
        if (!__all_sync(0xFFFFFFFFu, fbar_wait(&sm.full[stage], ph, sm.wait_ns))) {
            g.ok = false;
            break;
        }
        const int4 h = sm.hdr[stage];
        if (h.x < 0) break;
        const int w = h.x, pass = h.y, tile = h.z, n = h.w;
        const int col = tile * TS;
        if (w != cur_w) {  // a new unit (from the producer's header: no global loads)
            cur_w = w;
            const int4 uh = sm.uhdr[stage];  // read before the stage is released
            b = uh.x >> 8;
            u = uh.x & 0xFF;
            pair = !a.gumbel && u < uh.y;
            const float T = __int_as_float(uh.z);
            c = 1.4426950408889634f / T;
            cg = 1.0f / T;
            gbest = 0ull;
            gbs = -INFINITY;
            dead = false;
            Pf = __int_as_float(uh.w);
            invl = lenience_inv(sm.lhdr[stage]);
            nuc = Pf < 1.0f;
            fall = false;
            cutp = cutq = 0ull;
            op.init();
            oq.init();
            nf = false;
            alpha = KSum{0.0f, 0.0f};
            par ^= 1;
        }
        uint4 vp[kFVec], vq[kFVec];
        const uint4* sp4 = reinterpret_cast<const uint4*>(sm.buf[stage][0]);
        const uint4* sq4 = reinterpret_cast<const uint4*>(sm.buf[stage][1]);
#pragma unroll
        for (int i = 0; i < kFVec; ++i) {
            vp[i] = sp4[vbase + 32 * i];
            vq[i] = pair ? sq4[vbase + 32 * i] : make_uint4(0u, 0u, 0u, 0u);
        }
        __syncwarp();
        if (lane == 0) fbar_arrive(&sm.empty[stage]);
        if (++stage == kFStages) {
            stage = 0;
            ph ^= 1u;
        }

        if (pass == 0) {
            // ---- pass 0: online maximum and sum; non-finite logits flag the sequence
            if (n == TS) {  // a full tile: every vector of this thread is whole
                float mp = -INFINITY, mq = -INFINITY;
#pragma unroll
                for (int i = 0; i < kFVec; ++i) {
                    mp = fmax_nan(mp, F::vmax(vp[i]));
                    if (pair) mq = fmax_nan(mq, F::vmax(vq[i]));
                }
                nf |= isnan(mp) || mp == INFINITY || isnan(mq) || mq == INFINITY;
                op.add_tile<TIn>(vp, mp, c);
                if (pair) oq.add_tile<TIn>(vq, mq, c);
            } else {
#pragma unroll
                for (int i = 0; i < kFVec; ++i) {
                    const int e0 = (vbase + 32 * i) * F::VEC;
                    const int valid = min(F::VEC, n - e0);
                    if (valid <= 0) continue;
                    if (valid == F::VEC) {
                        const float mp = F::vmax(vp[i]);
                        nf |= isnan(mp) || mp == INFINITY;
                        op.add_full<TIn>(vp[i], mp, c);
                        if (pair) {
                            const float mq = F::vmax(vq[i]);
                            nf |= isnan(mq) || mq == INFINITY;
                            oq.add_full<TIn>(vq[i], mq, c);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < F::VEC; ++j)
                            if (j < valid) {
                                const float x = F::at(vp[i], j);
                                nf |= isnan(x) || x == INFINITY;
                                if (pair) {
                                    const float y = F::at(vq[i], j);
                                    nf |= isnan(y) || y == INFINITY;
                                }
                            }
                        op.add_part<TIn>(vp[i], valid, c);
                        if (pair) oq.add_part<TIn>(vq[i], valid, c);
                    }
                }
            }
            if (tile == ntiles - 1) {
                float wm, ws, wm2, ws2;
                warp_online(op, c, &wm, &ws);
                warp_online(oq, c, &wm2, &ws2);
                const bool wnf = __any_sync(0xFFFFFFFFu, nf);
                float(*red)[8] = sm.red[par];
                if (lane == 0) {
                    red[warp][0] = wm;
                    red[warp][1] = ws;
                    red[warp][2] = wm2;
                    red[warp][3] = ws2;
                    red[warp][4] = wnf ? 1.0f : 0.0f;
                }
                // the coarse histograms start empty (nothing reads them between
                // the previous unit's cut and this barrier)
                if (nuc)
                    for (int i = t; i < 4 * kNB1; i += kFConsumers) (&sm.h1[0][0][0])[i] = 0u;
                if (!fsync(sm, g)) break;
                // every warp combines the seven warps' statistics itself; red is
                // double-buffered by unit, so no second barrier is needed
                combine_stats<W>(red, 0, c, lane, &Mp, &Sp);
                combine_stats<W>(red, 2, c, lane, &Mq, &Sq);
                const bool anynf = __any_sync(0xFFFFFFFFu, lane < kFWarps && red[lane][4] != 0.0f);
                // a row with a NaN or +inf logit, or without any finite one
                dead = anynf || !(Mp > -INFINITY) || (pair && !(Mq > -INFINITY));
                invp = dead ? 0.0f : 1.0f / Sp;
                invq = (dead || !pair) ? 0.0f : 1.0f / Sq;
                nmcp = row_nmc(Mp, c);
                nmcq = pair ? row_nmc(Mq, c) : 0.0f;
                invp2 = invp;
                invq2 = invq;
                if (t == 0 && (dead || !nuc)) write_rec(w, dead ? kRecDead : 0u);
            }
            continue;
        }

        if (pass < kPassFinal) {
            // ---- nucleus passes: the last kept token of each row (top-p < 1)
            if (dead) continue;
            if (n == TS) {
                nucleus_tile<TIn, true, W>(sm, vp, n, vbase, col, pass, 0, c, nmcp, invp);
                if (pair) nucleus_tile<TIn, true, W>(sm, vq, n, vbase, col, pass, 1, c, nmcq, invq);
            } else {
                nucleus_tile<TIn, false, W>(sm, vp, n, vbase, col, pass, 0, c, nmcp, invp);
                if (pair) nucleus_tile<TIn, false, W>(sm, vq, n, vbase, col, pass, 1, c, nmcq, invq);
            }
            if (tile != ntiles - 1) continue;
            if (!fsync(sm, g)) break;
            const unsigned long long target = (unsigned long long)((double)Pf * (double)kMassScale);
            if (warp < (pair ? 2 : 1)) {
                const int r = warp;
                unsigned long long bef = 0ull;
                if (pass == 1) {
                    const int bin = warp_cross(sm.h1[r], target, &bef, lane);
                    if (lane == 0) {
                        sm.nb[r][0] = bin;
                        sm.nbase[r] = bef;
                    }
                } else if (pass == 2) {
                    const unsigned long long base = sm.nbase[r];
                    const int bin = sm.nb[r][0] < 0 ? -1
                                                    : warp_cross(sm.h2[r], target > base ? target - base : 0ull,
                                                                 &bef, lane);
                    if (lane == 0) {
                        sm.nb[r][1] = bin;
                        sm.nbase[r] = base + bef;
                    }
                } else {
                    uint32_t ck = 0u, ci = 0u;
                    double K = 0.0;
                    const int cnt = sm.ncnt[r];
                    const bool ok = sm.nb[r][1] >= 0 &&
                                    warp_cut(sm.list[r], min(cnt, kNCap + 1), sm.nbase[r], (double)Pf,
                                             c, r == 0 ? nmcp : nmcq, r == 0 ? invp : invq, &ck, &ci, &K, lane);
                    if (lane == 0) {
                        sm.cut_key[r] = ck;
                        sm.cut_id[r] = ci;
                        sm.kinv[r] = ok ? (float)(1.0 / ((double)(r == 0 ? Sp : Sq) * K)) : -1.0f;
                    }
                }
            }
            if (pass == 1)  // the fine histograms start empty
                for (int i = t; i < 4 * kNB2; i += kFConsumers) (&sm.h2[0][0][0])[i] = 0u;
            if (pass == 2 && t < 2) sm.ncnt[t] = 0;
            if (!fsync(sm, g)) break;
            if (pass == 3) {
                fall = sm.kinv[0] < 0.0f || (pair && sm.kinv[1] < 0.0f);
                if (!fall) {
                    cutp = ((unsigned long long)sm.cut_key[0] << 32) | (unsigned long long)(~sm.cut_id[0]);
                    invp2 = sm.kinv[0];
                    if (pair) {
                        cutq = ((unsigned long long)sm.cut_key[1] << 32) | (unsigned long long)(~sm.cut_id[1]);
                        invq2 = sm.kinv[1];
                    }
                }
                if (t == 0) {
                    write_rec(w, fall ? kRecFall : 0u);
                    if (fall) {  // too many logits at the cut to sort here: the cluster kernel takes the unit
                        const uint32_t slot = atomicAdd(&a.counts[kCntDenseUnits], 1u);
                        a.dense_units[slot] = a.free_units[w];
                    }
                }
            }
            continue;
        }
        if (fall || dead) continue;  // nothing more to sum (the cluster kernel, or the tail kernel's flags)

        if (a.gumbel) {
            // ---- shared noise ("Speculative decoding: the art of guessing well", section
            // 共享噪声的采样): the target's token is the argmax over the kept tokens of
            // l / T + g, g the Philox noise of the token at this position (ties: lower id)
            // The thread's Philox blocks of this tile first, in straight-line code (the
            // independent 10-round chains interleave); then each token: it beats the
            // thread's best only if g(u) >= D = best - l / T, i.e. u >= U(D) =
            // exp(-exp(-D)) (g increases with u), and no noise on the 24-bit grid exceeds
            // g(1 - 2^-25) = 25 ln 2 = 17.33 (kGMax adds a margin).  U is formed with fast
            // base-2 exponentials (error below 1e-6); tokens with u below U - 1e-5 are
            // rejected without their exact noise.  Exact: a rejected token scores strictly
            // below the thread's best.
            constexpr float kGMax = 17.5f;
            constexpr int NB = kFVec * F::VEC / 4;  // Philox blocks per thread per tile
            const float lcp = key_value32((uint32_t)(cutp >> 32));
            const uint32_t icp = ~(uint32_t)cutp;
            const uint32_t k0 = (uint32_t)a.seed, k1 = (uint32_t)(a.seed >> 32);
            uint4 wq[NB];
#pragma unroll
            for (int i = 0; i < kFVec; ++i)
#pragma unroll
                for (int h = 0; h < F::VEC / 4; ++h) {
                    const uint32_t id0 = (uint32_t)(col + (vbase + 32 * i) * F::VEC);  // a multiple of 4
                    wq[i * (F::VEC / 4) + h] = philox4((uint32_t)b, (uint32_t)(u + 1), 2u, (id0 >> 2) + h, k0, k1);
                }
#pragma unroll
            for (int i = 0; i < kFVec; ++i) {
                const int e0 = (vbase + 32 * i) * F::VEC;
                const int valid = min(F::VEC, n - e0);
                if (valid <= 0) continue;
                float x[F::VEC];
                F::unpack(vp[i], x);
                const uint32_t id0 = (uint32_t)(col + e0);
#pragma unroll
                for (int j = 0; j < F::VEC; ++j) {
                    if (j >= valid) continue;
                    const uint4 w4 = wq[i * (F::VEC / 4) + j / 4];
                    const uint32_t wj = (j & 3) == 0 ? w4.x : (j & 3) == 1 ? w4.y : (j & 3) == 2 ? w4.z : w4.w;
                    const float xv = x[j];
                    const uint32_t id = id0 + (uint32_t)j;
                    nf |= (xv != xv) || xv == INFINITY;
                    if (!(xv > -INFINITY)) continue;  // p = 0 (and NaN)
                    if (nuc && !kept_at(xv, id, lcp, icp)) continue;
                    const float s0 = xv * cg;
                    const float D = gbs - s0;
                    if (!(D < kGMax)) continue;
                    const float uf = fmaf((float)(wj >> 8), 5.9604644775390625e-8f, 2.98023223876953125e-8f);
                    if (uf < fex2(-fex2(-D * 1.44269504088896341f) * 1.44269504088896341f) - 1e-5f) continue;
                    const float sc = s0 + gumbel_of_word(wj);
                    const unsigned long long kk = score_key(sc, id);
                    if (kk > gbest) {
                        gbest = kk;
                        gbs = sc;
                    }
                }
            }
            if (tile == ntiles - 1) {
                unsigned long long bk = gbest;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const unsigned long long y = __shfl_xor_sync(0xFFFFFFFFu, bk, o);
                    bk = y > bk ? y : bk;
                }
                const bool wnf = __any_sync(0xFFFFFFFFu, nf);
                if (lane == 0) {  // this warp's best key: high word (0xFFFFFFFF: a NaN or +inf seen), id
                    float* rrow = a.free_blk + (size_t)w * 2 * nblk;
                    rrow[warp] = __uint_as_float(wnf ? 0xFFFFFFFFu : (uint32_t)(bk >> 32));
                    rrow[nblk + warp] = __uint_as_float((uint32_t)score_key_id(bk));
                }
            }
            continue;
        }

        // ---- final pass: alpha and the residual weights, summed per block
        float tr = 0.0f, tp = 0.0f;
        // the per-element work, specialised on whether the rows are filtered (one
        // branch per tile instead of a test per element)
        auto final_tile = [&](auto cut_on) {
            constexpr bool CUT = decltype(cut_on)::value;
#pragma unroll
            for (int i = 0; i < kFVec; ++i) {
                const int e0 = (vbase + 32 * i) * F::VEC;
                const int valid = min(F::VEC, n - e0);
                if (valid <= 0) continue;
                float xp[F::VEC], xq[F::VEC];
                F::unpack(vp[i], xp);
                F::unpack(vq[i], xq);
                float am = 0.0f;
                if (pair) {
                    float ma[F::VEC], ra[F::VEC], pa[F::VEC];
#pragma unroll
                    for (int j = 0; j < F::VEC; ++j) {
                        const uint32_t id = (uint32_t)(col + e0 + j);
                        const float p = j < valid ? kept_prob<CUT>(xp[j], id, c, nmcp, invp2, cutp) : 0.0f;
                        const float q = j < valid ? kept_prob<CUT>(xq[j], id, c, nmcq, invq2, cutq) : 0.0f;
                        ma[j] = accept_mass(p, q, invl);
                        ra[j] = resid_f(p, q);
                        pa[j] = p;
                    }
#pragma unroll
                    for (int w2 = F::VEC / 2; w2 > 0; w2 >>= 1)
#pragma unroll
                        for (int j = 0; j < w2; ++j) {
                            ma[j] += ma[j + w2];
                            ra[j] += ra[j + w2];
                            pa[j] += pa[j + w2];
                        }
                    am = ma[0];
                    tr += ra[0];
                    tp += pa[0];
                } else {
#pragma unroll
                    for (int j = 0; j < F::VEC; ++j)
                        if (j < valid) tp += kept_prob<CUT>(xp[j], (uint32_t)(col + e0 + j), c, nmcp, invp2, cutp);
                }
                alpha.add(am);
                if (a.p_out || a.q_out) {  // debug outputs
#pragma unroll
                    for (int j = 0; j < F::VEC; ++j)
                        if (j < valid) {
                            if (a.p_out)
                                a.p_out[((size_t)b * (G + 1) + u) * V + col + e0 + j] =
                                    kept_prob<CUT>(xp[j], (uint32_t)(col + e0 + j), c, nmcp, invp2, cutp);
                            if (a.q_out && pair)
                                a.q_out[((size_t)b * G + u) * V + col + e0 + j] =
                                    kept_prob<CUT>(xq[j], (uint32_t)(col + e0 + j), c, nmcq, invq2, cutq);
                        }
                }
            }
        };
        // a full tile without the debug outputs: packed pairs, no bounds per element;
        // the sums run over the thread's pairs in order
        auto final_fast = [&](auto cut_on, auto len_on) {
            constexpr bool CUT = decltype(cut_on)::value;
            constexpr bool LEN = decltype(len_on)::value;  // lenience < 1: alpha term min(q, p / l)
            constexpr int H = F::VEC / 2;
            const float2 c2 = make_float2(c, c), np2 = make_float2(nmcp, nmcp), nq2 = make_float2(nmcq, nmcq);
            const float2 ip2 = make_float2(invp2, invp2), iq2 = make_float2(invq2, invq2);
            const float2 m1 = make_float2(-1.0f, -1.0f);
            // the cut element of each row as (logit, id)
            const float lcp = key_value32((uint32_t)(cutp >> 32)), lcq = key_value32((uint32_t)(cutq >> 32));
            const uint32_t icp = ~(uint32_t)cutp, icq = ~(uint32_t)cutq;
            float2 am = make_float2(0.0f, 0.0f), ar = am, ap = am;
#pragma unroll
            for (int i = 0; i < kFVec; ++i) {
                float2 xp[H], xq[H];
                F::pairs(vp[i], xp);
                if (pair) F::pairs(vq[i], xq);
                const uint32_t id0 = (uint32_t)(col + (vbase + 32 * i) * F::VEC);
#pragma unroll
                for (int k = 0; k < H; ++k) {
                    float2 p = __fmul2_rn(fex2x2(__ffma2_rn(xp[k], c2, np2)), ip2);
                    if (CUT) {
                        if (!kept_at(xp[k].x, id0 + 2 * k, lcp, icp)) p.x = 0.0f;
                        if (!kept_at(xp[k].y, id0 + 2 * k + 1, lcp, icp)) p.y = 0.0f;
                    }
                    if (pair) {
                        float2 q = __fmul2_rn(fex2x2(__ffma2_rn(xq[k], c2, nq2)), iq2);
                        if (CUT) {
                            if (!kept_at(xq[k].x, id0 + 2 * k, lcq, icq)) q.x = 0.0f;
                            if (!kept_at(xq[k].y, id0 + 2 * k + 1, lcq, icq)) q.y = 0.0f;
                        }
                        const float2 d = __ffma2_rn(q, m1, p);  // p - q, one rounding
                        if (LEN)
                            am = __fadd2_rn(am, make_float2(accept_mass(p.x, q.x, invl), accept_mass(p.y, q.y, invl)));
                        else
                            am = __fadd2_rn(am, make_float2(fminf(p.x, q.x), fminf(p.y, q.y)));
                        ar = __fadd2_rn(ar, make_float2(fmaxf(d.x, 0.0f), fmaxf(d.y, 0.0f)));
                    }
                    ap = __fadd2_rn(ap, p);
                }
            }
            tr = ar.x + ar.y;
            tp = ap.x + ap.y;
            alpha.add(am.x + am.y);
        };
        if (n == TS && !(a.p_out || a.q_out)) {
            if (invl != 1.0f) {
                if (nuc)
                    final_fast(std::true_type{}, std::true_type{});
                else
                    final_fast(std::false_type{}, std::true_type{});
            } else if (nuc) {
                final_fast(std::true_type{}, std::false_type{});
            } else {
                final_fast(std::false_type{}, std::false_type{});
            }
        } else if (nuc) {
            final_tile(std::true_type{});
        } else {
            final_tile(std::false_type{});
        }
        // this warp's block of the tile: sums of r (pairs only) and of p, in the record
        const float wtr = warp_ksum(KSum{tr, 0.0f}), wtp = warp_ksum(KSum{tp, 0.0f});
        if (lane == 0) {
            float* blk = a.free_blk + (size_t)w * 2 * nblk + (size_t)tile * kFWarps + warp;
            if (pair) blk[0] = wtr;
            blk[nblk] = wtp;
        }
        if (tile == ntiles - 1 && pair) {
            const float wa = warp_ksum(alpha);
            if (lane == 0) a.free_rec[w].alpha[warp] = wa;
        }
    }
    if (!g.ok && lane == 0) atomicOr(&a.counts[kCntError], 1u);
}

// The residual / bonus draw, the acceptance test and the outputs of the free
// kernel's units, a warp per unit, from the units' records.
template <typename TIn>
__global__ void __launch_bounds__(32 * kTailWarps) free_tail_kernel(Args a) {
    using F = FE<TIn>;
    constexpr int BS = kFreeBlockBytes / (int)sizeof(TIn);  // elements per block
    constexpr int CH = 32 * F::VEC;                         // a block is read in chunks of VEC per lane
    constexpr int NCH = BS / CH;
    static_assert(NCH * CH == BS, "block geometry");
    const int lane = threadIdx.x & 31;
    if (a.counts[kCntFreeUnits] == 0u) return;  // no unit: no wait (the plan's count, as in free_kernel)
    grid_dependency_wait();  // the free kernel's records
    grid_dependents_go();
    const uint32_t n_units = a.counts[kCntFreeUnits];
    const bool failed = a.counts[kCntError] != 0u;
    const int G = a.G, V = a.V, nblk = a.free_nblk;
    const uint32_t stride = gridDim.x * kTailWarps;
    for (uint32_t w = blockIdx.x * kTailWarps + (threadIdx.x >> 5); w < n_units; w += stride) {
        const uint32_t item = a.free_units[w];
        const int b = (int)(item >> 8), u = (int)(item & 0xFFu);
        const SeqInfo si = a.seq[b];
        const bool pair = u < si.gamma;
        if (failed) {  // a free CTA gave up waiting: no record of this call can be trusted
            if (lane == 0) atomicOr(&a.seq_status[b], SV_ROW_INTERNAL);
            unit_finished_warp(a, b, lane);
            continue;
        }
        const FreeRec* rec = a.free_rec + w;
        // (shared noise without top-p: no statistics pass, so no record was written)
        const uint32_t flags = (a.gumbel && !(si.P < 1.0f)) ? 0u : rec->flags;
        if (flags & kRecFall) continue;  // the cluster kernel finishes this unit
        if (flags & kRecDead) {
            if (lane == 0) atomicOr(&a.seq_status[b], SV_ROW_NONFINITE);
            unit_finished_warp(a, b, lane);
            continue;
        }
        if (a.gumbel) {
            // the target's token: the best of the warps' (score, id) keys
            const float* rrow = a.free_blk + (size_t)w * 2 * nblk;
            const uint32_t hi = lane < a.free_warps ? __float_as_uint(rrow[lane]) : 0u;
            const uint32_t id = lane < a.free_warps ? __float_as_uint(rrow[nblk + lane]) : 0u;
            const bool bad = __any_sync(0xFFFFFFFFu, hi == 0xFFFFFFFFu);
            unsigned long long bk = hi ? (((unsigned long long)hi << 32) | (unsigned long long)(~id)) : 0ull;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const unsigned long long y = __shfl_xor_sync(0xFFFFFFFFu, bk, o);
                bk = y > bk ? y : bk;
            }
            if (bad || bk == 0ull) {  // a NaN or +inf logit, or no finite one
                if (lane == 0) atomicOr(&a.seq_status[b], SV_ROW_NONFINITE);
                unit_finished_warp(a, b, lane);
                continue;
            }
            const int token = score_key_id(bk);
            if (lane == 0) {
                if (pair) {
                    const int acc = a.draft_tokens[(size_t)b * G + u] == token ? 1 : 0;
                    a.unit_acc[(size_t)b * G + u] = acc;
                    if (a.pos_accept) a.pos_accept[(size_t)b * G + u] = acc;
                }
                a.unit_tok[(size_t)b * (G + 1) + u] = token;
                if (a.pos_token) a.pos_token[(size_t)b * (G + 1) + u] = token;
            }
            unit_finished_warp(a, b, lane);
            continue;
        }
        const float Mp = rec->Mp, Mq = rec->Mq, invp2 = rec->invp, invq2 = rec->invq;
        const unsigned long long cutp = rec->cutp, cutq = rec->cutq;
        const float c = 1.4426950408889634f / si.T;  // the free kernel's expressions
        const float nmcp = row_nmc(Mp, c), nmcq = pair ? row_nmc(Mq, c) : 0.0f;
        const TIn* trow = (const TIn*)a.target + ((size_t)b * (G + 1) + u) * (size_t)V;
        const TIn* drow = (const TIn*)a.draft + ((size_t)b * G + u) * (size_t)V;

        // total residual mass; fall back to p when it is zero (p <= q everywhere)
        const float* br = a.free_blk + (size_t)w * 2 * nblk;
        const float* bp = br + nblk;
        CF zr{0.0f, 0.0f}, zp{0.0f, 0.0f};
        for (int j = lane; j < nblk; j += 32) {
            if (pair) zr = cf_add(zr, CF{br[j], 0.0f});
            zp = cf_add(zp, CF{bp[j], 0.0f});
        }
        zr = warp_cf_sum(zr);
        zp = warp_cf_sum(zp);
        const bool use_p = !pair || !(cf_val(zr) > 0.0f);
        const float* bs = use_p ? bp : br;
        const CF zt = use_p ? zp : zr;
        const double v = uniform01(a.seed, (uint32_t)b, (uint32_t)(u + 1), 1u) * ((double)zt.s - (double)zt.c);

        // the block (blocks are in token-id order) whose running sum passes v,
        // else the last block with weight
        int blk = -1, lastb = -1;
        double bef = 0.0, bef_last = 0.0;
        CF carry{0.0f, 0.0f};
        for (int c0 = 0; c0 < nblk; c0 += 32) {
            const int j = c0 + lane;
            const float x = j < nblk ? bs[j] : 0.0f;
            const CF inc = cf_add(carry, warp_cf_scan(CF{x, 0.0f}, lane));
            const double incd = (double)inc.s - (double)inc.c;
            const double excd = incd - (double)x;
            const unsigned hit = __ballot_sync(0xFFFFFFFFu, x > 0.0f && incd > v);
            if (hit) {
                const int l = __ffs(hit) - 1;
                blk = c0 + l;
                bef = __shfl_sync(0xFFFFFFFFu, excd, l);
                break;
            }
            const unsigned pos = __ballot_sync(0xFFFFFFFFu, x > 0.0f);
            if (pos) {
                const int l = 31 - __clz(pos);
                lastb = c0 + l;
                bef_last = __shfl_sync(0xFFFFFFFFu, excd, l);
            }
            carry = CF{__shfl_sync(0xFFFFFFFFu, inc.s, 31), __shfl_sync(0xFFFFFFFFu, inc.c, 31)};
        }
        if (blk < 0) {
            blk = lastb;
            bef = bef_last;
        }

        // the token inside the block: re-read it (each row) and recompute the
        // free kernel's per-element values; the first id whose running sum
        // passes v, else the block's last id with weight
        int token = -1;
        if (blk >= 0) {
            const double vrel = v - bef;
            const int e_start = blk * BS;  // blocks are consecutive in the row whatever the warp count
            const int e_end = min(V, e_start + BS);
            CF run{0.0f, 0.0f};
            int lastel = -1;
            for (int ch = 0; ch < NCH && token < 0; ++ch) {
                const int e0 = e_start + ch * CH + lane * F::VEC;
                float rv[F::VEC];
                float own = 0.0f;
                int mylast = -1;
#pragma unroll
                for (int j = 0; j < F::VEC; ++j) {
                    const int e = e0 + j;
                    rv[j] = 0.0f;
                    if (e < e_end) {
                        const float p = kept_prob<true>(F::load(trow, e), (uint32_t)e, c, nmcp, invp2, cutp);
                        const float q =
                            use_p ? 0.0f : kept_prob<true>(F::load(drow, e), (uint32_t)e, c, nmcq, invq2, cutq);
                        rv[j] = use_p ? p : resid_f(p, q);
                        own += rv[j];
                        if (rv[j] > 0.0f) mylast = e;
                    }
                }
                lastel = max(lastel, __reduce_max_sync(0xFFFFFFFFu, mylast));
                const CF inc = cf_add(run, warp_cf_scan(CF{own, 0.0f}, lane));
                const unsigned hit =
                    __ballot_sync(0xFFFFFFFFu, own > 0.0f && (double)inc.s - (double)inc.c > vrel);
                if (hit) {
                    const int l = __ffs(hit) - 1;
                    int tk = mylast;  // rounding: the lane's last id with weight
                    if (lane == l) {
                        CF cum = cf_add(inc, CF{-own, 0.0f});  // the sum before this lane's ids
#pragma unroll
                        for (int j = 0; j < F::VEC; ++j)
                            if (rv[j] > 0.0f && tk == mylast) {
                                cum = cf_add(cum, CF{rv[j], 0.0f});
                                if ((double)cum.s - (double)cum.c > vrel) tk = e0 + j;
                            }
                    }
                    token = __shfl_sync(0xFFFFFFFFu, tk, l);
                }
                run = CF{__shfl_sync(0xFFFFFFFFu, inc.s, 31), __shfl_sync(0xFFFFFFFFu, inc.c, 31)};
            }
            if (token < 0) token = lastel;
        }

        // alpha and the acceptance test u * q(x) < p(x), from the two logits of x
        int accept = 0;
        float alpha_v = 0.0f;
        if (pair) {
            alpha_v = cf_val(warp_cf_sum(CF{lane < kFreeWarpsWide ? rec->alpha[lane] : 0.0f, 0.0f}));
            if (lane == 0) {
                const int xt = a.draft_tokens[(size_t)b * G + u];
                const float lpx = F::load(trow, xt), lqx = F::load(drow, xt);
                const float clo = (float)(1.4426950408889634 / (double)si.T - (double)c);  // c + clo = log2(e) / T
                const unsigned long long kx =
                    ((unsigned long long)okey32(__float_as_uint(lpx)) << 32) | (unsigned long long)(~(uint32_t)xt);
                const unsigned long long kqx =
                    ((unsigned long long)okey32(__float_as_uint(lqx)) << 32) | (unsigned long long)(~(uint32_t)xt);
                const double px = kx < cutp ? 0.0 : (double)exp2_prod(lpx, Mp, c, clo, nmcp) * (double)invp2;
                const double qx = kqx < cutq ? 0.0 : (double)exp2_prod(lqx, Mq, c, clo, nmcq) * (double)invq2;
                const double ua = uniform01(a.seed, (uint32_t)b, (uint32_t)(u + 1), 0u);
                accept = lenient_accept(ua, si.L, qx, px) ? 1 : 0;
            }
        }
        if (lane == 0) {
            if (pair) {
                a.alpha[(size_t)b * G + u] = alpha_v;
                a.unit_acc[(size_t)b * G + u] = accept;
                if (a.pos_accept) a.pos_accept[(size_t)b * G + u] = accept;
            }
            a.unit_tok[(size_t)b * (G + 1) + u] = token;
            if (a.pos_token) a.pos_token[(size_t)b * (G + 1) + u] = token;
        }
        unit_finished_warp(a, b, lane);
    }
}

template <typename TIn, bool TMA, int W>
cudaError_t launch_free_w(const Args& a0, int sms, cudaStream_t s, void* const ev[2]) {
    auto k = free_kernel<TIn, TMA, W>;
    const int smem = (int)sizeof(FreeSmem<W>);
    static const bool attr_ok = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) ==
                                cudaSuccess;
    if (!attr_ok) return cudaErrorInvalidValue;
    static const int occ = [&] {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, FGeo<W>::kThreads, smem) != cudaSuccess) n = 1;
        return n > 0 ? n : 1;
    }();
    Args a = a0;
    a.free_nblk = free_blocks(a.V, sizeof(TIn) == 2 ? SV_BF16 : SV_F32, W);  // the record stride of this variant
    a.free_warps = W;
    const long long units = (long long)a.B * (a.G + 1);
    long long grid = (long long)occ * sms;
    if (grid > units) grid = units;
    if (grid < 1) grid = 1;
    if (ev && ev[0]) cudaEventRecord((cudaEvent_t)ev[0], s);
    cudaError_t e = launch_pdl(k, dim3((unsigned)grid), dim3(FGeo<W>::kThreads), (size_t)smem, s, a);
    if (e != cudaSuccess) return e;
    if (ev && ev[1]) cudaEventRecord((cudaEvent_t)ev[1], s);
    // the tail: a warp per unit, up to 4 CTAs of 8 warps per SM in flight
    long long tgrid = (units + kTailWarps - 1) / kTailWarps;
    if (tgrid > 4LL * sms) tgrid = 4LL * sms;
    if (tgrid < 1) tgrid = 1;
    return launch_pdl(free_tail_kernel<TIn>, dim3((unsigned)tgrid), dim3(32 * kTailWarps), 0, s, a);
}

// The narrow variant (7 consumer warps, 2 CTAs per SM) unless the batch has
// fewer units than its CTA slots: then each unit gets a whole SM's 15 warps.
template <typename TIn, bool TMA>
cudaError_t launch_free_t(const Args& a, int sms, cudaStream_t s, void* const ev[2]) {
    const long long units = (long long)a.B * (a.G + 1);
    if (units < 2LL * sms) return launch_free_w<TIn, TMA, kFreeWarpsWide>(a, sms, s, ev);
    return launch_free_w<TIn, TMA, kFreeWarpsNarrow>(a, sms, s, ev);
}

}  // namespace

cudaError_t launch_free_kernel(int dtype, bool vector, const Args& a, int sms, cudaStream_t s, void* const ev[2]) {
    if (dtype == SV_BF16)
        return vector ? launch_free_t<__nv_bfloat16, true>(a, sms, s, ev) : launch_free_t<__nv_bfloat16, false>(a, sms, s, ev);
    return vector ? launch_free_t<float, true>(a, sms, s, ev) : launch_free_t<float, false>(a, sms, s, ev);
}

}  // namespace sv
