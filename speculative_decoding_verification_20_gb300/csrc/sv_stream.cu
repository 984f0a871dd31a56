// sv_stream.cu -- streaming top-k path (greedy and 1 <= top_k <= 256 sequences).
//
// Normalisation with top-k ("Fast Inference from Transformers via Speculative
// Decoding" review page, section "Method: Speculative Decoding": top-k and
// argmax are standard sampling from an adjusted distribution) only ever needs
// the k largest logits of a row: the softmax normaliser of the whole
// vocabulary cancels when the kept set is renormalised.  So every logit is
// read from HBM exactly once and no exponential is evaluated on the bulk of
// the vocabulary.
//
// select_kernel (persistent, 2 CTAs per SM, 8 consumer warps + 1 producer warp)
//   producer: pieces of rows are taken from a global counter; each 32 KB tile
//     is brought into a 3-stage shared-memory ring by one cp.async.bulk
//     (TMA) whose completion is counted on the stage's mbarrier.
//   consumers: per 16-byte vector, a packed max tree (NaN-propagating, so it
//     also detects non-finite logits) is compared once with the running
//     threshold theta; only vectors that beat theta build a per-element pass
//     mask and append those (key, token id) candidates to a shared buffer.
//     theta starts at a lower bound of the k-th largest key of the piece's
//     first tile (per-warp ballots over the per-thread maxima); whenever the
//     buffer exceeds 2k entries, a block-wide 4-bit radix select finds the
//     exact k-th key of the buffer, the buffer keeps only keys >= it, and the
//     filter becomes strict (a later tie has a larger id, so it can never
//     enter the top-k).
//   At the end of a piece every candidate >= its exact k-th key (ties
//   included, at most 512) is written to the workspace.
// combine_kernel (one CTA per unit)
//   merges the pieces of the unit's target and draft rows and does, in fp64,
//   softmax over the kept logits, top-p, alpha, the acceptance test and the
//   residual / bonus draw (inverse CDF in ascending token id).
//
// Every mbarrier wait is bounded (2 s on %globaltimer); on timeout the CTA
// records kCntError, stops issuing copies, waits (bounded) for the copies it
// issued and leaves; the combine kernel then marks the affected sequences.
#include "sv_finalize.cuh"

namespace sv {

constexpr int kStages = 3;
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kSelThreads = kConsumers + 32;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;
constexpr int kCombineThreads = 128;

// ---------------------------------------------------------------------------
// PTX helpers: mbarriers, TMA bulk copies, the consumer-only named barrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
// try_wait with a suspend-time hint: the thread sleeps until the phase completes
// (or about 1 ms passes) instead of spinning and taking issue slots
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(1000000u)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// bounded wait for the phase of parity `parity` to complete
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > kWaitLimitNs) return false;
    return true;
}
__device__ __forceinline__ void tma_load_1d(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory"); }
__device__ __forceinline__ int cbar_count(bool p) {
    int r;
    asm volatile("{\n .reg .pred q;\n setp.ne.u32 q, %1, 0;\n bar.red.popc.u32 %0, 1, %2, q;\n}"
                 : "=r"(r)
                 : "r"((uint32_t)p), "n"(kConsumers)
                 : "memory");
    return r;
}

// ---------------------------------------------------------------------------
// keys and composites
// ---------------------------------------------------------------------------
template <typename TIn>
struct Elem;
template <>
struct Elem<__nv_bfloat16> {
    static constexpr int VEC = 8, KB = 16;
    __device__ static uint32_t bits(const uint4& v, int j) {
        const uint32_t w = j < 2 ? v.x : j < 4 ? v.y : j < 6 ? v.z : v.w;
        return (j & 1) ? (w >> 16) : (w & 0xFFFFu);
    }
    __device__ static uint32_t key(uint32_t b) { return okey16(b); }
    __device__ static float value(uint32_t b) { return __uint_as_float(b << 16); }
    __device__ static double key_value(uint32_t k) { return (double)key_value16(k); }
    __device__ static bool bad(uint32_t b) { return bad16(b); }
    static constexpr uint32_t kNegInfBits = 0xFF80u;
};
template <>
struct Elem<float> {
    static constexpr int VEC = 4, KB = 32;
    __device__ static uint32_t bits(const uint4& v, int j) { return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w; }
    __device__ static uint32_t key(uint32_t b) { return okey32(b); }
    __device__ static float value(uint32_t b) { return __uint_as_float(b); }
    __device__ static double key_value(uint32_t k) { return (double)key_value32(k); }
    __device__ static bool bad(uint32_t b) { return bad32(b); }
    static constexpr uint32_t kNegInfBits = 0xFF800000u;
};

// composite sort key: logit key descending, then token id ascending
__device__ __forceinline__ unsigned long long composite(uint32_t key, uint32_t id) {
    return ((unsigned long long)key << 32) | (unsigned long long)(~id);
}
__device__ __forceinline__ uint32_t comp_key(unsigned long long c) { return (uint32_t)(c >> 32); }
__device__ __forceinline__ int comp_id(unsigned long long c) { return (int)(~(uint32_t)c); }

__device__ __forceinline__ int next_pow2(int n) {
    int p = 1;
    while (p < n) p <<= 1;
    return p;
}

// NaN-propagating max of the 16-byte vector (as float), used both as the
// fast-path filter and for non-finite detection
__device__ __forceinline__ float vmax_nan(const uint4& v, __nv_bfloat16*) {
    __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&v.x);
    __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&v.y);
    __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&v.z);
    __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&v.w);
    const __nv_bfloat162 m = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
    return __bfloat162float(__hmax_nan(__low2bfloat16(m), __high2bfloat16(m)));
}
__device__ __forceinline__ float fmax_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float vmax_nan(const uint4& v, float*) {
    return fmax_nan(fmax_nan(__uint_as_float(v.x), __uint_as_float(v.y)),
                    fmax_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
}

// Fast-path test of one full 16-byte vector: updates the running NaN-propagating
// maximum and says whether any element may pass the threshold.
struct RunBf16 {
    __nv_bfloat162 run, th2;
};
__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t w) { return *reinterpret_cast<__nv_bfloat162*>(&w); }
__device__ __forceinline__ bool vec_test(const uint4& v, RunBf16& r, bool strict) {
    const __nv_bfloat162 m = __hmax2_nan(__hmax2_nan(as_bf2(v.x), as_bf2(v.y)), __hmax2_nan(as_bf2(v.z), as_bf2(v.w)));
    r.run = __hmax2_nan(r.run, m);
    return (strict ? __hgt2_mask(m, r.th2) : __hge2_mask(m, r.th2)) != 0u;
}
__device__ __forceinline__ void run_init(RunBf16& r, float thv) {
    r.run = __float2bfloat162_rn(-INFINITY);
    r.th2 = __float2bfloat162_rn(thv);
}
__device__ __forceinline__ float run_value(const RunBf16& r) {
    return __bfloat162float(__hmax_nan(__low2bfloat16(r.run), __high2bfloat16(r.run)));
}
struct RunF32 {
    float run, th;
};
__device__ __forceinline__ bool vec_test(const uint4& v, RunF32& r, bool strict) {
    const float m = fmax_nan(fmax_nan(__uint_as_float(v.x), __uint_as_float(v.y)),
                             fmax_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
    r.run = fmax_nan(r.run, m);
    return strict ? (m > r.th) : (m >= r.th);
}
__device__ __forceinline__ void run_init(RunF32& r, float thv) {
    r.run = -INFINITY;
    r.th = thv;
}
__device__ __forceinline__ float run_value(const RunF32& r) { return r.run; }
template <typename TIn>
struct RunOf {
    using type = RunF32;
};
template <>
struct RunOf<__nv_bfloat16> {
    using type = RunBf16;
};

// ---------------------------------------------------------------------------
// select kernel
// ---------------------------------------------------------------------------
constexpr int kBufCap = 2048;   // candidate buffer
constexpr int kPerThread = kBufCap / kConsumers;
// a piece with at most this many candidates at its end hands them all over unselected
constexpr int kFinalList = 512;
static_assert(kFinalList <= kListCap && kFinalList >= kStreamMaxK, "final list bounds");

struct SelSmem {
    alignas(128) uint8_t buf[kStages][kTileBytes];
    unsigned long long cand[kBufCap];  // (key << 32 | ~id), unsorted
    uint64_t full[kStages];
    uint64_t empty[kStages];
    int4 hdr[kStages];  // piece index (-1: no more work), tile index, elements, first column
    int2 seqk[kStages]; // sequence b and its top-k for the piece
    int red[kConsumerWarps];
    int scan[kConsumerWarps];
    int hist[16];
    unsigned int count;
    uint32_t theta_key;
    int strict;
};

// block sum over the consumers
__device__ __forceinline__ int csum(int v, SelSmem& sm) {
    v = __reduce_add_sync(0xFFFFFFFFu, v);
    if ((threadIdx.x & 31) == 0) sm.red[threadIdx.x >> 5] = v;
    cbar();
    int tot = 0;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) tot += sm.red[w];
    cbar();
    return tot;
}
// exclusive scan over the consumers in thread order
__device__ __forceinline__ int cscan(int v, SelSmem& sm, int* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sm.scan[wid] = x;
    cbar();
    int before = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
        before += (w < wid) ? sm.scan[w] : 0;
        tot += sm.scan[w];
    }
    cbar();
    *total = tot;
    return before + x - v;
}

__device__ __forceinline__ void append(SelSmem& sm, unsigned long long c) {
    const unsigned slot = atomicAdd(&sm.count, 1u);
    if (slot < (unsigned)kBufCap) sm.cand[slot] = c;
}

// Reserve `mine` consecutive buffer slots for this lane with one shared atomic
// per warp (all lanes of the warp call it); returns the lane's first slot.
__device__ __forceinline__ unsigned warp_reserve(SelSmem& sm, unsigned mine) {
    const int lane = threadIdx.x & 31;
    unsigned x = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
    }
    const unsigned total = __shfl_sync(0xFFFFFFFFu, x, 31);
    unsigned base = 0u;
    if (lane == 31 && total) base = atomicAdd(&sm.count, total);
    return __shfl_sync(0xFFFFFFFFu, base, 31) + x - mine;
}

// Exact k-th largest key of the buffer (4-bit radix, shared histogram).
// Every consumer holds up to kPerThread buffer entries in `mine`.  Returns the
// key; *gt receives the number of entries strictly above it.
template <int KB>
__device__ uint32_t buffer_kth_key(SelSmem& sm, const unsigned long long (&mine)[kPerThread], int nmine, int k,
                                   int* gt) {
    uint32_t prefix = 0u;
    int above = 0;
#pragma unroll 1
    for (int sh = KB - 4; sh >= 0; sh -= 4) {
        if (threadIdx.x < 16) sm.hist[threadIdx.x] = 0;
        cbar();
#pragma unroll
        for (int i = 0; i < kPerThread; ++i) {
            if (!__any_sync(0xFFFFFFFFu, i < nmine)) break;
            int digit = -1;
            if (i < nmine) {
                const uint32_t key = comp_key(mine[i]);
                const bool match = (sh + 4 >= KB) || ((key >> (sh + 4)) == (prefix >> (sh + 4)));
                if (match) digit = (int)((key >> sh) & 15u);
            }
            // one shared atomic per distinct digit of the warp
            const unsigned grp = __match_any_sync(0xFFFFFFFFu, digit);
            if (digit >= 0 && (threadIdx.x & 31) == __ffs(grp) - 1) atomicAdd(&sm.hist[digit], __popc(grp));
        }
        cbar();
        int acc = above, dsel = 0;
        for (int d = 15; d >= 0; --d) {
            const int h = sm.hist[d];
            if (acc + h >= k) {
                dsel = d;
                break;
            }
            acc += h;
        }
        above = acc;
        prefix |= (uint32_t)dsel << sh;
        cbar();
    }
    *gt = above;
    return prefix;
}

// Keep the buffer entries with key >= kth (every consumer re-appends its own).
__device__ __forceinline__ void buffer_keep_ge(SelSmem& sm, const unsigned long long (&mine)[kPerThread], int nmine,
                                               uint32_t kth) {
    if (threadIdx.x == 0) sm.count = 0u;
    cbar();
    unsigned keep = 0u;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) keep += (i < nmine && comp_key(mine[i]) >= kth) ? 1u : 0u;
    unsigned slot = warp_reserve(sm, keep);
#pragma unroll
    for (int i = 0; i < kPerThread; ++i)
        if (i < nmine && comp_key(mine[i]) >= kth) sm.cand[slot++] = mine[i];
    cbar();
}

__device__ __forceinline__ int load_mine(SelSmem& sm, unsigned long long (&mine)[kPerThread]) {
    const int cnt = min((int)sm.count, kBufCap);
    int n = 0;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
        const int idx = threadIdx.x + i * kConsumers;
        mine[i] = idx < cnt ? sm.cand[idx] : 0ull;
        n += idx < cnt;
    }
    return n;
}

// per-element pass mask of one 16-byte vector against the threshold value
__device__ __forceinline__ unsigned pass_mask(const uint4& v, float thv, bool strict, __nv_bfloat16*) {
    const __nv_bfloat162 th2 = __float2bfloat162_rn(thv);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    unsigned msk = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
        const unsigned m = strict ? __hgt2_mask(x, th2) : __hge2_mask(x, th2);
        msk |= ((m & 1u) | ((m >> 15) & 2u)) << (2 * i);
    }
    return msk;
}
__device__ __forceinline__ unsigned pass_mask(const uint4& v, float thv, bool strict, float*) {
    const float x[4] = {__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z), __uint_as_float(v.w)};
    unsigned msk = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) msk |= (strict ? (x[i] > thv) : (x[i] >= thv)) ? (1u << i) : 0u;
    return msk;
}

// Exact top-k of one tile appended to the buffer (used when a tile would
// overflow it): k-th largest key by a bitwise search, then the keys above it
// and the lowest-id ties at it.
template <typename TIn>
__device__ void tile_exact_append(SelSmem& sm, const uint4* tile, int nvec, int n, int col0, int k) {
    using E = Elem<TIn>;
    constexpr int Q = kTileBytes / 16 / kConsumers;
    const int t = threadIdx.x;
    uint32_t kth = 0u;
    for (int bit = E::KB - 1; bit >= 0; --bit) {
        const uint32_t c = kth | (1u << bit);
        int mine = 0;
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            const int vi = q * kConsumers + t;
            if (vi < nvec) {
                const uint4 v = tile[vi];
#pragma unroll
                for (int j = 0; j < E::VEC; ++j)
                    mine += (vi * E::VEC + j < n) && !E::bad(E::bits(v, j)) && E::key(E::bits(v, j)) >= c;
            }
        }
        if (csum(mine, sm) >= k) kth = c;
    }
    int gt = 0;
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        const int vi = q * kConsumers + t;
        if (vi < nvec) {
            const uint4 v = tile[vi];
#pragma unroll
            for (int j = 0; j < E::VEC; ++j) {
                const uint32_t b = E::bits(v, j);
                if (vi * E::VEC + j < n && !E::bad(b) && E::key(b) > kth) {
                    append(sm, composite(E::key(b), (uint32_t)(col0 + vi * E::VEC + j)));
                    ++gt;
                }
            }
        }
    }
    const int need = k - csum(gt, sm);
    int base = 0;
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        const int vi = q * kConsumers + t;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        int mine = 0;
        if (vi < nvec) {
            v = tile[vi];
#pragma unroll
            for (int j = 0; j < E::VEC; ++j)
                mine += (vi * E::VEC + j < n) && !E::bad(E::bits(v, j)) && E::key(E::bits(v, j)) == kth;
        }
        int tot;
        int rank = base + cscan(mine, sm, &tot);
        if (mine) {
#pragma unroll
            for (int j = 0; j < E::VEC; ++j) {
                const uint32_t b = E::bits(v, j);
                if (vi * E::VEC + j < n && !E::bad(b) && E::key(b) == kth) {
                    if (rank < need) append(sm, composite(kth, (uint32_t)(col0 + vi * E::VEC + j)));
                    ++rank;
                }
            }
        }
        base += tot;
    }
    cbar();
}

// bitonic sort (descending) of n = 2^m buffer entries by the consumers
__device__ __forceinline__ void csort_desc(unsigned long long* s, int n) {
    for (int k2 = 2; k2 <= n; k2 <<= 1)
        for (int j = k2 >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < n; i += kConsumers) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const unsigned long long x = s[i], y = s[ixj];
                    if (((i & k2) == 0) ? (x < y) : (x > y)) {
                        s[i] = y;
                        s[ixj] = x;
                    }
                }
            }
            cbar();
        }
}

template <typename TIn, bool TMA>
__global__ void __launch_bounds__(kSelThreads, 2) select_kernel(Args a) {
    using E = Elem<TIn>;
    constexpr int TE = kTileBytes / (int)sizeof(TIn);  // elements per tile
    constexpr int Q = kTileBytes / 16 / kConsumers;    // 16-byte vectors per consumer per tile
    extern __shared__ __align__(128) uint8_t smem_raw[];
    SelSmem& sm = *reinterpret_cast<SelSmem*>(smem_raw);
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int V = a.V, G = a.G, ppr = a.ppr;
    const int PE = kTilesPerPiece * TE;

    if (t == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], kConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const uint32_t n_pieces = a.counts[kCntStreamRows] * (uint32_t)ppr;

    if (warp == kConsumerWarps) {
        // ------------------------------ producer ------------------------------
        if (!TMA || lane == 0) {
            int stage = 0;
            uint32_t ph = 1;  // fresh empty barriers count as released
            int issued[kStages];
#pragma unroll
            for (int s = 0; s < kStages; ++s) issued[s] = -1;  // full-barrier parity of the last copy per stage
            bool ok = true;
            // the next piece is claimed (and its row looked up) one piece ahead
            uint32_t w = 0;
            if (lane == 0) w = atomicAdd(&a.counts[kCntPieceNext], 1u);
            if (!TMA) w = __shfl_sync(0xFFFFFFFFu, w, 0);
            int b = 0, r = 0, gamma = 0, k = 1;
            if (w < n_pieces) {
                const uint32_t item = a.stream_rows[w / (uint32_t)ppr];
                b = (int)(item >> 8);
                r = (int)(item & 0xFFu);
                const SeqInfo si = a.seq[b];
                gamma = si.gamma;
                k = si.k;
            }
            while (ok && w < n_pieces) {
                uint32_t w_next = 0;
                if (lane == 0) w_next = atomicAdd(&a.counts[kCntPieceNext], 1u);
                if (!TMA) w_next = __shfl_sync(0xFFFFFFFFu, w_next, 0);
                int b_next = 0, r_next = 0, gamma_next = 0, k_next = 1;
                if (w_next < n_pieces) {
                    const uint32_t item = a.stream_rows[w_next / (uint32_t)ppr];
                    b_next = (int)(item >> 8);
                    r_next = (int)(item & 0xFFu);
                    const SeqInfo si = a.seq[b_next];
                    gamma_next = si.gamma;
                    k_next = si.k;
                }
                const uint32_t row_slot = w / (uint32_t)ppr;
                const int piece = (int)(w - row_slot * (uint32_t)ppr);
                const TIn* row = (r <= gamma) ? (const TIn*)a.target + ((size_t)b * (G + 1) + r) * (size_t)V
                                              : (const TIn*)a.draft + ((size_t)b * G + (r - gamma - 1)) * (size_t)V;
                const int c0 = piece * PE, c1 = min(V, c0 + PE);
                for (int col = c0, tile = 0; col < c1 && ok; col += TE, ++tile) {
                    const int n = min(TE, c1 - col);
                    if (!mbar_wait(&sm.empty[stage], ph)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        sm.hdr[stage] = make_int4((int)w, tile, n, col);
                        sm.seqk[stage] = make_int2(b, k);
                    }
                    if (TMA) {
                        mbar_arrive_expect_tx(&sm.full[stage], (uint32_t)(n * sizeof(TIn)));
                        tma_load_1d(sm.buf[stage], row + col, (uint32_t)(n * sizeof(TIn)), &sm.full[stage]);
                        issued[stage] = (int)(ph ^ 1u);
                    } else {
                        TIn* dst = reinterpret_cast<TIn*>(sm.buf[stage]);
                        for (int i = lane; i < n; i += 32) dst[i] = row[col + i];
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&sm.full[stage]);
                    }
                    if (++stage == kStages) {
                        stage = 0;
                        ph ^= 1u;
                    }
                }
                w = w_next;
                b = b_next;
                r = r_next;
                gamma = gamma_next;
                k = k_next;
            }
            if (ok && mbar_wait(&sm.empty[stage], ph)) {
                if (lane == 0) {
                    sm.hdr[stage] = make_int4(-1, 0, 0, 0);
                    mbar_arrive(&sm.full[stage]);
                }
            } else if (lane == 0) {
                atomicOr(&a.counts[kCntError], 1u);
                // let every copy already issued land before the CTA leaves
                for (int s = 0; s < kStages; ++s)
                    if (issued[s] >= 0) (void)mbar_wait(&sm.full[s], (uint32_t)issued[s]);
            }
        }
        return;
    }

    // ------------------------------ consumers ------------------------------
    int stage = 0;
    uint32_t ph = 0;
    int k = 1, b = 0;
    float run_max = -INFINITY;
    unsigned long long mine[kPerThread];
    while (true) {
        if (!mbar_wait(&sm.full[stage], ph)) {
            if (t == 0) atomicOr(&a.counts[kCntError], 1u);
            break;
        }
        const int4 h = sm.hdr[stage];
        if (h.x < 0) break;
        const int w = h.x, tile_idx = h.y, n = h.z, col0 = h.w;
        const uint32_t row_slot = (uint32_t)w / (uint32_t)ppr;
        const int piece = w - (int)row_slot * ppr;
        const bool first = tile_idx == 0;
        const bool last = col0 + n >= min(V, piece * PE + PE);
        const uint4* tile = reinterpret_cast<const uint4*>(sm.buf[stage]);
        const int nvec = (n + E::VEC - 1) / E::VEC;

        if (first) {
            const int2 bk = sm.seqk[stage];
            b = bk.x;
            k = bk.y;
            run_max = -INFINITY;
            // theta_0: each warp takes the ceil(k/8)-th largest of its lanes' maxima
            // (ballot/popc, no block barrier); the minimum over the 8 warps leaves at
            // least 8 * ceil(k/8) >= k elements of the tile >= theta_0, so every
            // element of the piece's top-k passes the filter
            uint32_t tmax = 0u;
            if (n == TE) {  // full tile: max tree per vector (a NaN/+inf maximum is left out)
#pragma unroll
                for (int q = 0; q < Q; ++q) {
                    typename RunOf<TIn>::type rs;
                    run_init(rs, 0.0f);
                    (void)vec_test(tile[q * kConsumers + t], rs, false);
                    const float mv = run_value(rs);
                    if (!(isnan(mv) || mv == INFINITY)) tmax = max(tmax, okey32(__float_as_uint(mv)) >> (32 - E::KB));
                }
            } else {
#pragma unroll
                for (int q = 0; q < Q; ++q) {
                    const int vi = q * kConsumers + t;
                    if (vi < nvec) {
                        const uint4 v = tile[vi];
#pragma unroll
                        for (int j = 0; j < E::VEC; ++j) {
                            const uint32_t bb = E::bits(v, j);
                            if (vi * E::VEC + j < n && !E::bad(bb)) tmax = max(tmax, E::key(bb));
                        }
                    }
                }
            }
            const int kw = (k + kConsumerWarps - 1) / kConsumerWarps;
            uint32_t thw = 0u;
            for (int bit = E::KB - 1; bit >= 0; --bit) {
                const uint32_t c = thw | (1u << bit);
                if (__popc(__ballot_sync(0xFFFFFFFFu, tmax >= c)) >= kw) thw = c;
            }
            if (lane == 0) sm.red[warp] = (int)thw;
            cbar();
            uint32_t th = 0xFFFFFFFFu;
#pragma unroll
            for (int w2 = 0; w2 < kConsumerWarps; ++w2) th = min(th, (uint32_t)sm.red[w2]);
            if (t == 0) {
                sm.count = 0u;
                sm.theta_key = th;
                sm.strict = 0;
            }
        }
        cbar();
        const unsigned count_before = sm.count;
        const uint32_t th_key = sm.theta_key;
        const bool strict = sm.strict != 0;
        const float thv = th_key == 0u ? -INFINITY : (float)E::key_value(th_key);

        if (n == TE && th_key != 0u) {
            // fast path for a full tile: all loads first, then one max tree and one
            // packed comparison per vector
            uint4 v[Q];
#pragma unroll
            for (int q = 0; q < Q; ++q) v[q] = tile[q * kConsumers + t];
            typename RunOf<TIn>::type rs;
            run_init(rs, thv);
            bool pass[Q];
            bool any = false;
#pragma unroll
            for (int q = 0; q < Q; ++q) {
                pass[q] = vec_test(v[q], rs, strict);
                any |= pass[q];
            }
            run_max = fmax_nan(run_max, run_value(rs));
            if (__any_sync(0xFFFFFFFFu, any)) {
                // per-element masks, then one slot reservation per warp
                unsigned msk[Q];
                unsigned mine = 0u;
#pragma unroll
                for (int q = 0; q < Q; ++q) {
                    msk[q] = pass[q] ? pass_mask(v[q], thv, strict, (TIn*)nullptr) : 0u;
                    mine += __popc(msk[q]);
                }
                unsigned slot = warp_reserve(sm, mine);
#pragma unroll
                for (int q = 0; q < Q; ++q) {
                    const int e0 = (q * kConsumers + t) * E::VEC;
                    unsigned mm = msk[q];
                    while (mm) {
                        const int j = __ffs(mm) - 1;
                        mm &= mm - 1u;
                        // a non-finite logit may be kept here; the piece is flagged by its maximum
                        const uint32_t bb = E::bits(v[q], j);
                        if (slot < (unsigned)kBufCap) sm.cand[slot] = composite(E::key(bb), (uint32_t)(col0 + e0 + j));
                        ++slot;
                    }
                }
            }
        } else {
            // partial tile, or no threshold yet: element by element
#pragma unroll
            for (int q = 0; q < Q; ++q) {
                const int vi = q * kConsumers + t;
                if (vi >= nvec) continue;
                const uint4 v = tile[vi];
                const int e0 = vi * E::VEC;
#pragma unroll
                for (int j = 0; j < E::VEC; ++j) {
                    if (e0 + j >= n) continue;
                    const uint32_t bb = E::bits(v, j);
                    run_max = fmax_nan(run_max, E::value(bb));
                    if (E::bad(bb)) continue;
                    const uint32_t key = E::key(bb);
                    if (strict ? (key > th_key) : (key >= th_key)) append(sm, composite(key, (uint32_t)(col0 + e0 + j)));
                }
            }
        }
        cbar();
        if (sm.count > (unsigned)kBufCap) {  // this tile overflowed the buffer: append its exact top-k instead
            cbar();
            if (t == 0) sm.count = count_before;
            cbar();
            tile_exact_append<TIn>(sm, tile, nvec, n, col0, k);
        }
        // the stage can be refilled
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[stage]);
        if (++stage == kStages) {
            stage = 0;
            ph ^= 1u;
        }

        const int cnt = (int)sm.count;
        if (!last) {
            if (cnt > max(4 * k, 256)) {
                // raise theta to the exact k-th key of the buffer and drop what is below it;
                // from then on the filter is strict: a later tie has a larger id
                const int nmine = load_mine(sm, mine);
                int gt = 0;
                const uint32_t kth = buffer_kth_key<E::KB>(sm, mine, nmine, k, &gt);
                buffer_keep_ge(sm, mine, nmine, kth);
                if (t == 0) {
                    sm.theta_key = kth;
                    sm.strict = 1;
                }
                cbar();
            }
        } else {
            // hand the candidates to the combine kernel: all of them when few (a superset of
            // the piece's top-k, which the combine kernel's exact sort resolves), else every
            // candidate >= the k-th key (ties included)
            int total = cnt;
            if (cnt > kFinalList) {
                const int nmine = load_mine(sm, mine);
                int gt = 0;
                const uint32_t kth = buffer_kth_key<E::KB>(sm, mine, nmine, k, &gt);
                buffer_keep_ge(sm, mine, nmine, kth);
                total = (int)sm.count;
                if (total > kListCap) {  // very many ties: resolve them exactly here
                    const int n2 = next_pow2(total);
                    for (int i = total + t; i < n2; i += kConsumers) sm.cand[i] = 0ull;
                    cbar();
                    csort_desc(sm.cand, n2);
                    total = k;
                }
            }
            unsigned long long* out = a.cand + (size_t)w * kListCap;
            for (int i = t; i < total; i += kConsumers) out[i] = sm.cand[i];
            // non-finite logits in this piece (NaN or +inf dominate the NaN-propagating max)
            const bool nf = isnan(run_max) || run_max == INFINITY;
            const int any_nf = cbar_count(nf);
            if (t == 0) {
                a.cand_cnt[w] = (uint32_t)total;
                if (any_nf) atomicOr(&a.seq_status[b], SV_ROW_NONFINITE);
            }
            cbar();
        }
    }
}

// ---------------------------------------------------------------------------
// combine kernel
// ---------------------------------------------------------------------------
struct CombSmem {
    unsigned long long sort[kSortCap];
    unsigned long long top[2][kStreamMaxK];
    double prob[2][kStreamMaxK];
    double resid[kStreamMaxK];
    int rid[kStreamMaxK];
    int kept[2];
};

// Exact top-k of a row, sorted by (logit desc, id asc), from its pieces' candidate
// lists (each a superset of that piece's top-k); returns how many were found (k normally).
__device__ int merge_row(const Args& a, uint32_t row_slot, int k, unsigned long long* out, CombSmem& sm) {
    const int ppr = a.ppr;
    int total = 0;
    for (int j = 0; j < ppr; ++j) total += (int)__ldcg(&a.cand_cnt[(size_t)row_slot * ppr + j]);
    const int n2 = next_pow2(total < 2 ? 2 : total);
    int off = 0;
    for (int j = 0; j < ppr; ++j) {
        const size_t piece = (size_t)row_slot * ppr + j;
        const int c = (int)__ldcg(&a.cand_cnt[piece]);
        for (int i = threadIdx.x; i < c; i += blockDim.x) sm.sort[off + i] = __ldcg(&a.cand[piece * kListCap + i]);
        off += c;
    }
    for (int i = total + threadIdx.x; i < n2; i += blockDim.x) sm.sort[i] = 0ull;
    __syncthreads();
    for (int k2 = 2; k2 <= n2; k2 <<= 1)
        for (int j = k2 >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < n2; i += blockDim.x) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const unsigned long long x = sm.sort[i], y = sm.sort[ixj];
                    if (((i & k2) == 0) ? (x < y) : (x > y)) {
                        sm.sort[i] = y;
                        sm.sort[ixj] = x;
                    }
                }
            }
            __syncthreads();
        }
    const int kk = total < k ? total : k;
    for (int i = threadIdx.x; i < kk; i += blockDim.x) out[i] = sm.sort[i];
    __syncthreads();
    return kk;
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
    const double vmax = Elem<TIn>::key_value(comp_key(top[0]));
    double s = 0.0;
    for (int j = lane; j < k; j += 32) {
        const double v = Elem<TIn>::key_value(comp_key(top[j]));
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
            const unsigned hit = __ballot_sync(0xFFFFFFFFu, j < k && carry + x >= P);
            if (hit) {
                keep = c0 + __ffs(hit);
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
__device__ void combine_unit(const Args& a, int b, int unit, const SeqInfo& si, CombSmem& sm) {
    const int G = a.G;
    const bool pair = unit < si.gamma;
    const uint32_t slot_t = si.row_off + (uint32_t)unit;
    const uint32_t slot_d = si.row_off + (uint32_t)si.gamma + 1u + (uint32_t)unit;
    const int kt = merge_row(a, slot_t, si.k, sm.top[0], sm);  // exact top-k, ties to the lower id
    const int kd = pair ? merge_row(a, slot_d, si.k, sm.top[1], sm) : 0;

    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        // a row without a finite logit (or with non-finite ones, already flagged)
        const uint32_t ninf_key = Elem<TIn>::key(Elem<TIn>::kNegInfBits);
        const bool dead = kt < 1 || comp_key(sm.top[0][0]) <= ninf_key ||
                          (pair && (kd < 1 || comp_key(sm.top[1][0]) <= ninf_key));
        if (dead) {
            if (lane == 0) atomicOr(&a.seq_status[b], SV_ROW_NONFINITE);
        } else {
            normalise_kept<TIn>(sm.top[0], kt, si.T, si.P, sm.prob[0]);
            if (pair) normalise_kept<TIn>(sm.top[1], kd, si.T, si.P, sm.prob[1]);

            // alpha_i = sum_x min(p, q) over the ids kept in both rows; residual weights
            double alpha = 0.0;
            for (int j = lane; j < kt; j += 32) {
                const int id = comp_id(sm.top[0][j]);
                double q = 0.0;
                if (pair)
                    for (int e = 0; e < kd; ++e)
                        if (comp_id(sm.top[1][e]) == id) q = sm.prob[1][e];
                const double p = sm.prob[0][j];
                alpha += fmin(p, q);
                sm.resid[j] = pair ? fmax(p - q, 0.0) : p;  // bonus: q_{gamma+1} := 0
            }
            alpha = warp_sum(alpha);
            __syncwarp();

            // acceptance test u * q(x) < p(x)
            int accept = 0;
            if (pair) {
                const int x = a.draft_tokens[(size_t)b * G + unit];
                double px = 0.0, qx = 0.0;
                for (int j = lane; j < kt; j += 32)
                    if (comp_id(sm.top[0][j]) == x) px = sm.prob[0][j];
                for (int j = lane; j < kd; j += 32)
                    if (comp_id(sm.top[1][j]) == x) qx = sm.prob[1][j];
                px = warp_sum(px);
                qx = warp_sum(qx);
                const double u = uniform01(a.seed, (uint32_t)b, (uint32_t)(unit + 1), 0u);
                accept = (u * qx < px) ? 1 : 0;
            }

            // residual (or bonus) draw: inverse CDF in ascending token id
            double Z = 0.0;
            for (int j = lane; j < kt; j += 32) Z += sm.resid[j];
            Z = warp_sum(Z);
            if (!(Z > 0.0)) {  // p <= q everywhere: fall back to p
                Z = 0.0;
                for (int j = lane; j < kt; j += 32) {
                    sm.resid[j] = sm.prob[0][j];
                    Z += sm.resid[j];
                }
                Z = warp_sum(Z);
            }
            __syncwarp();
            double rr[kStreamMaxK / 32];
            int rank[kStreamMaxK / 32];
#pragma unroll
            for (int m = 0; m < kStreamMaxK / 32; ++m) {
                const int j = lane + 32 * m;
                rank[m] = -1;
                rr[m] = 0.0;
                if (j < kt) {
                    const int id = comp_id(sm.top[0][j]);
                    int r = 0;
                    for (int e = 0; e < kt; ++e) r += comp_id(sm.top[0][e]) < id;
                    rank[m] = r;
                    rr[m] = sm.resid[j];
                }
            }
            __syncwarp();
#pragma unroll
            for (int m = 0; m < kStreamMaxK / 32; ++m) {
                const int j = lane + 32 * m;
                if (j < kt) {
                    sm.resid[rank[m]] = rr[m];
                    sm.rid[rank[m]] = comp_id(sm.top[0][j]);
                }
            }
            __syncwarp();
            const double v = uniform01(a.seed, (uint32_t)b, (uint32_t)(unit + 1), 1u) * Z;
            int token = -1, last_pos = -1;
            double carry = 0.0;
            for (int c0 = 0; c0 < kt && token < 0; c0 += 32) {
                const int j = c0 + lane;
                const double r = (j < kt) ? sm.resid[j] : 0.0;
                double x = r;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const double y = __shfl_up_sync(0xFFFFFFFFu, x, o);
                    if (lane >= o) x += y;
                }
                const unsigned pos = __ballot_sync(0xFFFFFFFFu, j < kt && r > 0.0);
                if (pos) last_pos = c0 + 31 - __clz(pos);
                const unsigned hit = __ballot_sync(0xFFFFFFFFu, j < kt && r > 0.0 && carry + x > v);
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
                for (int j = lane; j < kt; j += 32)
                    a.p_out[((size_t)b * (G + 1) + unit) * a.V + comp_id(sm.top[0][j])] = (float)sm.prob[0][j];
            if (a.q_out && pair)
                for (int j = lane; j < kd; j += 32)
                    a.q_out[((size_t)b * G + unit) * a.V + comp_id(sm.top[1][j])] = (float)sm.prob[1][j];
        }
    }
    unit_finished(a, b);
}

template <typename TIn>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(Args a) {
    __shared__ CombSmem sm;
    const uint32_t n_units = a.counts[kCntStreamUnits];
    const bool failed = a.counts[kCntError] != 0u;
    for (uint32_t w = blockIdx.x; w < n_units; w += gridDim.x) {
        const uint32_t item = a.stream_units[w];
        const int b = (int)(item >> 8), unit = (int)(item & 0xFFu);
        const SeqInfo si = a.seq[b];
        if (failed) {  // a select CTA gave up waiting: no result of this call can be trusted
            if (threadIdx.x == 0) atomicOr(&a.seq_status[b], SV_ROW_INTERNAL);
            unit_finished(a, b);
            continue;
        }
        combine_unit<TIn>(a, b, unit, si, sm);
    }
}

// ---------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------
namespace {
template <typename TIn, bool TMA>
cudaError_t launch_t(const Args& a, int sms, cudaStream_t s, void* const ev[2]) {
    auto sel = select_kernel<TIn, TMA>;
    auto comb = combine_kernel<TIn>;
    const int smem = (int)sizeof(SelSmem);
    static const bool attr_ok = cudaFuncSetAttribute(sel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) ==
                                cudaSuccess;
    if (!attr_ok) return cudaErrorInvalidValue;
    static const int occ = [&] {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, sel, kSelThreads, smem) != cudaSuccess) n = 1;
        return n > 0 ? n : 1;
    }();
    const long long pieces = (long long)a.B * (2 * a.G + 1) * a.ppr;
    long long grid = (long long)occ * sms;
    if (grid > pieces) grid = pieces;
    if (grid < 1) grid = 1;
    if (ev && ev[0]) cudaEventRecord((cudaEvent_t)ev[0], s);
    sel<<<(unsigned)grid, kSelThreads, smem, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (ev && ev[1]) cudaEventRecord((cudaEvent_t)ev[1], s);
    long long cgrid = (long long)a.B * (a.G + 1);
    if (cgrid > (long long)sms * 16) cgrid = (long long)sms * 16;
    if (cgrid < 1) cgrid = 1;
    comb<<<(unsigned)cgrid, kCombineThreads, 0, s>>>(a);
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_stream_kernel(int dtype, bool vector, const Args& a, int sms, cudaStream_t s, void* const ev[2]) {
    if (dtype == SV_BF16)
        return vector ? launch_t<__nv_bfloat16, true>(a, sms, s, ev) : launch_t<__nv_bfloat16, false>(a, sms, s, ev);
    return vector ? launch_t<float, true>(a, sms, s, ev) : launch_t<float, false>(a, sms, s, ev);
}

}  // namespace sv
