// sv_stream.cu -- select kernel of the streaming top-k path (greedy and 1 <= top_k <= 256 sequences).
//
// Normalisation with top-k ("Fast Inference from Transformers via Speculative
// Decoding" review page, section "Method: Speculative Decoding": top-k and
// argmax are standard sampling from an adjusted distribution) only ever needs
// the k largest logits of a row: the softmax normaliser of the whole
// vocabulary cancels when the kept set is renormalised.  So every logit is
// read from HBM exactly once and no exponential is evaluated on the bulk of
// the vocabulary.
//
// select_kernel (persistent, 2 CTAs per SM, 7 consumer warps + 1 producer warp)
//   producer: pieces of rows are taken from a global counter (one piece ahead);
//     each 28 KB tile is brought into a 3-stage shared-memory ring by one
//     cp.async.bulk (TMA) whose completion is counted on the stage's mbarrier.
//   consumers: every warp takes its own 16-byte vectors of each tile into
//     registers.  A packed max tree per vector (NaN-propagating, so it also
//     detects non-finite logits) is compared with the threshold; the thread's
//     passing elements make one 64-bit mask, and only those few are read back
//     from the tile and appended, as (key, token id), to the warp's own list in
//     shared memory (then the stage goes back to the producer).
//   threshold, speculative: a piece spanning several tiles starts from the
//     (3k / tiles)-th largest of the warps' top lane maxima in its first tile,
//     which aims at about the piece's 3k-th largest logit.  At the end of the
//     piece it is checked: at least k logits reached it, so the piece's k-th
//     largest logit is at or above it and the whole top-k was appended.  If
//     not, the consumers redo the piece conservatively from global memory.
//   threshold, conservative (single-tile pieces, large k, redo): the larger of
//     the warp's own k-th largest key so far and the block floor min_w pub[w],
//     where warp w publishes its ceil(k/W)-th largest key; the W warps then
//     hold at least k keys >= the floor, so it never exceeds the piece's k-th
//     largest key.  The list is re-selected after every tile it grew in.
//   A list about to overflow is cut to its exact top-k (ties to the lower id).
//   Warps meet only on a piece's first tile and at its end, on a bounded
//   mbarrier.  At the end of a piece the warps' lists (a superset of the
//   piece's top-k, at most 512 entries; else cut to exactly k) are written to
//   the workspace.
// The candidate lists go to the combine kernel (sv_combine.cu), which keeps
// the exact top-k of each row and finishes the unit.
//
// Every mbarrier wait is bounded (2 s on %globaltimer); on timeout the CTA
// records kCntError, stops issuing copies, waits (bounded) for the copies it
// issued and leaves; the combine kernel then marks the affected sequences.
#include "sv_keys.cuh"

namespace sv {

constexpr int kStages = 3;
constexpr int kConsumerWarps = 7;  // with the producer, 8 warps: 2 CTAs per SM at up to 128 registers
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kSelThreads = kConsumers + 32;

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
// (or about hint_ns passes) instead of spinning and taking issue slots
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// bounded wait for the phase of parity `parity` to complete: false after
// about limit_ns (each try sleeps at most min(limit_ns, 1 ms))
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned long long limit_ns) {
    const uint32_t hint = limit_ns < 1000000ull ? (uint32_t)limit_ns : 1000000u;
    if (mbar_try_wait(bar, parity, hint)) return true;
    if (limit_ns < 1000ull) return false;  // below the timer's ~1 us resolution: one try only
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity, hint))
        if (global_ns() - t0 > limit_ns) return false;
    return true;
}
__device__ __forceinline__ void tma_load_1d(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// ---------------------------------------------------------------------------
// select kernel
// ---------------------------------------------------------------------------
constexpr int kWarpCap = kStreamMaxK + 32;          // a warp's list: its exact top-k plus one step of appends
constexpr int kWarpSlots = kWarpCap / 32;           // list entries per lane
constexpr int kBufCap = kConsumerWarps * kWarpCap;  // the warps' lists side by side
constexpr int kPerThread = kBufCap / kConsumers;
static_assert(kWarpCap % 32 == 0 && kBufCap % kConsumers == 0, "list geometry");
static_assert(kListCap <= kBufCap, "a piece's list fits the buffer");


struct SelSmem {
    alignas(128) uint8_t buf[kStages][kTileBytes];
    unsigned long long cand[kBufCap];  // warp w's list at [w * kWarpCap, ...): (key << 32 | ~id), unsorted
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t gsync;                    // consumer-warp barrier (one arrival per warp, bounded waits)
    int4 hdr[kStages];                 // piece index (-1: no more work), tile index, elements, first column
    int2 seqk[kStages];                // sequence b and its top-k for the piece
    int2 pce[kStages];                 // the piece's end column and its number of tiles
    uint32_t pub[kConsumerWarps];      // per warp: its ceil(k/W)-th largest key of the piece so far (0: none)
    uint32_t spec[32];                 // warp w's largest lane maxima of a piece's first tile at [4w, 4w + 4)
    int red[kConsumerWarps];
    int scan[kConsumerWarps];
    int hist[16];
    unsigned long long wait_ns;        // limit of every wait on another warp or a copy (Args::wait_ns)
};


// Barrier of the consumer warps on an mbarrier (8 arrivals per phase): bounded
// like every other wait, so a lost copy cannot leave warps parked for good.
// Once a wait has failed the warp stops taking part and reports false.
struct GSync {
    uint32_t ph;
    bool ok;
};
__device__ __forceinline__ bool gbar(SelSmem& sm, GSync& g) {
    __syncwarp();
    if (!g.ok) return false;
    if ((threadIdx.x & 31) == 0) mbar_arrive(&sm.gsync);
    g.ok = __all_sync(0xFFFFFFFFu, mbar_wait(&sm.gsync, g.ph, sm.wait_ns));
    g.ph ^= 1u;
    return g.ok;
}

// block sum over the consumers
__device__ __forceinline__ int gsum(int v, SelSmem& sm, GSync& g) {
    v = __reduce_add_sync(0xFFFFFFFFu, v);
    if ((threadIdx.x & 31) == 0) sm.red[threadIdx.x >> 5] = v;
    gbar(sm, g);
    int tot = 0;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) tot += sm.red[w];
    gbar(sm, g);
    return tot;
}
// exclusive scan over the consumers in thread order
__device__ __forceinline__ int gscan(int v, SelSmem& sm, GSync& g, int* total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sm.scan[wid] = x;
    gbar(sm, g);
    int before = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
        before += (w < wid) ? sm.scan[w] : 0;
        tot += sm.scan[w];
    }
    gbar(sm, g);
    *total = tot;
    return before + x - v;
}

// Exclusive prefix over the warp of a per-lane count c < 2^NB, and the warp total.
template <int NB>
__device__ __forceinline__ int warp_prefix(unsigned c, int* total) {
    const unsigned lt = lanemask_lt();
    int pre = 0, tot = 0;
#pragma unroll
    for (int bit = 0; bit < NB; ++bit) {
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, (c >> bit) & 1u);
        pre += __popc(bal & lt) << bit;
        tot += __popc(bal) << bit;
    }
    *total = tot;
    return pre;
}

// The ka-th and kb-th largest of the warp's keys (N per lane, the first `used`
// slots in use, 0 = no entry): the largest c with at least ka (kb) keys >= c,
// found bit by bit below the common prefix of the smallest and largest key;
// 0 when the warp holds fewer keys.
template <int KB, int N>
__device__ __forceinline__ void warp_two_kth(const uint32_t (&key)[N], int used, int ka, int kb, uint32_t* xa,
                                             uint32_t* xb) {
    uint32_t lo = 0xFFFFFFFFu, hi = 0u;
    unsigned cnt = 0u;
#pragma unroll
    for (int m = 0; m < N; ++m)
        if (m < used && key[m] != 0u) {
            lo = min(lo, key[m]);
            hi = max(hi, key[m]);
            ++cnt;
        }
    lo = __reduce_min_sync(0xFFFFFFFFu, lo);
    hi = __reduce_max_sync(0xFFFFFFFFu, hi);
    cnt = __reduce_add_sync(0xFFFFFFFFu, cnt);
    if (cnt < (unsigned)ka && cnt < (unsigned)kb) {
        *xa = *xb = 0u;
        return;
    }
    const uint32_t diff = lo ^ hi;
    const int nb = diff ? 32 - __clz(diff) : 0;  // bits below the common prefix
    const uint32_t base = nb >= 32 ? 0u : (lo & ~((1u << nb) - 1u));
    uint32_t pa = base, pb = base;
#pragma unroll 1
    for (int bit = nb - 1; bit >= 0; --bit) {
        const uint32_t ca = pa | (1u << bit), cb = pb | (1u << bit);
        unsigned na = 0u, nbb = 0u;
#pragma unroll
        for (int m = 0; m < N; ++m)
            if (m < used) {
                na += key[m] >= ca;
                nbb += key[m] >= cb;
            }
        na = __reduce_add_sync(0xFFFFFFFFu, na);
        nbb = __reduce_add_sync(0xFFFFFFFFu, nbb);
        if (na >= (unsigned)ka) pa = ca;
        if (nbb >= (unsigned)kb) pb = cb;
    }
    *xa = cnt >= (unsigned)ka ? pa : 0u;
    *xb = cnt >= (unsigned)kb ? pb : 0u;
    (void)KB;
}

// lower bound of the piece's k-th key from every warp's published estimate (a
// stale value is lower, so still a lower bound)
__device__ __forceinline__ uint32_t block_floor(const SelSmem& sm, int lane) {
    const uint32_t pv = lane < kConsumerWarps ? ((const volatile uint32_t*)sm.pub)[lane] : 0xFFFFFFFFu;
    return __reduce_min_sync(0xFFFFFFFFu, pv);
}

struct WarpList {
    int cnt;          // entries in the warp's list
    uint32_t th_own;  // the warp's own threshold key (its k-th largest so far; 0: none)
};

// Refresh a warp's list (N slots per lane cover it): publish its ceil(k/8)-th
// largest key, raise its own threshold to its k-th largest key and keep only
// the keys >= max(that, the block floor).  With `exact`, ties at the k-th key
// beyond k entries are cut too (lowest ids kept), so at most k entries remain.
template <int KB, int N>
__device__ __forceinline__ WarpList warp_refresh_n(SelSmem& sm, int warp, int lane, WarpList st, int k, int kw,
                                                   bool exact) {
    unsigned long long* L = sm.cand + warp * kWarpCap;
    const int used = (st.cnt + 31) >> 5;
    unsigned long long e[N];
    uint32_t key[N];
#pragma unroll
    for (int m = 0; m < N; ++m) {
        const int i = lane + 32 * m;
        e[m] = (m < used && i < st.cnt) ? L[i] : 0ull;
        key[m] = comp_key(e[m]);
    }
    uint32_t xw, xk;
    warp_two_kth<KB, N>(key, used, kw, k, &xw, &xk);
    if (lane == 0 && xw > ((volatile uint32_t*)sm.pub)[warp]) ((volatile uint32_t*)sm.pub)[warp] = xw;
    if (xk > st.th_own) st.th_own = xk;
    const uint32_t floor = block_floor(sm, lane);
    const uint32_t cut = max(st.th_own, floor);
    uint32_t id_cut = 0xFFFFFFFFu;
    if (exact && xk > 0u && xk >= floor) {  // ties at the k-th key beyond k entries: lowest ids (< 2^18)
        unsigned gt = 0u, eq = 0u;
#pragma unroll
        for (int m = 0; m < N; ++m) {
            gt += key[m] > xk;
            eq += key[m] == xk;
        }
        gt = __reduce_add_sync(0xFFFFFFFFu, gt);
        eq = __reduce_add_sync(0xFFFFFFFFu, eq);
        const unsigned need = (unsigned)k - gt;
        if (eq > need) {
            uint32_t lo = 0u;
#pragma unroll 1
            for (int bit = 17; bit >= 0; --bit) {
                const uint32_t c = lo | (1u << bit);
                unsigned nlt = 0u;
#pragma unroll
                for (int m = 0; m < N; ++m) nlt += key[m] == xk && (uint32_t)comp_id(e[m]) < c;
                nlt = __reduce_add_sync(0xFFFFFFFFu, nlt);
                if (nlt < need) lo = c;
            }
            id_cut = lo;
        }
    }
    // compact in place: every entry is already in registers
    __syncwarp();
    const unsigned lt = lanemask_lt();
    int base = 0;
#pragma unroll
    for (int m = 0; m < N; ++m) {
        if (m < used) {
            const bool keep = key[m] != 0u && key[m] >= cut && !(key[m] == xk && (uint32_t)comp_id(e[m]) > id_cut);
            const unsigned bal = __ballot_sync(0xFFFFFFFFu, keep);
            if (keep) L[base + __popc(bal & lt)] = e[m];
            base += __popc(bal);
        }
    }
    __syncwarp();
    st.cnt = base;
    return st;
}
template <int KB>
__device__ __noinline__ WarpList warp_refresh(SelSmem& sm, int warp, int lane, WarpList st, int k, int kw,
                                              bool exact) {
    if (st.cnt <= 64) return warp_refresh_n<KB, 2>(sm, warp, lane, st, k, kw, exact);
    if (st.cnt <= 128) return warp_refresh_n<KB, 4>(sm, warp, lane, st, k, kw, exact);
    return warp_refresh_n<KB, kWarpSlots>(sm, warp, lane, st, k, kw, exact);
}
// out-of-line exact refresh for the rare overflow path inside the tile loop
template <int KB>
__device__ __noinline__ WarpList warp_refresh_out(SelSmem& sm, int warp, int lane, WarpList st, int k, int kw) {
    return warp_refresh_n<KB, kWarpSlots>(sm, warp, lane, st, k, kw, true);
}

// per-element pass mask of one 16-byte vector: value >= the threshold value
__device__ __forceinline__ unsigned pass_mask(const uint4& v, float thv, __nv_bfloat16*) {
    const __nv_bfloat162 th2 = __float2bfloat162_rn(thv);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    unsigned msk = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
        const unsigned m = __hge2_mask(x, th2);
        msk |= ((m & 1u) | ((m >> 15) & 2u)) << (2 * i);
    }
    return msk;
}
__device__ __forceinline__ unsigned pass_mask(const uint4& v, float thv, float*) {
    const float x[4] = {__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z), __uint_as_float(v.w)};
    unsigned msk = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) msk |= (x[i] >= thv) ? (1u << i) : 0u;
    return msk;
}

// Rare fallback at the end of a piece whose warps' lists together exceed
// kListCap: gather them, find the exact k-th key of the union (4-bit radix),
// resolve ties at it by id, and write exactly k entries.  Returns the count.
template <int KB>
__device__ __noinline__ int piece_cut(SelSmem& sm, GSync& g, int warp, int lane, int cnt, int off, int total, int k,
                         unsigned long long* out) {
    const int t = threadIdx.x;
    // gather into one contiguous array (through registers: the lists overlap it)
    unsigned long long e[kWarpSlots];
    const unsigned long long* L = sm.cand + warp * kWarpCap;
#pragma unroll
    for (int m = 0; m < kWarpSlots; ++m) {
        const int i = lane + 32 * m;
        e[m] = i < cnt ? L[i] : 0ull;
    }
    gbar(sm, g);
#pragma unroll
    for (int m = 0; m < kWarpSlots; ++m) {
        const int i = lane + 32 * m;
        if (i < cnt) sm.cand[off + i] = e[m];
    }
    gbar(sm, g);
    total = min(total, kBufCap);
    unsigned long long mine[kPerThread];
    int nmine = 0;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
        const int idx = t + i * kConsumers;
        mine[i] = idx < total ? sm.cand[idx] : 0ull;
        nmine += idx < total;
    }
    // k-th largest key of the union: 4-bit digits from the top, shared histogram
    uint32_t prefix = 0u;
    int above = 0;
#pragma unroll 1
    for (int sh = KB - 4; sh >= 0; sh -= 4) {
        if (t < 16) sm.hist[t] = 0;
        gbar(sm, g);
#pragma unroll
        for (int i = 0; i < kPerThread; ++i) {
            if (i < nmine) {
                const uint32_t key = comp_key(mine[i]);
                const bool match = (sh + 4 >= KB) || ((key >> (sh + 4)) == (prefix >> (sh + 4)));
                if (match) atomicAdd(&sm.hist[(key >> sh) & 15u], 1);
            }
        }
        gbar(sm, g);
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
        gbar(sm, g);
    }
    const uint32_t kth = prefix;
    const int need = k - above;  // ties at kth to keep, lowest ids first
    int eq = 0;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) eq += i < nmine && comp_key(mine[i]) == kth;
    uint32_t id_cut = 0xFFFFFFFFu;
    if (gsum(eq, sm, g) > need) {
        uint32_t lo = 0u;
#pragma unroll 1
        for (int bit = 17; bit >= 0; --bit) {
            const uint32_t c = lo | (1u << bit);
            int nlt = 0;
#pragma unroll
            for (int i = 0; i < kPerThread; ++i)
                nlt += i < nmine && comp_key(mine[i]) == kth && (uint32_t)comp_id(mine[i]) < c;
            if (gsum(nlt, sm, g) < need) lo = c;
        }
        id_cut = lo;
    }
    int keep = 0;
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
        const uint32_t key = comp_key(mine[i]);
        keep += i < nmine && (key > kth || (key == kth && (uint32_t)comp_id(mine[i]) <= id_cut));
    }
    int written;
    int slot = gscan(keep, sm, g, &written);
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
        const uint32_t key = comp_key(mine[i]);
        if (i < nmine && (key > kth || (key == kth && (uint32_t)comp_id(mine[i]) <= id_cut)) && slot < kListCap)
            out[slot++] = mine[i];
    }
    return min(written, kListCap);
}

// ---------------------------------------------------------------------------
// consumer steps
// ---------------------------------------------------------------------------
constexpr int kSpecFactor = 3;  // the speculative threshold aims at the piece's (3k)-th largest logit
constexpr int kSpecPub = 4;     // lane maxima each warp publishes for it
constexpr int kSpecMaxRank = kSpecPub * kConsumerWarps;
static_assert(kSpecMaxRank <= 32, "the published maxima fit one per lane");

// Bitonic sort of one value per lane across the warp, descending: lane i ends
// with the i-th largest.
__device__ __forceinline__ uint32_t warp_sort_desc(uint32_t x, int lane) {
#pragma unroll
    for (int k2 = 2; k2 <= 32; k2 <<= 1)
#pragma unroll
        for (int j = k2 >> 1; j > 0; j >>= 1) {
            const uint32_t y = __shfl_xor_sync(0xFFFFFFFFu, x, j);
            const bool lower = (lane & j) == 0;
            const bool desc = (lane & k2) == 0;  // this block's direction (all descending at the end)
            x = (lower == desc) ? max(x, y) : min(x, y);
        }
    return x;
}

// Rank (in the piece's first tile) whose value is the speculative threshold of
// a piece of `tiles` tiles, or 0 when the piece is handled conservatively from
// the start (a single tile, where it would gain nothing, or a large k).
__device__ __forceinline__ int spec_rank(int k, int tiles) {
    if (tiles < 2) return 0;
    const int j = min(k, max(1, (kSpecFactor * k + tiles - 1) / tiles));
    return j <= kSpecMaxRank ? j : 0;
}

struct CState {
    WarpList st;
    int since;        // appends since the last refresh
    int appended;     // appends in this piece
    bool overflow;    // the list had to be cut inside the piece
    bool spec;        // the piece runs on a speculative threshold
    float run_max;    // NaN-propagating maximum of the piece's logits seen by this warp
    uint32_t th_spec; // speculative threshold key
};

// The vectors of one tile held by a warp (v; the tile's elements at elem, n of
// them from column col0): filter against the warp's threshold, append what
// passes to its list.
//   first tile of a piece: reset, then the starting thresholds from the
//     per-vector maxima (one barrier): speculative -- the spec_rank-th largest
//     of the warps' top maxima together; conservative -- every warp publishes
//     its ceil(k/8)-th largest maximum and starts at its own k-th.
//   conservative pieces refresh the list after every tile that appended.
// Returns false if a barrier wait gave up.
template <typename TIn>
__device__ __forceinline__ bool consume_tile(SelSmem& sm, GSync& g, const uint4 (&v)[kTileBytes / 16 / kConsumers],
                                             const TIn* elem, int n, int col0, bool first, bool last, int tiles,
                                             int k, CState& cs, int warp, int lane) {
    using E = Elem<TIn>;
    constexpr int Q = kTileBytes / 16 / kConsumers;
    const int t = threadIdx.x;
    const int kw = (k + kConsumerWarps - 1) / kConsumerWarps;
    unsigned long long* L = sm.cand + warp * kWarpCap;
    if (first) {
        cs.st = WarpList{0, 0u};
        cs.since = cs.appended = 0;
        cs.overflow = false;
        cs.run_max = -INFINITY;
        cs.th_spec = 0u;
        // per-vector maxima (a NaN or +inf maximum is left out)
        uint32_t vk[Q];
#pragma unroll
        for (int q = 0; q < Q; ++q) {
            const int e0 = (q * kConsumers + t) * E::VEC;
            float mv = -INFINITY;
            if (e0 + E::VEC <= n) {
                mv = vmax_nan(v[q], (TIn*)nullptr);
            } else {
#pragma unroll
                for (int j = 0; j < E::VEC; ++j)
                    if (e0 + j < n) mv = fmax_nan(mv, E::value(E::bits(v[q], j)));
            }
            vk[q] = (isnan(mv) || mv == INFINITY || e0 >= n) ? 0u : E::key(E::bits_of(mv));
        }
        if (cs.spec) {
            // every warp publishes its kSpecPub largest lane maxima; the threshold is
            // the j-th largest of them all
            const int j = spec_rank(k, tiles);
            uint32_t lm = 0u;
#pragma unroll
            for (int q = 0; q < Q; ++q) lm = max(lm, vk[q]);
            lm = warp_sort_desc(lm, lane);
            if (lane < kSpecPub) sm.spec[warp * kSpecPub + lane] = lm;
            if (!gbar(sm, g)) return false;
            uint32_t u = lane < kSpecMaxRank ? sm.spec[lane] : 0u;
            u = warp_sort_desc(u, lane);
            cs.th_spec = __shfl_sync(0xFFFFFFFFu, u, j - 1);
        } else {
            uint32_t xw, xk;
            warp_two_kth<E::KB, Q>(vk, Q, kw, k, &xw, &xk);
            if (lane == 0) sm.pub[warp] = xw;
            cs.st.th_own = xk;
            if (!gbar(sm, g)) return false;
        }
    }

    const uint32_t th = cs.spec ? max(cs.th_spec, cs.st.th_own) : max(cs.st.th_own, block_floor(sm, lane));
    const float thv = th == 0u ? -INFINITY : (float)E::key_value(th);
    // filter: one pass bit per element of this thread's vectors (bit q * VEC + j)
    static_assert(Q * E::VEC <= 64, "a thread's elements of a tile fit one mask");
    static_assert(Q * kConsumers * E::VEC * (int)sizeof(TIn) == kTileBytes, "a full tile is whole vectors");
    unsigned long long pm = 0ull;
    if (n == kTileBytes / (int)sizeof(TIn)) {
        // A full tile: the NaN-propagating maximum of each vector, then of the
        // thread's Q vectors (a tree); only when that reaches the threshold are
        // the vectors tested one by one.  A NaN anywhere makes the thread's
        // maximum NaN, which passes nothing and flags the row (whose outputs
        // are then the defaults of a non-finite sequence, whatever was appended).
        if constexpr (sizeof(TIn) == 2) {
            const __nv_bfloat162 th2 = __float2bfloat162_rn(thv);
            __nv_bfloat162 mq[Q];
#pragma unroll
            for (int q = 0; q < Q; ++q)
                mq[q] = __hmax2_nan(__hmax2_nan(as_bf2(v[q].x), as_bf2(v[q].y)),
                                    __hmax2_nan(as_bf2(v[q].z), as_bf2(v[q].w)));
            __nv_bfloat162 tm[Q];
#pragma unroll
            for (int q = 0; q < Q; ++q) tm[q] = mq[q];
#pragma unroll
            for (int w2 = Q / 2; w2 > 0; w2 >>= 1)
#pragma unroll
                for (int q = 0; q < w2; ++q) tm[q] = __hmax2_nan(tm[q], tm[q + w2]);
            cs.run_max = fmax_nan(cs.run_max, __bfloat162float(__hmax_nan(__low2bfloat16(tm[0]), __high2bfloat16(tm[0]))));
            if (__hge2_mask(tm[0], th2)) {
#pragma unroll
                for (int q = 0; q < Q; ++q)
                    if (__hge2_mask(mq[q], th2))
                        pm |= (unsigned long long)pass_mask(v[q], thv, (TIn*)nullptr) << (q * E::VEC);
            }
        } else {
            float mq[Q], tm[Q];
#pragma unroll
            for (int q = 0; q < Q; ++q) {
                mq[q] = vmax_nan(v[q], (TIn*)nullptr);
                tm[q] = mq[q];
            }
#pragma unroll
            for (int w2 = Q / 2; w2 > 0; w2 >>= 1)
#pragma unroll
                for (int q = 0; q < w2; ++q) tm[q] = fmax_nan(tm[q], tm[q + w2]);
            cs.run_max = fmax_nan(cs.run_max, tm[0]);
            if (tm[0] >= thv) {
#pragma unroll
                for (int q = 0; q < Q; ++q)
                    if (mq[q] >= thv) pm |= (unsigned long long)pass_mask(v[q], thv, (TIn*)nullptr) << (q * E::VEC);
            }
        }
    } else {
    typename RunOf<TIn>::type rs;
    run_init(rs, thv);
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        const int e0 = (q * kConsumers + t) * E::VEC;
        unsigned msk = 0u;
        if (e0 + E::VEC <= n) {
            if (vec_test(v[q], rs, false)) msk = pass_mask(v[q], thv, (TIn*)nullptr);
        } else if (e0 < n) {  // the tile's ragged end
#pragma unroll
            for (int j = 0; j < E::VEC; ++j) {
                const uint32_t bb = E::bits(v[q], j);
                if (e0 + j < n) {
                    cs.run_max = fmax_nan(cs.run_max, E::value(bb));
                    if (!E::bad(bb) && E::key(bb) >= th) msk |= 1u << j;
                }
            }
        }
        pm |= (unsigned long long)msk << (q * E::VEC);
    }
    cs.run_max = fmax_nan(cs.run_max, run_value(rs));
    }

    // append: what passed is read back from the tile (elem) by index
    if (__any_sync(0xFFFFFFFFu, pm != 0ull)) {
        int tot, pre;
        const int cl = __popcll(pm);
        if (__all_sync(0xFFFFFFFFu, cl <= 1)) {  // the usual case: at most one per lane, one ballot
            const unsigned bal = __ballot_sync(0xFFFFFFFFu, cl != 0);
            pre = __popc(bal & lanemask_lt());
            tot = __popc(bal);
        } else {
            pre = warp_prefix<7>((unsigned)cl, &tot);
        }
        if (cs.st.cnt + tot <= kWarpCap) {
            int slot = cs.st.cnt + pre;
            while (pm) {
                const int i = __ffsll((long long)pm) - 1;
                pm &= pm - 1ull;
                const int e = ((i / E::VEC) * kConsumers + t) * E::VEC + (i % E::VEC);
                L[slot++] = composite(E::key(E::load_bits(elem, e)), (uint32_t)(col0 + e));
            }
            cs.st.cnt += tot;
            cs.since += tot;
            cs.appended += tot;
        } else {
            // the list would overflow: append one element position at a time (at most
            // 32 entries) and cut the list to its exact top-k when it is full (a cut
            // leaves at most k <= kWarpCap - 32 entries)
#pragma unroll 1
            for (int i = 0; i < Q * E::VEC; ++i) {
                bool p = (pm >> i) & 1ull;
                unsigned bal = __ballot_sync(0xFFFFFFFFu, p);
                if (!bal) continue;
                const int e = ((i / E::VEC) * kConsumers + t) * E::VEC + (i % E::VEC);
                const uint32_t key = p ? E::key(E::load_bits(elem, e)) : 0u;
                if (cs.st.cnt + __popc(bal) > kWarpCap) {
                    cs.st = warp_refresh_out<E::KB>(sm, warp, lane, cs.st, k, kw);
                    cs.overflow = true;
                    cs.since = 0;
                    const uint32_t th2 = cs.spec ? max(cs.th_spec, cs.st.th_own)
                                                 : max(cs.st.th_own, block_floor(sm, lane));
                    p = p && key >= th2;
                    bal = __ballot_sync(0xFFFFFFFFu, p);
                }
                if (p) L[cs.st.cnt + __popc(bal & lanemask_lt())] = composite(key, (uint32_t)(col0 + e));
                cs.st.cnt += __popc(bal);
                cs.since += __popc(bal);
                cs.appended += __popc(bal);
            }
        }
    }

    if (!cs.spec && (cs.since > 0 || last)) {
        __syncwarp();
        cs.st = warp_refresh<E::KB>(sm, warp, lane, cs.st, k, kw, false);
        cs.since = 0;
    }
    return true;
}

// End of a piece: every warp's list goes to the workspace (at most kListCap
// entries together; else cut to exactly k).  A speculative piece is only
// accepted if at least k of its logits reached the threshold (or a list had to
// be cut, which needs more than k): then the piece's k-th largest logit is at
// or above it and every logit of the top-k was appended.
// Returns 1 when written, 0 when the speculation failed (nothing written, the
// piece must be redone conservatively), -1 when a barrier wait gave up.
template <int KB>
__device__ __forceinline__ int finish_piece(SelSmem& sm, GSync& g, const Args& a, int w, int b, int k, CState& cs, int warp,
                           int lane) {
    unsigned long long* L = sm.cand + warp * kWarpCap;
    if (!gbar(sm, g)) return -1;  // every warp's final estimate is published
    if (!cs.spec) {
        const uint32_t floor = block_floor(sm, lane);
        const int used = (cs.st.cnt + 31) >> 5;
        const unsigned lt = lanemask_lt();
        int base = 0;
        for (int m = 0; m < used; ++m) {  // drop what is below the final floor
            const int i = lane + 32 * m;
            const unsigned long long e = i < cs.st.cnt ? L[i] : 0ull;
            const bool keep = i < cs.st.cnt && comp_key(e) >= floor;
            const unsigned bal = __ballot_sync(0xFFFFFFFFu, keep);
            __syncwarp();
            if (keep) L[base + __popc(bal & lt)] = e;
            base += __popc(bal);
        }
        cs.st.cnt = base;
    }
    const bool nf = __any_sync(0xFFFFFFFFu, isnan(cs.run_max) || cs.run_max == INFINITY);
    if (lane == 0) {
        sm.scan[warp] = cs.st.cnt | (nf ? 0x10000 : 0) | (cs.overflow ? 0x20000 : 0);
        sm.red[warp] = cs.appended;
    }
    if (!gbar(sm, g)) return -1;
    int off = 0, total = 0, appended = 0;
    bool any_nf = false, any_overflow = false;
#pragma unroll
    for (int w2 = 0; w2 < kConsumerWarps; ++w2) {
        const int sv = sm.scan[w2];
        off += w2 < warp ? (sv & 0xFFFF) : 0;
        total += sv & 0xFFFF;
        any_nf |= (sv & 0x10000) != 0;
        any_overflow |= (sv & 0x20000) != 0;
        appended += sm.red[w2];
    }
    if (lane == 0) sm.pub[warp] = 0u;  // every warp has read the floor: reset for the next piece
    if (cs.spec && !any_overflow && appended < k) return 0;
    const uint32_t row_slot = (uint32_t)w / (uint32_t)a.ppr;
    unsigned long long* out = a.cand + (size_t)row_slot * a.cand_rowcap + (size_t)(w - row_slot * a.ppr) * kListCap;
    int written = total;
    if (total <= kListCap) {
        for (int i = lane; i < cs.st.cnt; i += 32) out[off + i] = L[i];
    } else {
        GSync g2 = g;  // the out-of-line call gets a copy, so g stays in registers
        written = piece_cut<KB>(sm, g2, warp, lane, cs.st.cnt, off, total, k, out);
        g = g2;
        if (!g.ok) return -1;
    }
    if (threadIdx.x == 0) {
        a.cand_cnt[w] = (uint32_t)written;
        if (any_nf) atomicOr(&a.seq_status[b], SV_ROW_NONFINITE);
    }
    return 1;
}

// A tile's vectors for this consumer straight from global memory (the redo of
// a piece): 16-byte loads when rows are 16-byte aligned, else element loads.
template <typename TIn, bool VEC16>
__device__ __forceinline__ void load_global_tile(const TIn* row, int col0, int n, int t,
                                                 uint4 (&v)[kTileBytes / 16 / kConsumers]) {
    using E = Elem<TIn>;
    constexpr int Q = kTileBytes / 16 / kConsumers;
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        const int e0 = (q * kConsumers + t) * E::VEC;
        if (VEC16) {
            v[q] = e0 < n ? __ldg(reinterpret_cast<const uint4*>(row + col0) + (q * kConsumers + t))
                          : make_uint4(0u, 0u, 0u, 0u);
        } else {
            uint32_t wd[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int j = 0; j < E::VEC; ++j) {
                if (e0 + j < n) {
                    uint32_t bits;
                    if (sizeof(TIn) == 2)
                        bits = __ldg(reinterpret_cast<const unsigned short*>(row + col0) + e0 + j);
                    else
                        bits = __ldg(reinterpret_cast<const unsigned int*>(row + col0) + e0 + j);
                    if (sizeof(TIn) == 2)
                        wd[j >> 1] |= bits << (16 * (j & 1));
                    else
                        wd[j] = bits;
                }
            }
            v[q] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
        }
    }
}

// The speculative threshold was too high for piece w (fewer than k logits
// reached it): do the piece again, conservatively, reading it straight from
// global memory.  Out of line, so that the main loop keeps its registers.
template <typename TIn, bool TMA>
__device__ __noinline__ bool redo_piece(SelSmem& sm, GSync& g, const Args& a, int w, int b, int k, int c0, int c1,
                                        int warp, int lane) {
    constexpr int TE = kTileBytes / (int)sizeof(TIn);
    const int V = a.V, G = a.G;
    const uint32_t item = a.stream_rows[(uint32_t)w / (uint32_t)a.ppr];
    const int r = (int)(item & 0xFFu);
    const int gamma = a.seq[b].gamma;
    const TIn* row = a.kseq ? (const TIn*)(r == 0 ? a.target : a.draft) + (size_t)b * V  // K-SEQ: [B, V] rows
                     : (r <= gamma) ? (const TIn*)a.target + ((size_t)b * (G + 1) + r) * (size_t)V
                                    : (const TIn*)a.draft + ((size_t)b * G + (r - gamma - 1)) * (size_t)V;
    CState cs;
    cs.spec = false;
    uint4 v[kTileBytes / 16 / kConsumers];
    for (int col = c0; col < c1; col += TE) {
        const int n = min(TE, c1 - col);
        load_global_tile<TIn, TMA>(row, col, n, threadIdx.x, v);
        if (!consume_tile<TIn>(sm, g, v, row + col, n, col, col == c0, col + n >= c1, (c1 - c0 + TE - 1) / TE, k, cs,
                               warp, lane))
            return false;
    }
    return finish_piece<Elem<TIn>::KB>(sm, g, a, w, b, k, cs, warp, lane) >= 0;
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
        mbar_init(&sm.gsync, kConsumerWarps);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (t < kConsumerWarps) sm.pub[t] = 0u;
    if (t == 0) sm.wait_ns = a.wait_ns;
    __syncthreads();
    grid_dependency_wait();  // the plan kernel's lists and counters
    grid_dependents_go();
    const uint32_t n_pieces = a.counts[kCntStreamRows] * (uint32_t)ppr;
    if (n_pieces == 0) return;  // no sequence takes this path (the same value for every thread)

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
                const TIn* row =
                    a.kseq ? (const TIn*)(r == 0 ? a.target : a.draft) + (size_t)b * V  // K-SEQ: [B, V] rows
                    : (r <= gamma) ? (const TIn*)a.target + ((size_t)b * (G + 1) + r) * (size_t)V
                                   : (const TIn*)a.draft + ((size_t)b * G + (r - gamma - 1)) * (size_t)V;
                const int c0 = piece * PE, c1 = min(V, c0 + PE);
                for (int col = c0, tile = 0; col < c1 && ok; col += TE, ++tile) {
                    const int n = min(TE, c1 - col);
                    if (!mbar_wait(&sm.empty[stage], ph, sm.wait_ns)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0) {
                        sm.hdr[stage] = make_int4((int)w, tile, n, col);
                        sm.seqk[stage] = make_int2(b, k);
                        sm.pce[stage] = make_int2(c1, (c1 - c0 + TE - 1) / TE);
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
            if (ok && mbar_wait(&sm.empty[stage], ph, sm.wait_ns)) {
                if (lane == 0) {
                    sm.hdr[stage] = make_int4(-1, 0, 0, 0);
                    mbar_arrive(&sm.full[stage]);
                }
            } else if (lane == 0) {
                atomicOr(&a.counts[kCntError], 1u);
                // let every copy already issued land before the CTA leaves (always
                // with the full limit: a copy in flight must not outlive the CTA)
                for (int s = 0; s < kStages; ++s)
                    if (issued[s] >= 0) (void)mbar_wait(&sm.full[s], (uint32_t)issued[s], kWaitLimitNs);
            }
        }
        return;
    }

    // ------------------------------ consumers ------------------------------
    int stage = 0;
    uint32_t ph = 0;
    GSync g{0u, true};
    int k = 1, b = 0;
    CState cs;
    cs.st = WarpList{0, 0u};
    while (true) {
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(&sm.full[stage], ph, sm.wait_ns))) {
            g.ok = false;
            break;
        }
        const int4 h = sm.hdr[stage];
        if (h.x < 0) break;
        const int2 bk = sm.seqk[stage];
        const int2 pc = sm.pce[stage];
        const int w = h.x, tile_idx = h.y, n = h.z, col0 = h.w;
        const int c1 = pc.x, tiles = pc.y;
        const int c0 = col0 - tile_idx * TE;
        const bool last = col0 + n >= c1;
        // this warp's vectors of the tile into registers; the stage goes straight back
        // this warp's vectors of the tile into registers; the stage goes back once the
        // few elements that pass have been read again
        const uint4* tile = reinterpret_cast<const uint4*>(sm.buf[stage]);
        uint4 v[Q];
#pragma unroll
        for (int q = 0; q < Q; ++q) v[q] = tile[q * kConsumers + t];
        if (tile_idx == 0) {
            b = bk.x;
            k = bk.y;
            cs.spec = spec_rank(k, tiles) > 0;
        }
        const bool ok = consume_tile<TIn>(sm, g, v, reinterpret_cast<const TIn*>(sm.buf[stage]), n, col0,
                                          tile_idx == 0, last, tiles, k, cs, warp, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[stage]);
        if (++stage == kStages) {
            stage = 0;
            ph ^= 1u;
        }
        if (!ok) break;
        if (!last) continue;

        int r = finish_piece<E::KB>(sm, g, a, w, b, k, cs, warp, lane);
        if (r < 0) break;
        if (r == 0) {
            GSync g2 = g;  // the out-of-line call gets a copy, so g stays in registers
            const bool ok = redo_piece<TIn, TMA>(sm, g2, a, w, b, k, c0, c1, warp, lane);
            g = g2;
            if (!ok) break;
        }
    }
    if (!g.ok && lane == 0) atomicOr(&a.counts[kCntError], 1u);
}


// ---------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------
namespace {
template <typename TIn, bool TMA>
cudaError_t launch_t(const Args& a, int sms, cudaStream_t s, void* const ev[2]) {
    auto sel = select_kernel<TIn, TMA>;
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
    cudaError_t e = launch_pdl(sel, dim3((unsigned)grid), dim3(kSelThreads), (size_t)smem, s, a);
    if (e != cudaSuccess) return e;
    if (ev && ev[1]) cudaEventRecord((cudaEvent_t)ev[1], s);
    return launch_combine_kernel(sizeof(TIn) == 2 ? SV_BF16 : SV_F32, a, sms, s);
}
}  // namespace

cudaError_t launch_stream_kernel(int dtype, bool vector, const Args& a, int sms, cudaStream_t s, void* const ev[2]) {
    if (dtype == SV_BF16)
        return vector ? launch_t<__nv_bfloat16, true>(a, sms, s, ev) : launch_t<__nv_bfloat16, false>(a, sms, s, ev);
    return vector ? launch_t<float, true>(a, sms, s, ev) : launch_t<float, false>(a, sms, s, ev);
}

}  // namespace sv
