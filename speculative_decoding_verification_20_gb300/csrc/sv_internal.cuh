// sv_internal.cuh -- shared device/host internals of the GB300 verification library.
//
// Layout of one call on the GPU (all on the caller's stream, no host sync;
// each kernel after the plan is a programmatic dependent launch):
//   plan kernel    (1 CTA)  validates the per-sequence parameters, picks a path
//                           per sequence, zeroes the per-call counters and
//                           writes the work lists;
//   select kernel           top-k <= 256 (and greedy) sequences: rows are cut
//                           into pieces of up to 10 x 28 KB tiles, streamed
//                           once from HBM by TMA bulk copies into a shared-
//                           memory ring; each piece keeps a superset of its
//                           top-k (logit key, token id) candidates;
//   combine kernel          a warp pair per (target row, draft row) unit merges
//                           the pieces' lists into the exact top-k and does the
//                           per-position arithmetic (softmax over the kept
//                           logits, top-p, alpha, acceptance, residual draw);
//   free kernel             sequences with no top-k and temperature > 0 (top-p
//                           or none): each unit's two rows are streamed through
//                           a ring by TMA, once for the row statistics, three
//                           more times for an exact nucleus cut when top-p < 1,
//                           and once for alpha and the residual weights, summed
//                           per 2 KB block into a per-unit record;
//   free tail kernel        a warp per unit of the free kernel: residual draw
//                           (block search, re-read of one block), acceptance;
//   dense kernel            every other sequence (large top-k, and units the
//                           free kernel hands over): one thread-block cluster
//                           holds a whole unit in registers (DSMEM reductions).
// The last unit of a sequence to finish writes that sequence's outputs
// (last-block-done counters; no thread ever waits on another block).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "spec_verify.h"

namespace sv {

// ---------------------------------------------------------------------------
// configuration
// ---------------------------------------------------------------------------
constexpr int kPlanThreads = 1024;
// default limit of every bounded wait (an mbarrier phase, a peer warp): 2 s
constexpr unsigned long long kWaitLimitNs = 2000000000ull;
constexpr int kTileBytes = 28672;   // one TMA bulk copy: 7 16-byte vectors per consumer thread
constexpr int kTilesPerPiece = 10;  // a piece of a row: up to 280 KB of logits (a whole 128k bf16 row)
constexpr int kStreamMaxK = SV_STREAM_MAX_TOP_K;
constexpr int kListCap = 512;   // candidates one piece hands to the combine kernel
constexpr int kSortCap = 2048;  // candidates per row sorted in shared memory by the combine kernel
constexpr int kDenseThreads = 256;
// free kernel geometry: each consumer warp owns a contiguous 2 KB block of a
// ring segment, so block j of a row always starts at token j * block_elems.
// The kernel runs with 7 consumer warps (a 14 KB segment, 2 CTAs per SM) or,
// for batches with fewer units than those CTA slots, with 15 (30 KB, 1 CTA per
// SM, twice the warps per unit).
constexpr int kFreeBlockBytes = 2048;
constexpr int kFreeWarpsNarrow = 7;
constexpr int kFreeWarpsWide = 15;

// counters at the head of the workspace list area
enum : int {
    kCntStreamRows = 0,
    kCntDenseUnits = 1,
    kCntStreamUnits = 2,
    kCntPieceNext = 3,
    kCntError = 4,
    kCntFreeUnits = 5,
    kCntFreeNext = 6,
    kCntGumUnits = 7,
    kCntFreeNucUnits = 8  // whole-row units with top-p < 1: the only ones that can be handed over
};

// streaming top-k path; cluster path (top-k > 256, and handed-over units);
// whole-row path of rows with no top-k (with or without top-p); shared-noise
// rows with no filter at all (one pass of noise and argmax)
enum : uint32_t { kModeErr = 0, kModeStream = 1, kModeDense = 2, kModeFree = 3, kModeGumbel = 4 };

// Per-unit record of the free kernel for its tail kernel (one per entry of the
// free unit list).  flags: kRecDead (a row without a finite logit, or with a
// NaN / +inf), kRecFall (the unit was handed to the dense kernel).
enum : uint32_t { kRecDead = 1u, kRecFall = 2u };
struct FreeRec {
    float Mp, Mq;                   // row maxima (logits)
    float invp, invq;               // 1 / (sum x kept mass) of each row
    unsigned long long cutp, cutq;  // last kept element (okey << 32 | ~id); 0: the row is not cut
    uint32_t flags;
    float alpha[kFreeWarpsWide];    // per-warp partial sums of min(p, q) (0 past the kernel's warps)
};
static_assert(sizeof(FreeRec) == 96, "free record size");

// per-sequence plan (32 bytes)
struct SeqInfo {
    uint32_t mode;
    uint32_t status;
    int32_t gamma;
    int32_t k;        // effective top-k (0 = off); 1 for greedy
    float T;          // temperature (0 = greedy)
    float P;          // effective top-p (1 = off)
    uint32_t row_off; // index of this sequence's first row in the stream row list
    float L;          // lenience in [0, 1] (1 = the exact rule)
};

// Everything a kernel needs, passed by value.
struct Args {
    const void* target;
    const void* draft;
    const int32_t* draft_tokens;
    const int32_t* num_draft;
    const float* temperature;
    const int32_t* top_k;
    const float* top_p;
    const float* lenience;  // [B] or nullptr (1 everywhere)
    uint64_t seed;
    unsigned long long wait_ns;  // limit of each bounded wait on another warp (kWaitLimitNs by default)
    int B, G, V;
    int32_t* accepted_len;
    int32_t* out_tokens;
    float* alpha;
    float* p_out;
    float* q_out;
    uint32_t* row_status;
    int32_t* pos_accept;
    int32_t* pos_token;
    int force_dense;
    int gumbel;  // shared-noise verification: target rows only, accept iff x = argmax(log p + g)
    int kseq;    // K-SEQ: one position per row ([B, V] rows), draft_tokens = the k candidates
    int ppr;  // stream pieces per row
    // workspace
    SeqInfo* seq;
    uint32_t* seq_done;
    uint32_t* seq_status;
    int32_t* unit_acc;
    int32_t* unit_tok;
    uint32_t* stream_rows;
    uint32_t* dense_units;
    uint32_t* stream_units;
    uint32_t* free_units;
    uint32_t* counts;         // kCnt* above
    unsigned long long* cand; // per stream row, cand_rowcap entries: piece j's list at j * kListCap
                              // (key << 32 | ~id, unsorted), each at most min(kListCap, piece length)
    uint32_t* cand_cnt;       // [stream rows * ppr]
    int cand_rowcap;          // candidate entries reserved per stream row
    FreeRec* free_rec;        // [units] by free list index
    float* free_blk;          // [units][2][free_nblk]: per block sums of r (residual weights) and p
    int free_nblk;            // blocks per row of the free kernel's variant (set by its launcher)
    int free_warps;           // consumer warps of that variant (set by its launcher)
    uint32_t* gum_units;      // shared-noise rows with no filter: (b << 8) | position
    unsigned long long* gum_key;  // [gum units] best (score, id) key so far (score_key; 0 = none)
    uint32_t* gum_cnt;        // [gum units] CTAs done with their part of the unit's row
};

struct WsLayout {
    size_t seq, seq_done, seq_status, unit_acc, unit_tok, stream_rows, dense_units, stream_units, free_units,
        counts, cand, cand_cnt, free_rec, free_blk, gum_units, gum_key, gum_cnt, total;
    int ppr, free_nblk;
    int cand_rowcap;  // candidate entries per stream row: kListCap per piece, the last piece min(kListCap, its length)
};

__host__ __device__ inline int tile_elems(int dtype) { return kTileBytes / (dtype == SV_BF16 ? 2 : 4); }
__host__ __device__ inline int stream_piece_elems(int dtype) { return kTilesPerPiece * tile_elems(dtype); }
// the combine kernel sorts all pieces' lists of a row at once
static_assert(((SV_MAX_VOCAB + kTilesPerPiece * (kTileBytes / 4) - 1) / (kTilesPerPiece * (kTileBytes / 4))) *
                      kListCap <=
                  kSortCap,
              "pieces per row times the list cap must fit the combine sort");

// blocks per row written by the free kernel with `warps` consumer warps (whole segments)
__host__ __device__ inline int free_blocks(int V, int dtype, int warps) {
    const int seg = warps * (kFreeBlockBytes / (dtype == SV_BF16 ? 2 : 4));
    return (V + seg - 1) / seg * warps;
}

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline WsLayout ws_layout(int B, int G, int V, int dtype) {
    WsLayout L{};
    size_t o = 0;
    const size_t rows = (size_t)B * (2 * G + 1);
    const size_t units = (size_t)B * (G + 1);
    L.ppr = (V + stream_piece_elems(dtype) - 1) / stream_piece_elems(dtype);
    L.seq = o;         o = align_up(o + sizeof(SeqInfo) * B, 256);
    L.seq_done = o;    o = align_up(o + 4 * (size_t)B, 256);
    L.seq_status = o;  o = align_up(o + 4 * (size_t)B, 256);
    L.unit_acc = o;    o = align_up(o + 4 * (size_t)B * G, 256);
    L.unit_tok = o;    o = align_up(o + 4 * units, 256);
    L.stream_rows = o; o = align_up(o + 4 * rows, 256);
    L.dense_units = o; o = align_up(o + 4 * units, 256);
    L.stream_units = o; o = align_up(o + 4 * units, 256);
    L.free_units = o;  o = align_up(o + 4 * units, 256);
    L.counts = o;      o = align_up(o + 64, 256);
    L.cand_cnt = o;    o = align_up(o + 4 * rows * L.ppr, 256);
    {  // a piece's list never holds more entries than the piece has logits
        const int last_len = V - (L.ppr - 1) * stream_piece_elems(dtype);
        L.cand_rowcap = (L.ppr - 1) * kListCap + (last_len < kListCap ? last_len : kListCap);
    }
    L.cand = o;        o = align_up(o + 8 * rows * (size_t)L.cand_rowcap, 256);
    L.free_nblk = free_blocks(V, dtype, kFreeWarpsNarrow) > free_blocks(V, dtype, kFreeWarpsWide)
                      ? free_blocks(V, dtype, kFreeWarpsNarrow)
                      : free_blocks(V, dtype, kFreeWarpsWide);  // room for either variant
    L.free_rec = o;    o = align_up(o + sizeof(FreeRec) * units, 256);
    L.free_blk = o;    o = align_up(o + 4 * units * 2 * (size_t)L.free_nblk, 256);
    L.gum_units = o;   o = align_up(o + 4 * units, 256);
    L.gum_key = o;     o = align_up(o + 8 * units, 256);
    L.gum_cnt = o;     o = align_up(o + 4 * units, 256);
    L.total = o;
    return L;
}

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
#ifdef __CUDACC__

// wait for the previous kernel of the call (a no-op when launched without a
// programmatic dependency), and let the next one be scheduled
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dependents_go() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): 10 rounds of two 32x32->64
// multiplies with the Weyl-bumped key; only output word 0 is used here.
__device__ __forceinline__ uint32_t philox_w0(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                              uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t a_lo = 0xD2511F53u * c0, a_hi = __umulhi(0xD2511F53u, c0);
        const uint32_t b_lo = 0xCD9E8D57u * c2, b_hi = __umulhi(0xCD9E8D57u, c2);
        c0 = b_hi ^ c1 ^ k0;
        c1 = b_lo;
        c2 = a_hi ^ c3 ^ k1;
        c3 = a_lo;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c0;
}

// Acceptance under lenience L ("Fast Inference from Transformers via
// Speculative Decoding" review page, section Lenience: q(x) is multiplied by L
// in the test): accept iff u * (L * q(x)) < p(x), formed in double.  L = 1 is
// the exact rule u * q(x) < p(x).
__device__ __forceinline__ bool lenient_accept(double u, float L, double qx, double px) {
    return u * ((double)L * qx) < px;
}
// 1 / L for the acceptance mass below (a huge finite value for L = 0, so that
// 0 * invl stays 0); exactly 1 for L = 1.
__device__ __forceinline__ float lenience_inv(float L) { return L > 0.0f ? 1.0f / L : 3.0e38f; }
// Acceptance mass of one token, q(x) P(accept | x) = min(q(x), p(x) / L); with
// L = 1 it is min(p(x), q(x)) bit for bit.
__device__ __forceinline__ float accept_mass(float p, float q, float invl) { return fminf(q, p * invl); }

// All four output words of the same block function.
__device__ __forceinline__ uint4 philox4(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                         uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t a_lo = 0xD2511F53u * c0, a_hi = __umulhi(0xD2511F53u, c0);
        const uint32_t b_lo = 0xCD9E8D57u * c2, b_hi = __umulhi(0xCD9E8D57u, c2);
        c0 = b_hi ^ c1 ^ k0;
        c1 = b_lo;
        c2 = a_hi ^ c3 ^ k1;
        c3 = a_lo;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return make_uint4(c0, c1, c2, c3);
}

// Gumbel noise g = -ln(-ln u) of a uniform u = ((w >> 8) + 1/2) 2^-24 given by its
// Philox word w ("Speculative decoding: the art of guessing well", section
// 共享噪声的采样: sampling from softmax(l) is argmax(l + g)).  In fp32 with
// every input exact: for u < 1/2, u itself is exact and -ln u = -log2(u) ln 2
// (relative error about 2^-22); for u >= 1/2, 1 - u = (2 (2^24 - a) - 1) 2^-25 is
// exact and -ln u = -log1p(-(1 - u)) to about an ulp.  Then g = -log2(L) ln 2:
// an absolute error of a few 1e-6 at most (at the largest g), far below the
// 1e-4 gap by which decisions are compared with the fp64 oracle.
__device__ __forceinline__ float gumbel_of_word(uint32_t w) {
    const uint32_t a = w >> 8;
    float L;
    if (a < (1u << 23)) {
        const float u = ((float)a + 0.5f) * 5.9604644775390625e-8f;  // (a + 1/2) 2^-24, exact
        L = -__log2f(u) * 0.693147180559945309f;
    } else {
        const float y = (float)(2u * ((1u << 24) - a) - 1u) * 2.98023223876953125e-8f;  // 1 - u, exact
        L = -log1pf(-y);
    }
    return -__log2f(L) * 0.693147180559945309f;
}

// (score, token id) as one 64-bit key whose maximum is the largest score and,
// among equal scores, the lowest id: the argmax rule of the shared-noise test.
// A NaN score never wins (it maps below -inf).
__device__ __forceinline__ unsigned long long score_key(float s, uint32_t id) {
    const uint32_t bits = __float_as_uint(s);
    uint32_t k = (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
    if (s != s) k = 0u;
    return ((unsigned long long)k << 32) | (unsigned long long)(~id);
}
__device__ __forceinline__ int score_key_id(unsigned long long k) { return (int)(~(uint32_t)k); }

// U(seed, b, pos, draw) = ((w >> 8) + 0.5) * 2^-24 (exact in double)
__device__ __forceinline__ double uniform01(uint64_t seed, uint32_t b, uint32_t pos, uint32_t draw) {
    const uint32_t w = philox_w0(b, pos, draw, 0u, (uint32_t)seed, (uint32_t)(seed >> 32));
    return ((double)(w >> 8) + 0.5) * (1.0 / 16777216.0);
}

// Order-preserving unsigned keys of float bit patterns; -0 is folded onto +0
// so equal values get equal keys.
__device__ __forceinline__ uint32_t okey32(uint32_t bits) {
    bits = (bits == 0x80000000u) ? 0u : bits;
    return (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
}
__device__ __forceinline__ uint32_t okey16(uint32_t h) {
    h = (h == 0x8000u) ? 0u : h;
    return (h & 0x8000u) ? (~h & 0xFFFFu) : (h | 0x8000u);
}
__device__ __forceinline__ float key_value32(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
__device__ __forceinline__ float key_value16(uint32_t k) {
    const uint32_t h = (k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu);
    return __uint_as_float(h << 16);
}
// NaN or +inf (-inf is a legal, masked logit)
__device__ __forceinline__ bool bad32(uint32_t bits) {
    return ((bits & 0x7FFFFFFFu) > 0x7F800000u) || bits == 0x7F800000u;
}
__device__ __forceinline__ bool bad16(uint32_t h) { return ((h & 0x7FFFu) > 0x7F80u) || h == 0x7F80u; }

// streaming 16-byte load: read once, do not keep in L1
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

#endif  // __CUDACC__

// host launchers, one per kernel translation unit
cudaError_t launch_stream_kernel(int dtype, bool vector, const Args& a, int sms, cudaStream_t s, void* const ev[2]);

// Programmatic dependent launch: every kernel after the plan kernel is
// launched so that it may start (and run its prologue) while the previous
// kernel of the call is finishing; it waits for that kernel's completion and
// memory with grid_dependency_wait() before reading anything it produced.
// Each kernel lets the next one be scheduled once all its own blocks run.
template <typename K>
inline cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t s, const Args& a,
                              const cudaLaunchAttribute* extra = nullptr, int n_extra = 0) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[4];
    int n = 0;
    for (int i = 0; i < n_extra && n < 3; ++i) attr[n++] = extra[i];
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = (unsigned)n;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}
cudaError_t launch_combine_kernel(int dtype, const Args& a, int sms, cudaStream_t s);
cudaError_t launch_free_kernel(int dtype, bool vector, const Args& a, int sms, cudaStream_t s, void* const ev[2]);
cudaError_t launch_gumbel_kernel(int dtype, bool vector, const Args& a, int sms, cudaStream_t s, void* const ev[2]);
cudaError_t launch_dense_f32(bool vector, const Args& a, int sms, cudaStream_t s);
cudaError_t launch_dense_bf16(bool vector, const Args& a, int sms, cudaStream_t s);

}  // namespace sv
