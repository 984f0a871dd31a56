// spec_verify.cu -- host side of the C ABI declared in include/spec_verify.h.
//
// Validates arguments on the host (nothing is enqueued on an error), then
// enqueues on the caller's stream: plan kernel -> (shared-noise calls: the
// one-pass kernel ->) select (streaming top-k) -> combine -> whole-row kernel ->
// its per-unit tail -> dense cluster kernel, each after the plan as a
// programmatic dependent launch.  No host synchronisation (spec_verify_host
// excepted).
#include <cuda_runtime.h>

#include <cstdio>
#include <cstring>
#include <mutex>

#include "sv_finalize.cuh"

namespace sv {


// ---------------------------------------------------------------------------
// plan kernel: one CTA walks the batch in chunks of blockDim.x (<= 1024) sequences.
// ---------------------------------------------------------------------------
// Exclusive block scans of N per-thread counts at once (thread order), with the
// block totals; the N shuffle ladders run side by side.
template <int N>
__device__ __forceinline__ void block_excl_scan_n(const uint32_t (&v)[N], uint32_t (*s_warp)[N], uint32_t (&before)[N],
                                                  uint32_t (&total)[N]) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (int)(blockDim.x >> 5);
    uint32_t x[N];
#pragma unroll
    for (int i = 0; i < N; ++i) x[i] = v[i];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1)
#pragma unroll
        for (int i = 0; i < N; ++i) {
            const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x[i], o);
            if (lane >= o) x[i] += y;
        }
    if (lane == 31)
#pragma unroll
        for (int i = 0; i < N; ++i) s_warp[wid][i] = x[i];
    __syncthreads();
    if (wid == 0) {
        uint32_t w[N];
#pragma unroll
        for (int i = 0; i < N; ++i) w[i] = lane < nw ? s_warp[lane][i] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1)
#pragma unroll
            for (int i = 0; i < N; ++i) {
                const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, w[i], o);
                if (lane >= o) w[i] += y;
            }
#pragma unroll
        for (int i = 0; i < N; ++i) s_warp[lane][i] = w[i];  // inclusive warp-total prefix
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < N; ++i) {
        before[i] = (wid > 0 ? s_warp[wid - 1][i] : 0u) + x[i] - v[i];
        total[i] = s_warp[nw - 1][i];
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(Args a) {
    __shared__ uint32_t s_warp[32][6];
    grid_dependents_go();
    uint32_t base_rows = 0, base_units = 0, base_sunits = 0, base_funits = 0, base_gunits = 0, n_fnuc = 0;
    const int G = a.G, V = a.V;
    for (int b0 = 0; b0 < a.B; b0 += blockDim.x) {
        const int b = b0 + threadIdx.x;
        uint32_t nrows = 0, nunits = 0, st = 0, mode = kModeErr;
        int gamma = 0, k = 0;
        float T = 0.0f, P = 1.0f, L = 1.0f;
        if (b < a.B) {
            gamma = a.num_draft ? a.num_draft[b] : G;
            T = a.temperature[b];
            const int kr = a.top_k ? a.top_k[b] : 0;
            const float pr = a.top_p ? a.top_p[b] : 1.0f;
            L = a.lenience ? a.lenience[b] : 1.0f;
            if (!(T >= 0.0f) || isinf(T)) st |= SV_ROW_BAD_TEMPERATURE;
            if (kr < 0) st |= SV_ROW_BAD_TOP_K;
            if (!(pr > 0.0f && pr <= 1.0f)) st |= SV_ROW_BAD_TOP_P;
            if (!(L >= 0.0f && L <= 1.0f)) st |= SV_ROW_BAD_LENIENCE;
            if (gamma < 1 || gamma > G) {
                st |= SV_ROW_BAD_NUM_DRAFT;
            } else {
                const int32_t* tok = a.draft_tokens + (size_t)b * G;
                for (int i0 = 0; i0 < gamma; i0 += 8) {  // independent loads, 8 at a time
                    int x[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) x[j] = i0 + j < gamma ? tok[i0 + j] : 0;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        if (x[j] < 0 || x[j] >= V) st |= SV_ROW_BAD_DRAFT_TOKEN;
                }
            }
            k = (kr > 0 && kr < V) ? kr : 0;
            P = (pr < 1.0f) ? pr : 1.0f;
            if (!st) {
                if (T == 0.0f) {  // greedy: one-hot argmax, filters do not change it
                    k = 1;
                    P = 1.0f;
                }
                const bool stream = (k >= 1 && k <= kStreamMaxK);
                // no top-k: the whole-row kernel (with the nucleus cut when top-p < 1)
                mode = a.force_dense ? kModeDense : stream ? kModeStream : k == 0 ? kModeFree : kModeDense;
                // K-SEQ: one unit per row; top-k rows from their kept lists (select +
                // combine), the others held by a cluster
                if (a.kseq && mode != kModeStream) mode = kModeDense;
                // shared noise on a row with no filter: one pass of noise and argmax
                if (a.gumbel && mode == kModeFree && !(P < 1.0f)) mode = kModeGumbel;
                if (mode == kModeStream)
                    nrows = a.kseq ? 2 : a.gumbel ? gamma + 1 : 2 * gamma + 1;  // shared noise: target rows only
                else if (mode == kModeDense)
                    nunits = a.kseq ? 1 : gamma + 1;
            }
        }
        const uint32_t nsunits = (mode == kModeStream) ? (a.kseq ? 1u : (uint32_t)(gamma + 1)) : 0u;
        const uint32_t nfunits = (mode == kModeFree) ? (uint32_t)(gamma + 1) : 0u;
        const uint32_t ngunits = (mode == kModeGumbel) ? (uint32_t)(gamma + 1) : 0u;
        const uint32_t nfnuc = (mode == kModeFree && P < 1.0f) ? nfunits : 0u;
        // the six work lists' offsets and totals in one pass
        const uint32_t cnt[6] = {nrows, nunits, nsunits, nfunits, ngunits, nfnuc};
        uint32_t off[6], tot[6];
        block_excl_scan_n<6>(cnt, s_warp, off, tot);
        const uint32_t off_r = off[0], off_u = off[1], off_s = off[2], off_f = off[3], off_g = off[4];
        const uint32_t tot_r = tot[0], tot_u = tot[1], tot_s = tot[2], tot_f = tot[3], tot_g = tot[4], tot_n = tot[5];
        if (b < a.B) {
            SeqInfo si;
            si.mode = mode;
            si.status = st;
            si.gamma = gamma;
            si.k = k;
            si.T = T;
            si.P = P;
            si.row_off = base_rows + off_r;
            si.L = L;
            a.seq[b] = si;
            a.seq_done[b] = 0;
            a.seq_status[b] = st;
            for (uint32_t r = 0; r < nrows; ++r) a.stream_rows[base_rows + off_r + r] = ((uint32_t)b << 8) | r;
            for (uint32_t u = 0; u < nunits; ++u) a.dense_units[base_units + off_u + u] = ((uint32_t)b << 8) | u;
            for (uint32_t u = 0; u < nsunits; ++u) a.stream_units[base_sunits + off_s + u] = ((uint32_t)b << 8) | u;
            for (uint32_t u = 0; u < nfunits; ++u) a.free_units[base_funits + off_f + u] = ((uint32_t)b << 8) | u;
            for (uint32_t u = 0; u < ngunits; ++u) {
                const uint32_t w = base_gunits + off_g + u;
                a.gum_units[w] = ((uint32_t)b << 8) | u;
                a.gum_key[w] = 0ull;
                a.gum_cnt[w] = 0u;
            }
            if (a.kseq) {  // outputs [B]: the token and the accepted candidate's index
                if (st) {
                    a.accepted_len[b] = -1;
                    a.out_tokens[b] = -1;
                    if (a.row_status) a.row_status[b] = st;
                }
            } else {
                const int first_pad = st ? 0 : gamma;
                for (int i = first_pad; i < G; ++i) {
                    if (a.alpha) a.alpha[(size_t)b * G + i] = 0.0f;
                    if (a.pos_accept) a.pos_accept[(size_t)b * G + i] = -1;
                }
                if (a.pos_token)
                    for (int j = st ? 0 : gamma + 1; j <= G; ++j) a.pos_token[(size_t)b * (G + 1) + j] = -1;
                if (st) {
                    a.accepted_len[b] = 0;
                    for (int j = 0; j <= G; ++j) a.out_tokens[(size_t)b * (G + 1) + j] = -1;
                    if (a.row_status) a.row_status[b] = st;
                }
            }
        }
        base_rows += tot_r;
        base_units += tot_u;
        base_sunits += tot_s;
        base_funits += tot_f;
        base_gunits += tot_g;
        n_fnuc += tot_n;
    }
    if (threadIdx.x == 0) {
        a.counts[kCntStreamRows] = base_rows;
        a.counts[kCntDenseUnits] = base_units;
        a.counts[kCntStreamUnits] = base_sunits;
        a.counts[kCntFreeUnits] = base_funits;
        a.counts[kCntGumUnits] = base_gunits;
        a.counts[kCntFreeNucUnits] = n_fnuc;
        a.counts[kCntFreeNext] = 0u;
        a.counts[kCntPieceNext] = 0u;
        a.counts[kCntError] = 0u;
    }
}


namespace {

struct DeviceInfo {
    int sms = 0;
    bool ok = false;
};

// SM count of device `dev`, cached for the first 64 devices (a device
// attribute: it outlives any context); queried each time beyond them.
DeviceInfo device_info(int dev) {
    static DeviceInfo infos[64];
    static std::mutex mu;
    if (dev < 0 || dev >= 64) {
        DeviceInfo d;
        if (dev >= 0 && cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess)
            d.ok = d.sms > 0;
        return d;
    }
    std::lock_guard<std::mutex> lock(mu);
    DeviceInfo& d = infos[dev];
    if (!d.ok) {
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) d.sms = 0;
        d.ok = d.sms > 0;
    }
    return d;
}

cudaError_t launch_all(int dtype, bool vector, const Args& a, int sms, cudaStream_t s, const sv_options& o) {
    cudaError_t e;
    if (a.gumbel && (e = launch_gumbel_kernel(dtype, vector, a, sms, s, o.ev_gumbel)) != cudaSuccess) return e;
    if ((e = launch_stream_kernel(dtype, vector, a, sms, s, o.ev_stream)) != cudaSuccess) return e;
    if ((e = launch_free_kernel(dtype, vector, a, sms, s, o.ev_free)) != cudaSuccess) return e;
    if (o.ev_dense[0]) cudaEventRecord((cudaEvent_t)o.ev_dense[0], s);
    e = (dtype == SV_BF16) ? launch_dense_bf16(vector, a, sms, s) : launch_dense_f32(vector, a, sms, s);
    if (e != cudaSuccess) return e;
    if (o.ev_dense[1]) cudaEventRecord((cudaEvent_t)o.ev_dense[1], s);
    return cudaSuccess;
}

int check_shape(int B, int G, int V, int dtype) {
    if (dtype != SV_F32 && dtype != SV_BF16) return SV_EUNSUPPORTED;
    if (B < 0 || G < 1 || V < 1) return SV_EINVAL;
    if (B > SV_MAX_BATCH || G > SV_MAX_GAMMA || V > SV_MAX_VOCAB) return SV_ETOO_LARGE;
    return SV_OK;
}

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" size_t spec_verify_workspace_size(int B, int gamma_max, int V, int dtype) {
    if (check_shape(B, gamma_max, V, dtype) != SV_OK) return 0;
    return ws_layout(B, gamma_max, V, dtype).total;
}

extern "C" const char* spec_verify_strerror(int status) {
    switch (status) {
        case SV_OK: return "success";
        case SV_EINVAL: return "invalid argument (null pointer, bad size or misaligned buffer)";
        case SV_EUNSUPPORTED: return "unsupported argument combination (dtype)";
        case SV_ECUDA: return "a CUDA launch or runtime call failed";
        case SV_ETOO_LARGE: return "shape beyond the supported maximum (B, gamma_max or V)";
        case SV_EWORKSPACE: return "workspace missing or smaller than spec_verify_workspace_size()";
        case SV_ESCRATCH:
            return "shape needs more scratch than spec_verify_static's fixed buffer (SV_STATIC_SCRATCH_BYTES); "
                   "use spec_verify with a workspace";
        default: return "unknown status";
    }
}

namespace {
// One call of either verification rule: arguments checked on the host, then the
// plan and the path kernels enqueued on `stream`.  gumbel: shared-noise
// verification (target rows only; no draft logits, alpha or probabilities).
int verify_call(const void* target_logits, const void* draft_logits, int dtype, const int32_t* draft_tokens,
                const int32_t* num_draft, const float* temperature, const int32_t* top_k, const float* top_p,
                uint64_t seed, int B, int gamma_max, int V, int32_t* accepted_len, int32_t* out_tokens, float* alpha,
                float* p_out, float* q_out, uint32_t* row_status, void* workspace, size_t workspace_bytes,
                void* stream, const sv_options* options, bool gumbel, bool kseq = false) {
    const int rc = check_shape(B, gamma_max, V, dtype);
    if (rc != SV_OK) return rc;
    if (kseq && gamma_max > SV_MAX_KSEQ) return SV_ETOO_LARGE;
    if (B == 0) return SV_OK;
    if (!target_logits || !draft_tokens || !temperature || !accepted_len || !out_tokens) return SV_EINVAL;
    if (!gumbel && (!draft_logits || !alpha)) return SV_EINVAL;
    if (((uintptr_t)target_logits & 15u) || (!gumbel && ((uintptr_t)draft_logits & 15u))) return SV_EINVAL;
    if (options && options->struct_size < sizeof(uint32_t)) return SV_EINVAL;
    // K-SEQ rows are single positions: the workspace of one draft position per row
    const WsLayout L = kseq ? ws_layout(B, 1, V, dtype) : ws_layout(B, gamma_max, V, dtype);
    if (!workspace || workspace_bytes < L.total) return SV_EWORKSPACE;
    if ((uintptr_t)workspace & 255u) return SV_EINVAL;

    sv_options opt;
    memset(&opt, 0, sizeof opt);
    if (options) memcpy(&opt, options, options->struct_size < sizeof opt ? options->struct_size : sizeof opt);

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SV_ECUDA;
    const DeviceInfo di = device_info(dev);
    if (!di.ok) return SV_ECUDA;
    cudaStream_t s = (cudaStream_t)stream;

    char* ws = (char*)workspace;
    Args a;
    memset(&a, 0, sizeof a);
    a.target = target_logits;
    a.draft = gumbel ? target_logits : draft_logits;  // never read by the shared-noise rule
    a.draft_tokens = draft_tokens;
    a.num_draft = num_draft;
    a.temperature = temperature;
    a.top_k = top_k;
    a.top_p = top_p;
    a.lenience = gumbel ? nullptr : opt.lenience;
    a.seed = seed;
    a.wait_ns = opt.wait_limit_ns ? (unsigned long long)opt.wait_limit_ns : kWaitLimitNs;
    a.B = B;
    a.G = gamma_max;
    a.V = V;
    a.accepted_len = accepted_len;
    a.out_tokens = out_tokens;
    a.alpha = (gumbel || kseq) ? nullptr : alpha;
    a.p_out = gumbel ? nullptr : p_out;
    a.q_out = gumbel ? nullptr : q_out;
    a.row_status = row_status;
    a.pos_accept = opt.pos_accept;
    a.pos_token = opt.pos_token;
    a.force_dense = opt.path == SV_PATH_DENSE;
    a.gumbel = gumbel ? 1 : 0;
    a.kseq = kseq ? 1 : 0;
    a.ppr = L.ppr;
    a.seq = (SeqInfo*)(ws + L.seq);
    a.seq_done = (uint32_t*)(ws + L.seq_done);
    a.seq_status = (uint32_t*)(ws + L.seq_status);
    a.unit_acc = (int32_t*)(ws + L.unit_acc);
    a.unit_tok = (int32_t*)(ws + L.unit_tok);
    a.stream_rows = (uint32_t*)(ws + L.stream_rows);
    a.dense_units = (uint32_t*)(ws + L.dense_units);
    a.stream_units = (uint32_t*)(ws + L.stream_units);
    a.free_units = (uint32_t*)(ws + L.free_units);
    a.counts = (uint32_t*)(ws + L.counts);
    a.cand = (unsigned long long*)(ws + L.cand);
    a.cand_rowcap = L.cand_rowcap;
    a.cand_cnt = (uint32_t*)(ws + L.cand_cnt);
    a.free_rec = (FreeRec*)(ws + L.free_rec);
    a.free_blk = (float*)(ws + L.free_blk);
    a.free_nblk = L.free_nblk;
    a.gum_units = (uint32_t*)(ws + L.gum_units);
    a.gum_key = (unsigned long long*)(ws + L.gum_key);
    a.gum_cnt = (uint32_t*)(ws + L.gum_cnt);

    const size_t es = dtype == SV_BF16 ? 2 : 4;
    if (a.p_out && cudaMemsetAsync(a.p_out, 0, sizeof(float) * (size_t)B * (gamma_max + 1) * V, s) != cudaSuccess)
        return SV_ECUDA;
    if (a.q_out && cudaMemsetAsync(a.q_out, 0, sizeof(float) * (size_t)B * gamma_max * V, s) != cudaSuccess)
        return SV_ECUDA;
    // one CTA of min(1024, B rounded up to a warp) threads: a small batch pays
    // for no idle warps at the plan's block-wide scans
    const int plan_threads = B >= kPlanThreads ? kPlanThreads : (B + 31) / 32 * 32;
    plan_kernel<<<1, plan_threads, 0, s>>>(a);
    if (cudaGetLastError() != cudaSuccess) return SV_ECUDA;

    const bool vector = ((size_t)V * es) % 16 == 0;
    const cudaError_t e = launch_all(dtype, vector, a, di.sms, s, opt);
    return e == cudaSuccess ? SV_OK : SV_ECUDA;
}
}  // namespace

extern "C" int spec_verify_ex(const void* target_logits, const void* draft_logits, int dtype,
                              const int32_t* draft_tokens, const int32_t* num_draft, const float* temperature,
                              const int32_t* top_k, const float* top_p, uint64_t seed, int B, int gamma_max, int V,
                              int32_t* accepted_len, int32_t* out_tokens, float* alpha, float* p_out, float* q_out,
                              uint32_t* row_status, void* workspace, size_t workspace_bytes, void* stream,
                              const sv_options* options) {
    return verify_call(target_logits, draft_logits, dtype, draft_tokens, num_draft, temperature, top_k, top_p, seed,
                       B, gamma_max, V, accepted_len, out_tokens, alpha, p_out, q_out, row_status, workspace,
                       workspace_bytes, stream, options, false);
}

extern "C" size_t spec_verify_kseq_workspace_size(int B, int K, int V, int dtype) {
    if (check_shape(B, 1, V, dtype) != SV_OK || K < 1 || K > SV_MAX_KSEQ) return 0;
    return ws_layout(B, 1, V, dtype).total;
}

extern "C" int spec_verify_kseq(const void* target_logits, const void* draft_logits, int dtype,
                                const int32_t* candidates, const int32_t* num_candidates, const float* temperature,
                                const int32_t* top_k, const float* top_p, uint64_t seed, int B, int K, int V,
                                int32_t* out_token, int32_t* accepted, uint32_t* row_status, void* workspace,
                                size_t workspace_bytes, void* stream, const sv_options* options) {
    if (K < 1) return SV_EINVAL;
    if (K > SV_MAX_KSEQ) return SV_ETOO_LARGE;
    float dummy_alpha = 0.0f;  // satisfies the sampling rule's argument check; K-SEQ writes no alpha
    sv_options opt;
    memset(&opt, 0, sizeof opt);
    if (options) {
        if (options->struct_size < sizeof(uint32_t)) return SV_EINVAL;
        memcpy(&opt, options, options->struct_size < sizeof opt ? options->struct_size : sizeof opt);
    }
    opt.struct_size = sizeof opt;  // path is the caller's: SV_PATH_DENSE sends every row to the cluster kernel
    opt.pos_accept = nullptr;
    opt.pos_token = nullptr;
    opt.lenience = nullptr;
    return verify_call(target_logits, draft_logits, dtype, candidates, num_candidates, temperature, top_k, top_p, seed,
                       B, K, V, accepted, out_token, &dummy_alpha, nullptr, nullptr, row_status, workspace,
                       workspace_bytes, stream, &opt, false, true);
}

extern "C" int spec_verify_gumbel(const void* target_logits, int dtype, const int32_t* draft_tokens,
                                  const int32_t* num_draft, const float* temperature, const int32_t* top_k,
                                  const float* top_p, uint64_t seed, int B, int gamma_max, int V,
                                  int32_t* accepted_len, int32_t* out_tokens, int32_t* target_tokens,
                                  uint32_t* row_status, void* workspace, size_t workspace_bytes, void* stream,
                                  const sv_options* options) {
    sv_options opt;
    memset(&opt, 0, sizeof opt);
    if (options) {
        if (options->struct_size < sizeof(uint32_t)) return SV_EINVAL;
        memcpy(&opt, options, options->struct_size < sizeof opt ? options->struct_size : sizeof opt);
    }
    opt.struct_size = sizeof opt;
    if (target_tokens) opt.pos_token = target_tokens;
    return verify_call(target_logits, nullptr, dtype, draft_tokens, num_draft, temperature, top_k, top_p, seed, B,
                       gamma_max, V, accepted_len, out_tokens, nullptr, nullptr, nullptr, row_status, workspace,
                       workspace_bytes, stream, &opt, true);
}

extern "C" int spec_verify(const void* target_logits, const void* draft_logits, int dtype, const int32_t* draft_tokens,
                           const int32_t* num_draft, const float* temperature, const int32_t* top_k,
                           const float* top_p, uint64_t seed, int B, int gamma_max, int V, int32_t* accepted_len,
                           int32_t* out_tokens, float* alpha, float* p_out, float* q_out, uint32_t* row_status,
                           void* workspace, size_t workspace_bytes, void* stream) {
    return spec_verify_ex(target_logits, draft_logits, dtype, draft_tokens, num_draft, temperature, top_k, top_p,
                          seed, B, gamma_max, V, accepted_len, out_tokens, alpha, p_out, q_out, row_status,
                          workspace, workspace_bytes, stream, nullptr);
}

// ---------------------------------------------------------------------------
// host-buffer form
// ---------------------------------------------------------------------------
namespace {
struct HostLayout {
    size_t target, draft, tokens, num_draft, temp, top_k, top_p, acc, out, alpha, ws, total;
};
HostLayout host_layout(int B, int G, int V, int dtype, int has_nd, int has_k, int has_p) {
    HostLayout h{};
    const size_t es = dtype == SV_BF16 ? 2 : 4;
    size_t o = 0;
    h.target = o;    o = align_up(o + es * (size_t)B * (G + 1) * V, 256);
    h.draft = o;     o = align_up(o + es * (size_t)B * G * V, 256);
    h.tokens = o;    o = align_up(o + 4 * (size_t)B * G, 256);
    h.num_draft = o; o = align_up(o + (has_nd ? 4 * (size_t)B : 0), 256);
    h.temp = o;      o = align_up(o + 4 * (size_t)B, 256);
    h.top_k = o;     o = align_up(o + (has_k ? 4 * (size_t)B : 0), 256);
    h.top_p = o;     o = align_up(o + (has_p ? 4 * (size_t)B : 0), 256);
    h.acc = o;       o = align_up(o + 4 * (size_t)B, 256);
    h.out = o;       o = align_up(o + 4 * (size_t)B * (G + 1), 256);
    h.alpha = o;     o = align_up(o + 4 * (size_t)B * G, 256);
    h.ws = o;        o = align_up(o + ws_layout(B, G, V, dtype).total, 256);
    h.total = o;
    return h;
}
}  // namespace

extern "C" size_t spec_verify_host_staging_size(int B, int gamma_max, int V, int dtype, int has_num_draft,
                                                int has_top_k, int has_top_p) {
    if (check_shape(B, gamma_max, V, dtype) != SV_OK) return 0;
    return host_layout(B, gamma_max, V, dtype, has_num_draft, has_top_k, has_top_p).total;
}

extern "C" int spec_verify_host(const void* host_target_logits, const void* host_draft_logits, int dtype,
                                const int32_t* host_draft_tokens, const int32_t* host_num_draft,
                                const float* host_temperature, const int32_t* host_top_k, const float* host_top_p,
                                uint64_t seed, int B, int gamma_max, int V, int32_t* host_accepted_len,
                                int32_t* host_out_tokens, float* host_alpha, void* device_staging,
                                size_t staging_bytes, void* stream) {
    const int rc = check_shape(B, gamma_max, V, dtype);
    if (rc != SV_OK) return rc;
    if (B == 0) return SV_OK;
    if (!host_target_logits || !host_draft_logits || !host_draft_tokens || !host_temperature || !host_accepted_len ||
        !host_out_tokens || !host_alpha)
        return SV_EINVAL;
    const HostLayout h = host_layout(B, gamma_max, V, dtype, host_num_draft != nullptr, host_top_k != nullptr,
                                     host_top_p != nullptr);
    if (!device_staging || staging_bytes < h.total) return SV_EWORKSPACE;
    if ((uintptr_t)device_staging & 255u) return SV_EINVAL;
    cudaStream_t s = (cudaStream_t)stream;
    char* d = (char*)device_staging;
    const size_t es = dtype == SV_BF16 ? 2 : 4;
    const size_t G = (size_t)gamma_max;
    bool ok = true;
    auto h2d = [&](size_t off, const void* src, size_t bytes) {
        if (src && bytes) ok = ok && cudaMemcpyAsync(d + off, src, bytes, cudaMemcpyHostToDevice, s) == cudaSuccess;
    };
    h2d(h.target, host_target_logits, es * B * (G + 1) * V);
    h2d(h.draft, host_draft_logits, es * B * G * V);
    h2d(h.tokens, host_draft_tokens, 4 * B * G);
    h2d(h.num_draft, host_num_draft, 4 * (size_t)B);
    h2d(h.temp, host_temperature, 4 * (size_t)B);
    h2d(h.top_k, host_top_k, 4 * (size_t)B);
    h2d(h.top_p, host_top_p, 4 * (size_t)B);
    if (!ok) return SV_ECUDA;
    const int r = spec_verify(d + h.target, d + h.draft, dtype, (const int32_t*)(d + h.tokens),
                              host_num_draft ? (const int32_t*)(d + h.num_draft) : nullptr,
                              (const float*)(d + h.temp), host_top_k ? (const int32_t*)(d + h.top_k) : nullptr,
                              host_top_p ? (const float*)(d + h.top_p) : nullptr, seed, B, gamma_max, V,
                              (int32_t*)(d + h.acc), (int32_t*)(d + h.out), (float*)(d + h.alpha), nullptr, nullptr,
                              nullptr, d + h.ws, h.total - h.ws, stream);
    if (r != SV_OK) return r;
    ok = cudaMemcpyAsync(host_accepted_len, d + h.acc, 4 * (size_t)B, cudaMemcpyDeviceToHost, s) == cudaSuccess &&
         cudaMemcpyAsync(host_out_tokens, d + h.out, 4 * B * (G + 1), cudaMemcpyDeviceToHost, s) == cudaSuccess &&
         cudaMemcpyAsync(host_alpha, d + h.alpha, 4 * B * G, cudaMemcpyDeviceToHost, s) == cudaSuccess &&
         cudaStreamSynchronize(s) == cudaSuccess;
    return ok ? SV_OK : SV_ECUDA;
}
