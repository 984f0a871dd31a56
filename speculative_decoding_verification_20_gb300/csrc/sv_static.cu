// sv_static.cu -- spec_verify_static: the verification step with its scratch
// in a fixed device buffer that this library owns, so the call allocates
// nothing and needs no workspace from the caller.
//
// Who needs it: callers with no memory manager of their own (a plain C or C++
// serving loop that embeds the sampler and has no caching allocator), and
// decode loops that must not call cudaMalloc / cudaFree between steps --
// cudaFree waits for the whole device and cudaMalloc may, which stalls every
// other stream on the GPU.  Such a caller would otherwise have to keep a
// workspace alive itself; here the library keeps one, of a fixed size.
//
// The buffer is one file-scope __device__ array of SV_STATIC_SCRATCH_BYTES.
// Each device gets its own copy when this library's code is loaded into that
// device's context.  Its device address is looked up with
// cudaGetSymbolAddress by the first spec_verify_static call made with that
// device current, and kept for that context: the cache is keyed on the
// device and on the context's unique id, so after cudaDeviceReset (which
// destroys the context; the next CUDA call makes a new one and loads the
// module again, possibly elsewhere) the next call looks the address up again
// instead of handing the kernels a stale pointer.  Make the first call on a
// device (and the first after a reset) outside any stream capture.  Every
// call reuses the same buffer, so calls that could run at the same time on
// one device (different streams with nothing ordering them) race on it and
// give wrong results: order them on one stream or with events.
//
// Nothing in the buffer has to start at zero: the first kernel of each call
// resets every counter and flag the later kernels of that call read.
#include <cuda_runtime.h>

#include <mutex>

#include "spec_verify.h"

namespace {

static_assert(SV_STATIC_SCRATCH_BYTES % 256 == 0, "the scratch size keeps 256-byte alignment");

static __device__ __align__(256) unsigned char g_static_scratch[SV_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// The driver's context queries, fetched through the runtime so the library
// needs no link-time dependency on the driver library.
typedef int (*CtxGetCurrentFn)(void** ctx);
typedef int (*CtxGetIdFn)(void* ctx, unsigned long long* id);

// Unique id of the calling thread's current context (0: none, or the query
// is unavailable).  Context ids are never reused within a process.
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = (CtxGetCurrentFn)f;
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = (CtxGetIdFn)f;
        (void)cudaGetLastError();
    });
    if (!get_current || !get_id) return 0;
    void* ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != 0 || !ctx || get_id(ctx, &id) != 0) return 0;
    return id;
}

// The buffer's device address on device `dev` in the current context, or
// nullptr if the lookup failed.
void* static_scratch(int dev) {
    static void* addr[kMaxDevices] = {};
    static unsigned long long ctx_of[kMaxDevices] = {};
    static std::mutex mu;
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long ctx = current_context_id();
    if (!addr[dev] || ctx == 0 || ctx != ctx_of[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) {
            (void)cudaGetLastError();  // do not leave the failure for the caller's next check
            addr[dev] = nullptr;
            return nullptr;
        }
        addr[dev] = p;
        // the lookup has made the primary context current if there was none
        ctx_of[dev] = ctx != 0 ? ctx : current_context_id();
    }
    return addr[dev];
}

}  // namespace

extern "C" int spec_verify_static(const void* target_logits, const void* draft_logits, int dtype,
                                  const int32_t* draft_tokens, const int32_t* num_draft, const float* temperature,
                                  const int32_t* top_k, const float* top_p, uint64_t seed, int B, int gamma_max,
                                  int V, int32_t* accepted_len, int32_t* out_tokens, float* alpha, float* p_out,
                                  float* q_out, uint32_t* row_status, void* stream) {
    // the shape checks of spec_verify come first (0 = an invalid shape)
    const size_t need = spec_verify_workspace_size(B, gamma_max, V, dtype);
    if (need == 0)
        return spec_verify(target_logits, draft_logits, dtype, draft_tokens, num_draft, temperature, top_k, top_p,
                           seed, B, gamma_max, V, accepted_len, out_tokens, alpha, p_out, q_out, row_status,
                           nullptr, 0, stream);
    if (need > (size_t)SV_STATIC_SCRATCH_BYTES) return SV_ESCRATCH;
    if (B == 0) return SV_OK;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SV_ECUDA;
    void* scratch = static_scratch(dev);
    if (!scratch) return SV_ECUDA;
    return spec_verify(target_logits, draft_logits, dtype, draft_tokens, num_draft, temperature, top_k, top_p, seed,
                       B, gamma_max, V, accepted_len, out_tokens, alpha, p_out, q_out, row_status, scratch,
                       (size_t)SV_STATIC_SCRATCH_BYTES, stream);
}
