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
// Each device gets its own copy when this library's code is loaded there.
// Its device address is looked up once per device with cudaGetSymbolAddress,
// by the first spec_verify_static call made with that device current; make
// that first call outside any stream capture.  Every call reuses the same
// buffer, so calls that could run at the same time on one device (different
// streams with nothing ordering them) race on it and give wrong results:
// order them on one stream or with events.
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

// The buffer's device address on device `dev` (looked up once), or nullptr
// if the lookup failed.
void* static_scratch(int dev) {
    static void* addr[kMaxDevices] = {};
    static std::mutex mu;
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) {
            (void)cudaGetLastError();  // do not leave the failure for the caller's next check
            return nullptr;
        }
        addr[dev] = p;
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
