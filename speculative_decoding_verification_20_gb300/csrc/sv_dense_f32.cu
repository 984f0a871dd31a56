// sv_dense_f32.cu -- dense-path kernels for float logits and their host launcher.
#include "sv_dense.cuh"

namespace sv {

namespace {
template <int R, bool VECTOR>
cudaError_t launch_r(const Args& a, int cs, int sms, cudaStream_t s) { return launch_dense_cluster<float, R, VECTOR>(a, cs, sms, s); }

template <bool VECTOR>
cudaError_t launch_v(const Args& a, int sms, cudaStream_t s) {
    int R = 0, cs = 0;
    const long long units = a.kseq ? (long long)a.B : (long long)a.B * (a.G + 1);
    if (!dense_shape<float>(a.V, units, sms, &R, &cs)) return cudaErrorInvalidValue;
    switch (R) {
        case 1: return launch_r<1, VECTOR>(a, cs, sms, s);
        case 2: return launch_r<2, VECTOR>(a, cs, sms, s);
        case 4: return launch_r<4, VECTOR>(a, cs, sms, s);
        case 8: return launch_r<8, VECTOR>(a, cs, sms, s);
        case 16: return launch_r<16, VECTOR>(a, cs, sms, s);
        default: return cudaErrorInvalidValue;
    }
}
}  // namespace

cudaError_t launch_dense_f32(bool vector, const Args& a, int sms, cudaStream_t s) {
    return vector ? launch_v<true>(a, sms, s) : launch_v<false>(a, sms, s);
}

}  // namespace sv
