// sv_warp_sort.cuh -- bitonic sort of up to 256 64-bit keys held in the
// registers of one warp (shared by the combine kernel and the whole-row kernel).
#pragma once

#include <cstdint>

namespace sv {

// Bitonic sort across the warp of 32 * P 64-bit keys held P per lane (element
// m * 32 + lane in x[m]), descending or ascending.
template <int P>
__device__ __forceinline__ void warp_bitonic(unsigned long long (&x)[P], int lane, bool descending) {
    constexpr int N = 32 * P;
#pragma unroll
    for (int k2 = 2; k2 <= N; k2 <<= 1) {
#pragma unroll
        for (int j = k2 >> 1; j > 0; j >>= 1) {
            if (j >= 32) {  // partners in the same lane
#pragma unroll
                for (int m = 0; m < P; ++m) {
                    const int mp = m ^ (j >> 5);
                    if (mp > m) {
                        const bool lower_max = (((m * 32 + lane) & k2) == 0) == descending;
                        const unsigned long long lo = x[m], hi = x[mp];
                        const bool sw = lower_max ? (lo < hi) : (lo > hi);
                        x[m] = sw ? hi : lo;
                        x[mp] = sw ? lo : hi;
                    }
                }
            } else {  // partners in lane ^ j
#pragma unroll
                for (int m = 0; m < P; ++m) {
                    const unsigned long long y = __shfl_xor_sync(0xFFFFFFFFu, x[m], j);
                    const bool lower = (lane & j) == 0;
                    const bool lower_max = (((m * 32 + lane) & k2) == 0) == descending;
                    const bool take_max = lower == lower_max;
                    x[m] = take_max ? (x[m] > y ? x[m] : y) : (x[m] < y ? x[m] : y);
                }
            }
        }
    }
}

// Sort n <= 32 * P entries of src (pad: `pad`) into dst across the warp.
template <int P>
__device__ __forceinline__ void warp_sort_into(const unsigned long long* src, int n, unsigned long long* dst,
                                               bool descending, unsigned long long pad, int lane) {
    unsigned long long x[P];
#pragma unroll
    for (int m = 0; m < P; ++m) x[m] = m * 32 + lane < n ? src[m * 32 + lane] : pad;
    warp_bitonic<P>(x, lane, descending);
    __syncwarp();
#pragma unroll
    for (int m = 0; m < P; ++m)
        if (m * 32 + lane < n) dst[m * 32 + lane] = x[m];
    __syncwarp();
}
__device__ __forceinline__ void warp_sort(const unsigned long long* src, int n, unsigned long long* dst,
                                          bool descending, unsigned long long pad, int lane) {
    if (n <= 32)
        warp_sort_into<1>(src, n, dst, descending, pad, lane);
    else if (n <= 64)
        warp_sort_into<2>(src, n, dst, descending, pad, lane);
    else if (n <= 128)
        warp_sort_into<4>(src, n, dst, descending, pad, lane);
    else
        warp_sort_into<8>(src, n, dst, descending, pad, lane);
}

}  // namespace sv
