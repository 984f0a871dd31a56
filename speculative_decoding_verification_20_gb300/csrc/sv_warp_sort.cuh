// sv_warp_sort.cuh -- bitonic sort of up to 256 64-bit keys held in the
// registers of one warp (shared by the combine kernel and the whole-row kernel).
#pragma once

#include <cstdint>

namespace sv {

// One compare-exchange of a bitonic stage between x[m] and its partner value
// y: keep the larger value where this position's block sorts descending and
// this position is the lower one of the pair (or ascending and upper).
__device__ __forceinline__ unsigned long long bitonic_keep(unsigned long long v, unsigned long long y, bool take_max) {
    return take_max ? (v > y ? v : y) : (v < y ? v : y);
}

// One stage (k2, j) of the bitonic network over 32 * P 64-bit keys held P per
// lane (element m * 32 + lane in x[m]): partners at distance j < 32 are in
// lane ^ j (a shuffle), partners at j >= 32 are in the same lane, at register
// m ^ (j / 32).
template <int P>
__device__ __forceinline__ void bitonic_stage(unsigned long long (&x)[P], int lane, bool descending, int k2, int j) {
    if (j < 32) {
        const bool lower = (lane & j) == 0;
#pragma unroll
        for (int m = 0; m < P; ++m) {
            const unsigned long long y = __shfl_xor_sync(0xFFFFFFFFu, x[m], j);
            const bool lower_max = (((m * 32 + lane) & k2) == 0) == descending;
            x[m] = bitonic_keep(x[m], y, lower == lower_max);
        }
    } else {
        // in-lane partners m and m ^ s, s = j / 32 in {1, 2, 4, ...} < P
#pragma unroll
        for (int s = 1; s < P; s <<= 1) {
            if ((j >> 5) != s) continue;
#pragma unroll
            for (int m = 0; m < P; ++m) {
                const int mp = m ^ s;
                if (mp > m) {
                    const bool lower_max = (((m * 32 + lane) & k2) == 0) == descending;
                    const unsigned long long lo = x[m], hi = x[mp];
                    const bool sw = lower_max ? (lo < hi) : (lo > hi);
                    x[m] = sw ? hi : lo;
                    x[mp] = sw ? lo : hi;
                }
            }
        }
    }
}

// Bitonic sort across the warp of 32 * P 64-bit keys held P per lane,
// descending or ascending.  Up to 64 keys the network is unrolled (21 stages at
// most: every stage's partners and directions are constants); beyond, the
// merge stages run as loops so one copy of the code serves each size.
template <int P>
__device__ __forceinline__ void warp_bitonic(unsigned long long (&x)[P], int lane, bool descending) {
    constexpr int N = 32 * P;
    if constexpr (P <= 2) {
#pragma unroll
        for (int k2 = 2; k2 <= N; k2 <<= 1)
#pragma unroll
            for (int j = k2 >> 1; j > 0; j >>= 1) bitonic_stage<P>(x, lane, descending, k2, j);
    } else {
#pragma unroll 1
        for (int k2 = 2; k2 <= N; k2 <<= 1)
#pragma unroll 1
            for (int j = k2 >> 1; j > 0; j >>= 1) bitonic_stage<P>(x, lane, descending, k2, j);
    }
}

// Sort n <= 32 * P entries of src (pad: `pad`) into dst across the warp.  Kept
// out of line: one copy per size serves every caller.
template <int P>
__device__ __noinline__ void warp_sort_into(const unsigned long long* src, int n, unsigned long long* dst,
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
