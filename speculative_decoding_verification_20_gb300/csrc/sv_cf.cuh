// sv_cf.cuh -- compensated fp32 sums (a head and a running error term), used
// where a sum over many fp32 terms must stay close to the exact total without
// fp64 arithmetic (the fp64 pipe of this GPU is narrow).
#pragma once

#include "sv_internal.cuh"

namespace sv {

// compensated fp32 value s - c: sums of fp32 terms kept to about fp32
// rounding of the total, whatever the number of terms
struct CF {
    float s, c;
};
__device__ __forceinline__ CF cf_add(CF a, CF b) {  // exact two-sum of the heads
    const float t = a.s + b.s;
    const float bb = t - a.s;
    const float e = (a.s - (t - bb)) + (b.s - bb);
    return CF{t, (a.c + b.c) - e};
}
__device__ __forceinline__ float cf_val(CF a) { return a.s - a.c; }
__device__ __forceinline__ CF warp_cf_sum(CF a) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        a = cf_add(a, CF{__shfl_xor_sync(0xFFFFFFFFu, a.s, o), __shfl_xor_sync(0xFFFFFFFFu, a.c, o)});
    return a;
}
__device__ __forceinline__ CF warp_cf_scan(CF a, int lane) {  // inclusive, in lane order
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const CF y{__shfl_up_sync(0xFFFFFFFFu, a.s, o), __shfl_up_sync(0xFFFFFFFFu, a.c, o)};
        if (lane >= o) a = cf_add(y, a);
    }
    return a;
}

}  // namespace sv
