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

// x * a as a compensated pair (FMA two-product of the head)
__device__ __forceinline__ CF cf_scale(float x, CF a) {
    const float p = x * a.s;
    const float e = fmaf(x, a.s, -p);  // x * a.s = p + e exactly
    return CF{p, fmaf(x, a.c, -e)};
}
// a >= b, decided on the compensated difference
__device__ __forceinline__ bool cf_ge(CF a, CF b) {
    const CF d = cf_add(a, CF{-b.s, -b.c});
    return d.s - d.c >= 0.0f;
}
// 1 / a to about fp32 rounding: the rounded reciprocal of the head, then one
// Newton step on the exact residual 1 - r * a.s and the tail
__device__ __forceinline__ float cf_recip(CF a) {
    const float r = 1.0f / a.s;
    const float t = fmaf(-r, a.s, 1.0f) + r * a.c;
    return fmaf(r, t, r);
}

}  // namespace sv
