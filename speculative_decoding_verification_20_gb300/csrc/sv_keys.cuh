// sv_keys.cuh -- logit keys shared by the streaming top-k kernel and the
// combine kernel: order-preserving element keys, the (key, token id)
// composite, NaN-propagating maxima and the packed threshold test.
#pragma once

#include "sv_finalize.cuh"

namespace sv {

// ---------------------------------------------------------------------------
// keys and composites
// ---------------------------------------------------------------------------
template <typename TIn>
struct Elem;
template <>
struct Elem<__nv_bfloat16> {
    static constexpr int VEC = 8, KB = 16;
    __device__ static uint32_t bits(const uint4& v, int j) {
        const uint32_t w = j < 2 ? v.x : j < 4 ? v.y : j < 6 ? v.z : v.w;
        return (j & 1) ? (w >> 16) : (w & 0xFFFFu);
    }
    __device__ static uint32_t key(uint32_t b) { return okey16(b); }
    __device__ static float value(uint32_t b) { return __uint_as_float(b << 16); }
    __device__ static double key_value(uint32_t k) { return (double)key_value16(k); }
    __device__ static bool bad(uint32_t b) { return bad16(b); }
    // bit pattern of a float that holds a bf16 value exactly
    __device__ static uint32_t bits_of(float f) { return __float_as_uint(f) >> 16; }
    __device__ static uint32_t load_bits(const __nv_bfloat16* p, int i) {
        return reinterpret_cast<const unsigned short*>(p)[i];
    }
    static constexpr uint32_t kNegInfBits = 0xFF80u;
};
template <>
struct Elem<float> {
    static constexpr int VEC = 4, KB = 32;
    __device__ static uint32_t bits(const uint4& v, int j) { return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w; }
    __device__ static uint32_t key(uint32_t b) { return okey32(b); }
    __device__ static float value(uint32_t b) { return __uint_as_float(b); }
    __device__ static double key_value(uint32_t k) { return (double)key_value32(k); }
    __device__ static bool bad(uint32_t b) { return bad32(b); }
    __device__ static uint32_t bits_of(float f) { return __float_as_uint(f); }
    __device__ static uint32_t load_bits(const float* p, int i) { return reinterpret_cast<const uint32_t*>(p)[i]; }
    static constexpr uint32_t kNegInfBits = 0xFF800000u;
};

// composite sort key: logit key descending, then token id ascending
__device__ __forceinline__ unsigned long long composite(uint32_t key, uint32_t id) {
    return ((unsigned long long)key << 32) | (unsigned long long)(~id);
}
__device__ __forceinline__ uint32_t comp_key(unsigned long long c) { return (uint32_t)(c >> 32); }
__device__ __forceinline__ int comp_id(unsigned long long c) { return (int)(~(uint32_t)c); }

__device__ __forceinline__ int next_pow2(int n) {
    int p = 1;
    while (p < n) p <<= 1;
    return p;
}

// NaN-propagating max of the 16-byte vector (as float), used both as the
// fast-path filter and for non-finite detection
__device__ __forceinline__ float vmax_nan(const uint4& v, __nv_bfloat16*) {
    __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&v.x);
    __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&v.y);
    __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&v.z);
    __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&v.w);
    const __nv_bfloat162 m = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
    return __bfloat162float(__hmax_nan(__low2bfloat16(m), __high2bfloat16(m)));
}
__device__ __forceinline__ float fmax_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float vmax_nan(const uint4& v, float*) {
    return fmax_nan(fmax_nan(__uint_as_float(v.x), __uint_as_float(v.y)),
                    fmax_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
}

// Fast-path test of one full 16-byte vector: updates the running NaN-propagating
// maximum and says whether any element may pass the threshold.
struct RunBf16 {
    __nv_bfloat162 run, th2;
};
__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t w) { return *reinterpret_cast<__nv_bfloat162*>(&w); }
__device__ __forceinline__ bool vec_test(const uint4& v, RunBf16& r, bool strict) {
    const __nv_bfloat162 m = __hmax2_nan(__hmax2_nan(as_bf2(v.x), as_bf2(v.y)), __hmax2_nan(as_bf2(v.z), as_bf2(v.w)));
    r.run = __hmax2_nan(r.run, m);
    return (strict ? __hgt2_mask(m, r.th2) : __hge2_mask(m, r.th2)) != 0u;
}
__device__ __forceinline__ void run_init(RunBf16& r, float thv) {
    r.run = __float2bfloat162_rn(-INFINITY);
    r.th2 = __float2bfloat162_rn(thv);
}
__device__ __forceinline__ float run_value(const RunBf16& r) {
    return __bfloat162float(__hmax_nan(__low2bfloat16(r.run), __high2bfloat16(r.run)));
}
struct RunF32 {
    float run, th;
};
__device__ __forceinline__ bool vec_test(const uint4& v, RunF32& r, bool strict) {
    const float m = fmax_nan(fmax_nan(__uint_as_float(v.x), __uint_as_float(v.y)),
                             fmax_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
    r.run = fmax_nan(r.run, m);
    return strict ? (m > r.th) : (m >= r.th);
}
__device__ __forceinline__ void run_init(RunF32& r, float thv) {
    r.run = -INFINITY;
    r.th = thv;
}
__device__ __forceinline__ float run_value(const RunF32& r) { return r.run; }
template <typename TIn>
struct RunOf {
    using type = RunF32;
};
template <>
struct RunOf<__nv_bfloat16> {
    using type = RunBf16;
};

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

}  // namespace sv
