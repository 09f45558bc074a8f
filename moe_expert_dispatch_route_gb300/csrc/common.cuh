// Device-side helpers shared by the kernels of libmoe_gb300.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

constexpr int kQG = 128;            // FP8 quantisation group / block edge
constexpr int kMaxExperts = 512;    // E + S
constexpr int kMaxSlotsPerToken = 32;  // k + S

// Stores `code` into the caller's device error flag unless an earlier error is there.
__device__ __forceinline__ void set_err(int32_t* flag, int32_t code) {
    if (flag) atomicCAS(reinterpret_cast<int*>(flag), 0, code);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Exponent s of the power-of-two FP8 scale 2^s: the smallest integer with
// amax <= 448 * 2^s (448 = 0.875 * 2^9); amax == 0 gives 0.
__device__ __forceinline__ int fp8_scale_exp(float amax) {
    if (!(amax > 0.0f)) return 0;
    const uint32_t b = __float_as_uint(amax);
    const int ef = (int)(b >> 23);  // amax > 0: the sign bit is clear
    if (ef == 0 || ef == 255) {     // subnormal or infinite: the library's decomposition
        int e;
        const float f = frexpf(amax, &e);
        return (f <= 0.875f) ? e - 9 : e - 8;
    }
    // amax = (1 + m / 2^23) * 2^(ef - 127) and 448 = 1.75 * 2^8: s = ef - 135 when the
    // significand is at most 1.75 (m <= 0.75 * 2^23), else one more
    return ((b & 0x7fffffu) <= 0x600000u) ? ef - 135 : ef - 134;
}

// x * 2^n rounded once to nearest even, the value scalbnf(x, n) gives: the product of x
// and an exact power of two is the correctly rounded value of the same real number.  For
// n above the normal exponent range, two steps that both scale up (exact unless they
// overflow, which the one-step result would too); below it, scalbnf itself (two steps
// down could round twice).
__device__ __forceinline__ float mul_pow2(float x, int n) {
    if (n >= -126 && n <= 127) return x * __int_as_float((n + 127) << 23);
    if (n > 127 && n <= 254) return (x * 0x1p127f) * __int_as_float(n << 23);
    return scalbnf(x, n);
}

// 2^-s as two exact factors (m1, m2) for s in [-254, 126]: (x * m1) * m2 equals
// mul_pow2(x, -s) -- with 2^-s a normal float, m2 = 1 and the one product is the single
// rounding; above the normal range, m1 = 2^127 and both products scale up exactly.  An
// FP8 group scale exponent is always in range (at most 119 for a finite amax, at least
// -157 for a nonzero one).
struct Pow2Factors {
    float m1, m2;
};
__device__ __forceinline__ Pow2Factors pow2_neg(int s) {
    const int n = -s;
    const int n1 = n > 127 ? 127 : n;
    return {__uint_as_float((uint32_t)(n1 + 127) << 23), __uint_as_float((uint32_t)(n - n1 + 127) << 23)};
}
__device__ __forceinline__ float scale_by(float x, const Pow2Factors& f) { return (x * f.m1) * f.m2; }

// SwiGLU of the tensor-core FFNs: silu(g) * u = g / (1 + e^-g) * u with the fast
// exponential and division intrinsics (a few ulp of relative error, far below the bf16 /
// e4m3 rounding of h that follows).  The limits stay exact: for very negative g the
// divisor overflows to infinity and the quotient is 0; for very positive g it is g.
__device__ __forceinline__ float silu_mul_fast(float g, float u) { return __fdividef(g, 1.0f + __expf(-g)) * u; }

// Two floats -> two e4m3 codes (round to nearest even, saturating to +-448).
__device__ __forceinline__ uint16_t f2_to_e4m3x2(float a, float b) {
    return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ float e4m3_to_f(uint8_t c) {
    __half_raw hr = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)c, __NV_E4M3);
    return __half2float(__half(hr));
}

__device__ __forceinline__ float bf16_bits_to_f(uint16_t b) {
    return __uint_as_float(((uint32_t)b) << 16);
}

__device__ __forceinline__ uint16_t f_to_bf16_bits(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    return (uint32_t)f_to_bf16_bits(lo) | ((uint32_t)f_to_bf16_bits(hi) << 16);
}

// Programmatic dependent launch: let the next kernel on the stream be scheduled now,
// and wait until the previous kernel's writes are complete and visible.  Both are
// no-ops for a kernel launched without the programmatic-serialisation attribute.
__device__ __forceinline__ void pdl_begin() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

}  // namespace moe
