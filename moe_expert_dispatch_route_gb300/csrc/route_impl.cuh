// Device code of the gates shared by the route kernels (route.cu) and the fused
// low-latency head (head.cu): one warp routes one token.
#pragma once

#include <float.h>
#include <limits.h>

#include "common.cuh"

namespace moe {

// The grouped gate's sigma is SPECIFIED operation by operation so that expert
// selection is reproducible everywhere: e^x by Cody and Waite's reduction
// x = n ln2 + r with ln 2 split in a 24-bit-exact high part and a low part, then the
// degree-7 Taylor polynomial of e^r in Horner form with fused multiply-adds, then an
// exact scaling by 2^n; sigma(x) = 1 / (1 + e^-x) on x clamped to [-80, 80].  Every
// step is an explicit round-to-nearest binary32 operation (no contraction).
__device__ __forceinline__ float spec_exp(float x) {
    const float kLog2e = 0x1.715476p+0f;
    const float kLn2Hi = 0x1.62e400p-1f;
    const float kLn2Lo = 0x1.7f7d1cp-20f;
    float n = rintf(__fmul_rn(x, kLog2e));
    float r = __fmaf_rn(-n, kLn2Hi, x);
    r = __fmaf_rn(-n, kLn2Lo, r);
    float p = 0x1.a01a02p-13f;           // 1/5040
    p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);  // 1/720
    p = __fmaf_rn(p, r, 0x1.111112p-7f);   // 1/120
    p = __fmaf_rn(p, r, 0x1.555556p-5f);   // 1/24
    p = __fmaf_rn(p, r, 0x1.555556p-3f);   // 1/6
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    float two_n = __int_as_float(((int)n + 127) << 23);
    return __fmul_rn(p, two_n);
}

__device__ __forceinline__ float spec_sigmoid(float x) {
    float c = x < -80.0f ? -80.0f : (x > 80.0f ? 80.0f : x);
    return __fdiv_rn(1.0f, __fadd_rn(1.0f, spec_exp(-c)));
}

// The DeepSeek-V4-shaped gate's score s(x) = sqrt(softplus(x)) is SPECIFIED the same
// way: softplus(x) = max(x, 0) + log1p(e^-|x|) on x clamped to [-80, 80], e^x as above,
// log1p(y) (y in [0, 1]) as the series 2 atanh(z) = 2 (z + z^3/3 + ... + z^15/15) of
// z = y / (2 + y), Horner in z^2 with fused multiply-adds, each coefficient 1/n
// rounded to binary32; then the correctly rounded square root.
__device__ __forceinline__ float spec_log1p(float y) {
    const float z = __fdiv_rn(y, __fadd_rn(2.0f, y));
    const float z2 = __fmul_rn(z, z);
    float p = 0x1.111112p-4f;             // 1/15
    p = __fmaf_rn(p, z2, 0x1.3b13b2p-4f);  // 1/13
    p = __fmaf_rn(p, z2, 0x1.745d18p-4f);  // 1/11
    p = __fmaf_rn(p, z2, 0x1.c71c72p-4f);  // 1/9
    p = __fmaf_rn(p, z2, 0x1.24924ap-3f);  // 1/7
    p = __fmaf_rn(p, z2, 0x1.99999ap-3f);  // 1/5
    p = __fmaf_rn(p, z2, 0x1.555556p-2f);  // 1/3
    p = __fmaf_rn(p, z2, 1.0f);
    return __fmul_rn(__fmul_rn(2.0f, z), p);
}

__device__ __forceinline__ float spec_sqrt_softplus(float x) {
    const float c = x < -80.0f ? -80.0f : (x > 80.0f ? 80.0f : x);
    const float e = spec_exp(-fabsf(c));
    return __fsqrt_rn(__fadd_rn(fmaxf(c, 0.0f), spec_log1p(e)));
}

// sqrt(softplus(x)) for the weights (ordinary math, compared with a tolerance).
__device__ __forceinline__ float sqrt_softplus(float x) {
    return sqrtf(x > 30.0f ? x + log1pf(expf(-x)) : log1pf(expf(x)));
}

// A NaN score takes part in the selection as -inf: every comparison with NaN is false,
// so without this a row of NaNs would select no expert at all.  Finite scores, the
// only ones the gates are defined for, are unchanged.
__device__ __forceinline__ float nan_to_neg_inf(float v) { return v != v ? -INFINITY : v; }

// Warp arg-max: larger value wins, equal values -> smaller id.
__device__ __forceinline__ void warp_argmax(float& v, int& id) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        float ov = __shfl_xor_sync(0xffffffffu, v, o);
        int oi = __shfl_xor_sync(0xffffffffu, id, o);
        if (ov > v || (ov == v && oi < id)) {
            v = ov;
            id = oi;
        }
    }
}

// One warp: token t of the softmax gate.  Lane j < k returns the j-th choice
// (descending logit, equal logits -> lower id) and its weight.
template <int NPER>
__device__ __forceinline__ void route_token_softmax(int t, int E, int k, int renorm, const float* __restrict__ logits,
                                                    int& out_id, float& out_w) {
    const int lane = threadIdx.x & 31;
    const float* l = logits + (size_t)t * E;
    float v[NPER];
    uint32_t taken = 0;
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < NPER; ++i) {
        int e = lane + 32 * i;
        v[i] = e < E ? nan_to_neg_inf(__ldg(l + e)) : -INFINITY;
        if (e >= E) taken |= 1u << i;
        else m = fmaxf(m, v[i]);
    }
    m = warp_max(m);
    int my_id = 0;
    float my_v = -INFINITY;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = INT_MAX;
#pragma unroll
        for (int i = 0; i < NPER; ++i) {
            int e = lane + 32 * i;
            if (!((taken >> i) & 1u) && (v[i] > bv || (v[i] == bv && e < bi))) {
                bv = v[i];
                bi = e;
            }
        }
        warp_argmax(bv, bi);
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (lane == j) {
            my_id = bi;
            my_v = bv;
        }
    }
    float my_p = lane < k ? expf(my_v - m) : 0.0f;
    float z;
    if (renorm) {
        z = warp_sum(my_p);
    } else {
        float part = 0.0f;
#pragma unroll
        for (int i = 0; i < NPER; ++i)
            if (lane + 32 * i < E) part += expf(v[i] - m);
        z = warp_sum(part);
    }
    out_id = my_id;
    out_w = my_p / z;
}

// One warp: token t of the group-limited gate with the score sigma (kSqrtSoftplus =
// false, the DeepSeek-V3 shape) or sqrt(softplus) (true, the DeepSeek-V4 shape).  cs:
// this warp's E floats of shared memory.  Lane j < k returns the j-th choice and its
// weight.
template <int NPER, bool kSqrtSoftplus = false>
__device__ __forceinline__ void route_token_grouped(int t, int E, int k, int n_group, int topk_group, int renorm,
                                                    float scale, const float* __restrict__ logits,
                                                    const float* __restrict__ bias, float* cs, int& out_id,
                                                    float& out_w) {
    const int lane = threadIdx.x & 31;
    const int gsz = E / n_group;
    const float* l = logits + (size_t)t * E;
    float c[NPER];
#pragma unroll
    for (int i = 0; i < NPER; ++i) {
        int e = lane + 32 * i;
        if (e < E) {
            const float x = __ldg(l + e);
            const float s = kSqrtSoftplus ? spec_sqrt_softplus(x) : spec_sigmoid(x);
            c[i] = nan_to_neg_inf(__fadd_rn(s, bias ? __ldg(bias + e) : 0.0f));
            cs[e] = c[i];
        } else {
            c[i] = -INFINITY;
        }
    }
    __syncwarp();
    // group scores: lane g scans its group's choice scores for the two best
    float gs = -INFINITY;
    int gid = INT_MAX;
    if (lane < n_group) {
        float m1 = -INFINITY, m2 = -INFINITY;
        for (int i = 0; i < gsz; ++i) {
            float v = cs[lane * gsz + i];
            if (v > m1) {
                m2 = m1;
                m1 = v;
            } else if (v > m2) {
                m2 = v;
            }
        }
        gs = gsz >= 2 ? __fadd_rn(m1, m2) : m1;
        gid = lane;
    }
    uint32_t gsel = 0;
    for (int j = 0; j < topk_group; ++j) {
        float bv = gs;
        int bi = gid;
        warp_argmax(bv, bi);
        gsel |= 1u << bi;
        if (bi == lane) {
            gs = -INFINITY;
            gid = INT_MAX;
        }
    }
    uint32_t taken = 0;
#pragma unroll
    for (int i = 0; i < NPER; ++i) {
        int e = lane + 32 * i;
        if (e >= E || !((gsel >> (e / gsz)) & 1u)) taken |= 1u << i;
    }
    int my_id = 0;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = INT_MAX;
#pragma unroll
        for (int i = 0; i < NPER; ++i) {
            int e = lane + 32 * i;
            if (!((taken >> i) & 1u) && (c[i] > bv || (c[i] == bv && e < bi))) {
                bv = c[i];
                bi = e;
            }
        }
        warp_argmax(bv, bi);
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (lane == j) my_id = bi;
    }
    float sj = 0.0f;
    if (lane < k) {
        const float x = __ldg(l + (my_id < E ? my_id : 0));
        sj = kSqrtSoftplus ? sqrt_softplus(x) : 1.0f / (1.0f + expf(-x));
    }
    float sum = warp_sum(sj);
    out_id = my_id;
    out_w = (renorm ? sj / sum : sj) * scale;
    __syncwarp();  // cs is reused by this warp's next token
}

}  // namespace moe
