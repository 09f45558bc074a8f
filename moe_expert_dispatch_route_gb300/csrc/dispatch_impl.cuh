// Device code of dispatch shared by the dispatch kernels (dispatch.cu) and the fused
// plan + dispatch kernel (head.cu): one warp moves one (token, slice) work item.
#pragma once

#include "common.cuh"

namespace moe {

// fp32 / bf16 rows: slice of 128 16-byte vectors starting at v0, copied to the token's
// rows (my_slot: lane j < kk holds the row of entry j, -1 = not placed).
__device__ __forceinline__ void dispatch_copy_item(int kk, int nvec, const uint4* __restrict__ src, int v0,
                                                   int my_slot, uint4* __restrict__ xe, int lane) {
    uint4 val[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        int v = v0 + u * 32 + lane;
        if (v < nvec) val[u] = __ldg(src + v);
    }
    for (int j = 0; j < kk; ++j) {
        const int r = __shfl_sync(0xffffffffu, my_slot, j);
        if (r < 0) continue;
        uint4* dst = xe + (size_t)r * nvec;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            int v = v0 + u * 32 + lane;
            if (v < nvec) dst[v] = val[u];
        }
    }
}

// amax of the 8 bf16 values of a 16-byte vector, as fp32: |v| by clearing the sign
// bits, then max.bf16x2 (which, like fmaxf, returns the other operand when one is NaN;
// the max of magnitudes is exact, so the order does not matter).
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ float amax_bf16x8(const uint4& v) {
    const uint32_t m = bf16x2_max(bf16x2_max(v.x & 0x7fff7fffu, v.y & 0x7fff7fffu),
                                  bf16x2_max(v.z & 0x7fff7fffu, v.w & 0x7fff7fffu));
    return fmaxf(0.0f, fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xffff0000u)));
}

// Quantises and stores one (token, slice) item whose four 32-vector passes (8 bf16 per
// vector, vectors [vbeg, vend), whole 1x128 groups; zero vectors past vend) are already
// in registers: e4m3 codes + one power-of-two scale per group, to each placed row of
// the token.  All passes are quantised before any store, so the stores of one row go
// out back to back from one base address; the scales of pass p -- group 2p + h held by
// half h of the warp after its amax reduction -- are stored by lane 16h + j for entry j
// (and j + 16), one store instruction per pass for up to 16 entries.
__device__ __forceinline__ void dispatch_fp8_item_regs(int kk, int nvec, const uint4 (&raw)[4], int vbeg, int vend,
                                                       int my_slot, uint2* __restrict__ xe,
                                                       float* __restrict__ xe_scale, int64_t scale_cs, int lane) {
    const int ngroups = nvec / 16;
    uint2 q[4];
    float sc[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        float amax = amax_bf16x8(raw[p]);
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const int s = fp8_scale_exp(amax);
        const Pow2Factors f = pow2_neg(s);  // x * 2^-s, exactly as scalbnf
        const uint32_t wds[4] = {raw[p].x, raw[p].y, raw[p].z, raw[p].w};
        uint16_t pk[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            pk[i] = f2_to_e4m3x2(scale_by(bf16_bits_to_f((uint16_t)(wds[i] & 0xffffu)), f),
                                 scale_by(bf16_bits_to_f((uint16_t)(wds[i] >> 16)), f));
        q[p] = make_uint2((uint32_t)pk[0] | ((uint32_t)pk[1] << 16), (uint32_t)pk[2] | ((uint32_t)pk[3] << 16));
        sc[p] = mul_pow2(1.0f, s);
    }
    const int npass = (vend - vbeg + 31) / 32;
    const int g0 = vbeg / 16 + (lane >> 4);
    for (int jb = 0; jb < kk; jb += 16) {
        const int j = jb + (lane & 15);
        const int r = __shfl_sync(0xffffffffu, my_slot, j & 31);
        if (j < kk && r >= 0) {
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                if (vbeg + 32 * p + (lane & 16) >= vend) continue;  // this half's group is past the slice
                const int g = g0 + 2 * p;
                xe_scale[scale_cs ? (size_t)g * scale_cs + r : (size_t)r * ngroups + g] = sc[p];
            }
        }
    }
    for (int j = 0; j < kk; ++j) {
        const int r = __shfl_sync(0xffffffffu, my_slot, j);
        if (r < 0) continue;
        uint2* dst = xe + (size_t)r * nvec + vbeg + lane;
#pragma unroll
        for (int p = 0; p < 4; ++p)
            if (p < npass && vbeg + 32 * p + lane < vend) dst[32 * p] = q[p];
    }
}

// Loads one item's four passes of bf16 vectors (zero past vend).
__device__ __forceinline__ void load_item(const uint4* __restrict__ src, int vbeg, int vend, int lane,
                                          uint4 (&raw)[4]) {
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const int v = vbeg + 32 * p + lane;
        raw[p] = v < vend ? __ldg(src + v) : make_uint4(0u, 0u, 0u, 0u);
    }
}

// bf16 row -> e4m3 codes + one power-of-two scale per 1x128 group, vectors
// [vbeg, vend) of 8 bf16 each (whole groups), the slice's four passes loaded at once.
__device__ __forceinline__ void dispatch_fp8_item(int kk, int nvec, const uint4* __restrict__ src, int vbeg,
                                                  int vend, int my_slot, uint2* __restrict__ xe,
                                                  float* __restrict__ xe_scale, int64_t scale_cs, int lane) {
    uint4 raw[4];
    load_item(src, vbeg, vend, lane, raw);
    dispatch_fp8_item_regs(kk, nvec, raw, vbeg, vend, my_slot, xe, xe_scale, scale_cs, lane);
}

}  // namespace moe
