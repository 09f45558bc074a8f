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

// bf16 row -> e4m3 codes + one power-of-two scale per 1x128 group, vectors
// [vbeg, vend) of 8 bf16 each (whole groups), passes of 32 vectors read one ahead.
__device__ __forceinline__ void dispatch_fp8_item(int kk, int nvec, const uint4* __restrict__ src, int vbeg,
                                                  int vend, int my_slot, uint2* __restrict__ xe,
                                                  float* __restrict__ xe_scale, int64_t scale_cs, int lane) {
    const int ngroups = nvec / 16;
    uint4 next = vbeg + lane < vend ? __ldg(src + vbeg + lane) : make_uint4(0u, 0u, 0u, 0u);
    for (int v = vbeg + lane; v - lane < vend; v += 32) {
        // groups are 16 vectors, so a half-warp is either fully inside or fully out
        const bool in = v < vend;
        float f[8];
        float amax = 0.0f;
        const uint4 raw = next;
        if (v + 32 < vend) next = __ldg(src + v + 32);
        if (in) {
            const uint32_t wds[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                f[2 * i] = bf16_bits_to_f((uint16_t)(wds[i] & 0xffffu));
                f[2 * i + 1] = bf16_bits_to_f((uint16_t)(wds[i] >> 16));
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const int s = fp8_scale_exp(amax);
        uint2 q = make_uint2(0u, 0u);
        if (in) {
            uint16_t p[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) p[i] = f2_to_e4m3x2(scalbnf(f[2 * i], -s), scalbnf(f[2 * i + 1], -s));
            q.x = (uint32_t)p[0] | ((uint32_t)p[1] << 16);
            q.y = (uint32_t)p[2] | ((uint32_t)p[3] << 16);
        }
        const float scale = scalbnf(1.0f, s);
        for (int j = 0; j < kk; ++j) {
            const int r = __shfl_sync(0xffffffffu, my_slot, j);
            if (r < 0 || !in) continue;
            xe[(size_t)r * nvec + v] = q;
            if ((lane & 15) == 0)
                xe_scale[scale_cs ? (size_t)(v / 16) * scale_cs + r : (size_t)r * ngroups + v / 16] = scale;
        }
    }
}

}  // namespace moe
