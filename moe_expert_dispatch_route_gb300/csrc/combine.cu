// moe_combine kernel: a warp takes one token's slice of 64 16-byte column blocks,
// gathers the token's k+S expert-output rows there with 16-byte loads (two blocks a
// lane, up to 16 row loads in flight), accumulates w_j * ye in fp32 in the fixed
// (j, then s) order (optionally starting from a residual row) and stores once.
// No atomics: every output element is written by exactly one lane.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kCombineThreads = 256;

template <bool kF32>
__device__ __forceinline__ void unpack16(const uint4& v, float* f) {
    const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
    if (kF32) {
#pragma unroll
        for (int i = 0; i < 4; ++i) f[i] = __uint_as_float(wd[i]);
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = bf16_bits_to_f((uint16_t)(wd[i] & 0xffffu));
            f[2 * i + 1] = bf16_bits_to_f((uint16_t)(wd[i] >> 16));
        }
    }
}

template <bool kF32>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(
    int T, int k, int kk, int nvec, const uint4* __restrict__ ye, const float* __restrict__ w,
    const int32_t* __restrict__ slot_of, uint4* __restrict__ y, const uint4* __restrict__ resid) {
    pdl_begin();
    constexpr int kPer = kF32 ? 4 : 8;  // elements per 16-byte vector
    constexpr int kV = 2;               // column blocks per lane per pass
    const int lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    // work item = (token, slice of 32 * kV column blocks): small batches still spread
    // over many warps
    const int nslices = (nvec + 32 * kV - 1) / (32 * kV);
    const int items = T * nslices;
    for (int it = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; it < items; it += nwarps) {
        const int t = it / nslices;
        const int v0 = (it - t * nslices) * 32 * kV;
        const int my_slot = lane < kk ? __ldg(slot_of + (size_t)t * kk + lane) : -1;
        const float my_w = lane < k ? __ldg(w + (size_t)t * k + lane) : 1.0f;
        {
            float acc[kV][kPer];
#pragma unroll
            for (int b = 0; b < kV; ++b) {
                const int v = v0 + 32 * b + lane;
#pragma unroll
                for (int i = 0; i < kPer; ++i) acc[b][i] = 0.0f;
                if (resid && v < nvec) unpack16<kF32>(__ldg(resid + (size_t)t * nvec + v), acc[b]);
            }
            for (int j0 = 0; j0 < kk; j0 += 8) {
                uint4 val[8][kV];
                int r[8];
                float wj[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int j = j0 + u;
                    r[u] = __shfl_sync(0xffffffffu, my_slot, j & 31);
                    wj[u] = __shfl_sync(0xffffffffu, my_w, j & 31);
                    if (j >= kk) r[u] = -1;
#pragma unroll
                    for (int b = 0; b < kV; ++b) {
                        const int v = v0 + 32 * b + lane;
                        if (r[u] >= 0 && v < nvec) val[u][b] = __ldg(ye + (size_t)r[u] * nvec + v);
                    }
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    if (r[u] < 0) continue;
#pragma unroll
                    for (int b = 0; b < kV; ++b) {
                        if (v0 + 32 * b + lane >= nvec) continue;
                        float f[kPer];
                        unpack16<kF32>(val[u][b], f);
#pragma unroll
                        for (int i = 0; i < kPer; ++i) acc[b][i] = fmaf(wj[u], f[i], acc[b][i]);
                    }
                }
            }
#pragma unroll
            for (int b = 0; b < kV; ++b) {
                const int v = v0 + 32 * b + lane;
                if (v >= nvec) continue;
                uint4 out;
                if (kF32) {
                    out = make_uint4(__float_as_uint(acc[b][0]), __float_as_uint(acc[b][1]), __float_as_uint(acc[b][2]),
                                     __float_as_uint(acc[b][3]));
                } else {
                    out = make_uint4(pack_bf16x2(acc[b][0], acc[b][1]), pack_bf16x2(acc[b][2], acc[b][3]),
                                     pack_bf16x2(acc[b][4], acc[b][5]), pack_bf16x2(acc[b][6], acc[b][7]));
                }
                y[(size_t)t * nvec + v] = out;
            }
        }
    }
}

cudaError_t launch_combine(const moe_config& c, int T, const void* ye, const float* w,
                           const int32_t* slot_of, void* y, int grid_cap, cudaStream_t st, const void* resid) {
    if (T <= 0) return cudaSuccess;
    const int kk = c.top_k + c.num_shared;
    const int nvec = c.hidden * io_bytes(c.dtype) / 16;
    const long items = (long)T * ((nvec + 63) / 64);
    int grid = (int)((items + 7) / 8);
    if (grid > grid_cap) grid = grid_cap;
    if (c.dtype == MOE_F32)
        return launch_pdl(combine_kernel<true>, grid, kCombineThreads, 0, st, T, c.top_k, kk, nvec,
                          static_cast<const uint4*>(ye), w, slot_of, static_cast<uint4*>(y),
                          static_cast<const uint4*>(resid));
    return launch_pdl(combine_kernel<false>, grid, kCombineThreads, 0, st, T, c.top_k, kk, nvec,
                      static_cast<const uint4*>(ye), w, slot_of, static_cast<uint4*>(y),
                      static_cast<const uint4*>(resid));
}

}  // namespace moe
