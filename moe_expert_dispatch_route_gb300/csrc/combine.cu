// moe_combine kernel: one warp per token gathers its k+S expert-output rows with
// 16-byte loads (all k+S loads of a column block in flight together), accumulates
// w_j * ye in fp32 in the fixed (j, then s) order and stores the row once.
// No atomics: every output element is written by exactly one lane.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kCombineThreads = 256;

template <bool kF32>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(
    int T, int k, int kk, int nvec, const uint4* __restrict__ ye, const float* __restrict__ w,
    const int32_t* __restrict__ slot_of, uint4* __restrict__ y, const uint4* __restrict__ resid) {
    pdl_begin();
    constexpr int kPer = kF32 ? 4 : 8;  // elements per 16-byte vector
    const int lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += nwarps) {
        const int my_slot = lane < kk ? __ldg(slot_of + (size_t)t * kk + lane) : -1;
        const float my_w = lane < k ? __ldg(w + (size_t)t * k + lane) : 1.0f;
        for (int v = lane; v < nvec; v += 32) {
            float acc[kPer];
#pragma unroll
            for (int i = 0; i < kPer; ++i) acc[i] = 0.0f;
            if (resid) {  // the residual starts the sum (one rounding at the end)
                const uint4 rv = __ldg(resid + (size_t)t * nvec + v);
                const uint32_t rd[4] = {rv.x, rv.y, rv.z, rv.w};
                if (kF32) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[i] = __uint_as_float(rd[i]);
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        acc[2 * i] = bf16_bits_to_f((uint16_t)(rd[i] & 0xffffu));
                        acc[2 * i + 1] = bf16_bits_to_f((uint16_t)(rd[i] >> 16));
                    }
                }
            }
            int j = 0;
            for (; j + 8 <= kk; j += 8) {  // eight row loads in flight per lane
                uint4 val[8];
                int r[8];
                float wj[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    r[u] = __shfl_sync(0xffffffffu, my_slot, j + u);
                    wj[u] = __shfl_sync(0xffffffffu, my_w, j + u);
                    if (r[u] >= 0) val[u] = __ldg(ye + (size_t)r[u] * nvec + v);
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    if (r[u] < 0) continue;
                    const uint32_t wd[4] = {val[u].x, val[u].y, val[u].z, val[u].w};
                    if (kF32) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) acc[i] = fmaf(wj[u], __uint_as_float(wd[i]), acc[i]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            acc[2 * i] = fmaf(wj[u], bf16_bits_to_f((uint16_t)(wd[i] & 0xffffu)), acc[2 * i]);
                            acc[2 * i + 1] = fmaf(wj[u], bf16_bits_to_f((uint16_t)(wd[i] >> 16)), acc[2 * i + 1]);
                        }
                    }
                }
            }
            for (; j < kk; ++j) {
                const int r = __shfl_sync(0xffffffffu, my_slot, j);
                const float wj = __shfl_sync(0xffffffffu, my_w, j);
                if (r < 0) continue;
                const uint4 val = __ldg(ye + (size_t)r * nvec + v);
                const uint32_t wd[4] = {val.x, val.y, val.z, val.w};
                if (kF32) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[i] = fmaf(wj, __uint_as_float(wd[i]), acc[i]);
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        acc[2 * i] = fmaf(wj, bf16_bits_to_f((uint16_t)(wd[i] & 0xffffu)), acc[2 * i]);
                        acc[2 * i + 1] = fmaf(wj, bf16_bits_to_f((uint16_t)(wd[i] >> 16)), acc[2 * i + 1]);
                    }
                }
            }
            uint4 out;
            if (kF32) {
                out = make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]), __float_as_uint(acc[2]),
                                 __float_as_uint(acc[3]));
            } else {
                out = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                 pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
            }
            y[(size_t)t * nvec + v] = out;
        }
    }
}

cudaError_t launch_combine(const moe_config& c, int T, const void* ye, const float* w,
                           const int32_t* slot_of, void* y, int grid_cap, cudaStream_t st, const void* resid) {
    if (T <= 0) return cudaSuccess;
    const int kk = c.top_k + c.num_shared;
    const int nvec = c.hidden * io_bytes(c.dtype) / 16;
    int grid = (T + 7) / 8;
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
