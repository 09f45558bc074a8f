// moe_dispatch kernels: a warp takes one token's slice of 128 16-byte vectors; the
// slice is read once with coalesced 16-byte loads and written to each of the token's
// k+S destination rows with 16-byte (8-byte for fp8) stores.
//
// fp32 / bf16 layers: a grid of at most one CTA per SM whose warps walk the items with
// the next item's vectors and slots loaded before the current item's stores, so that
// loads and stores overlap within a warp.  FP8 layers quantise each 1x128 group on the
// fly (dispatch_impl.cuh: a half-warp per group, amax on packed bf16, power-of-two scale,
// cvt.rn.satfinite.e4m3x2), one item per warp.
//
// Measured on GB300 (bench's comm-kernel timing) against a shared-memory staged form
// (bulk async copies in, bulk async stores out, three CTAs per SM): that form was slower
// for every workload measured, as was pipelining the fp8 path (its extra registers
// halve the resident warps).
#include "common.cuh"
#include "dispatch_impl.cuh"
#include "kernels.h"

namespace moe {

constexpr int kDispatchThreads = 256;

// fp32 / bf16 layers: row copy, pipelined over the warp's items.  nvec = 16-byte
// vectors per row.
__global__ void __launch_bounds__(kDispatchThreads) dispatch_copy_kernel(
    int T, int kk, int nvec, const uint4* __restrict__ x, const int32_t* __restrict__ slot_of,
    uint4* __restrict__ xe) {
    pdl_begin();
    const int lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    const int nslices = (nvec + 127) / 128;
    const int items = T * nslices;
    int it = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    uint4 nval[4];
    int nslot = -1;
    auto load = [&](int item) {
        const int t = item / nslices;
        const int v0 = (item - t * nslices) * 128;
        nslot = lane < kk ? __ldg(slot_of + (size_t)t * kk + lane) : -1;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int v = v0 + u * 32 + lane;
            if (v < nvec) nval[u] = __ldg(x + (size_t)t * nvec + v);
        }
    };
    if (it < items) load(it);
    for (; it < items; it += nwarps) {
        const int t = it / nslices;
        const int v0 = (it - t * nslices) * 128;
        uint4 val[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) val[u] = nval[u];
        const int my_slot = nslot;
        if (it + nwarps < items) load(it + nwarps);  // in flight during this item's stores
        for (int j = 0; j < kk; ++j) {
            const int r = __shfl_sync(0xffffffffu, my_slot, j);
            if (r < 0) continue;
            uint4* dst = xe + (size_t)r * nvec;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int v = v0 + u * 32 + lane;
                if (v < nvec) dst[v] = val[u];
            }
        }
    }
}

// fp8 layers: bf16 row -> e4m3 codes + one power-of-two scale per 1x128 group.
__global__ void __launch_bounds__(kDispatchThreads) dispatch_fp8_kernel(
    int T, int kk, int H, const uint4* __restrict__ x, const int32_t* __restrict__ slot_of,
    uint2* __restrict__ xe, float* __restrict__ xe_scale, int64_t scale_cs) {
    pdl_begin();
    const int lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    const int nvec = H / 8;  // 8 bf16 per 16-byte vector
    const int nslices = (nvec + 127) / 128;
    const int items = T * nslices;
    for (int it = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; it < items; it += nwarps) {
        const int t = it / nslices;
        const int vbeg = (it - t * nslices) * 128;
        const int my_slot = lane < kk ? __ldg(slot_of + (size_t)t * kk + lane) : -1;
        dispatch_fp8_item(kk, nvec, x + (size_t)t * nvec, vbeg, min(nvec, vbeg + 128), my_slot, xe, xe_scale, scale_cs,
                          lane);
    }
}

// Fused gather (fp8 layers): every token's row quantised once -- e4m3 codes x_q [T][H]
// and the power-of-two 1x128 scales, column-major (group g of token t at g * scale_cs +
// t) -- with the arithmetic of dispatch_fp8_kernel, so the expert FFN that gathers x_q
// rows by token sees the bytes dispatch would have written to each slot.
__global__ void __launch_bounds__(kDispatchThreads) quantize_rows_kernel(int T, int H, const uint4* __restrict__ x,
                                                                         uint2* __restrict__ xq,
                                                                         float* __restrict__ xs, int64_t scale_cs) {
    pdl_begin();
    const int lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    const int nvec = H / 8;
    const int nslices = (nvec + 127) / 128;
    const int items = T * nslices;
    for (int it = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; it < items; it += nwarps) {
        const int t = it / nslices;
        const int vbeg = (it - t * nslices) * 128;
        dispatch_fp8_item(1, nvec, x + (size_t)t * nvec, vbeg, min(nvec, vbeg + 128), lane == 0 ? t : -1, xq, xs,
                          scale_cs, lane);
    }
}

cudaError_t launch_quantize_rows(const moe_config& c, int T, const void* x, void* xq, float* xs, int64_t scale_cs,
                                 int grid_cap, cudaStream_t st) {
    if (T <= 0) return cudaSuccess;
    const long items = (long)T * ((c.hidden / 8 + 127) / 128);
    int grid = (int)((items + 7) / 8);
    if (grid > grid_cap) grid = grid_cap;
    return launch_pdl(quantize_rows_kernel, grid, kDispatchThreads, 0, st, T, c.hidden, static_cast<const uint4*>(x),
                      static_cast<uint2*>(xq), xs, scale_cs);
}

cudaError_t launch_dispatch(const moe_config& c, int T, const void* x, const int32_t* slot_of,
                            void* xe, float* xe_scale, int64_t scale_cs, int grid_cap, cudaStream_t st) {
    if (T <= 0) return cudaSuccess;
    const int kk = c.top_k + c.num_shared;
    const int nvec_io = c.hidden * io_bytes(c.dtype) / 16;
    const long items = (long)T * ((nvec_io + 127) / 128);
    int grid = (int)((items + 7) / 8);
    if (c.dtype == MOE_FP8_E4M3) {
        if (grid > grid_cap) grid = grid_cap;
        return launch_pdl(dispatch_fp8_kernel, grid, kDispatchThreads, 0, st, T, kk, c.hidden,
                          static_cast<const uint4*>(x), slot_of, static_cast<uint2*>(xe), xe_scale, scale_cs);
    }
    // at most one CTA per SM: each warp then walks several items and overlaps them
    if (grid > device_info().num_sms) grid = device_info().num_sms;
    if (grid > grid_cap) grid = grid_cap;
    const int nvec = c.hidden * elt_bytes(c.dtype) / 16;
    return launch_pdl(dispatch_copy_kernel, grid, kDispatchThreads, 0, st, T, kk, nvec, static_cast<const uint4*>(x),
                      slot_of, static_cast<uint4*>(xe));
}

}  // namespace moe
