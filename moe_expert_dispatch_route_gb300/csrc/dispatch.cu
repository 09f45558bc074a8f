// moe_dispatch kernels: a warp takes one token's slice of 128 16-byte vectors; the
// slice is read once with coalesced 16-byte loads and written to each of the token's
// k+S destination rows with 16-byte (8-byte for fp8) stores.  FP8 layers quantise each 1x128 group on the fly: a
// half-warp owns one group (16 lanes x 8 bf16), reduces its amax with four
// shuffles and converts with cvt.rn.satfinite.e4m3x2.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int kDispatchThreads = 256;

// fp32 / bf16 layers: plain row copy.  nvec = 16-byte vectors per row.
__global__ void __launch_bounds__(kDispatchThreads) dispatch_copy_kernel(
    int T, int kk, int nvec, const uint4* __restrict__ x, const int32_t* __restrict__ slot_of,
    uint4* __restrict__ xe) {
    pdl_begin();
    const int lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    // work item = (token, slice of 128 16-byte vectors)
    const int nslices = (nvec + 127) / 128;
    const int items = T * nslices;
    for (int it = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; it < items; it += nwarps) {
        const int t = it / nslices;
        const int v0 = (it - t * nslices) * 128;
        const int my_slot = lane < kk ? __ldg(slot_of + (size_t)t * kk + lane) : -1;
        const uint4* src = x + (size_t)t * nvec;
        {
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
    }
}

// fp8 layers: bf16 row -> e4m3 codes + one power-of-two scale per 1x128 group.
__global__ void __launch_bounds__(kDispatchThreads) dispatch_fp8_kernel(
    int T, int kk, int H, const uint4* __restrict__ x, const int32_t* __restrict__ slot_of,
    uint2* __restrict__ xe, float* __restrict__ xe_scale) {
    pdl_begin();
    const int lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    const int nvec = H / 8;     // 8 bf16 per 16-byte vector
    const int ngroups = H / kQG;
    // work item = (token, slice of 128 vectors = 8 groups of 1x128), passes of 32
    const int nslices = (nvec + 127) / 128;
    const int items = T * nslices;
    for (int it = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; it < items; it += nwarps) {
        const int t = it / nslices;
        const int vbeg = (it - t * nslices) * 128;
        const int vend = min(nvec, vbeg + 128);
        const int my_slot = lane < kk ? __ldg(slot_of + (size_t)t * kk + lane) : -1;
        const uint4* src = x + (size_t)t * nvec;
        // the row is read ahead one pass (two 16-byte loads a lane in flight)
        uint4 next = vbeg + lane < vend ? __ldg(src + vbeg + lane) : make_uint4(0u, 0u, 0u, 0u);
        for (int v = vbeg + lane; v - lane < vend; v += 32) {
            // H is a multiple of 128, so a half-warp is either fully inside or fully out
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
                if ((lane & 15) == 0) xe_scale[(size_t)r * ngroups + v / 16] = scale;
            }
        }
    }
}

cudaError_t launch_dispatch(const moe_config& c, int T, const void* x, const int32_t* slot_of,
                            void* xe, float* xe_scale, int grid_cap, cudaStream_t st) {
    if (T <= 0) return cudaSuccess;
    const int kk = c.top_k + c.num_shared;
    const int nvec_io = c.hidden * io_bytes(c.dtype) / 16;
    const long items = (long)T * ((nvec_io + 127) / 128);
    int grid = (int)((items + 7) / 8);
    if (grid > grid_cap) grid = grid_cap;
    if (c.dtype == MOE_FP8_E4M3)
        return launch_pdl(dispatch_fp8_kernel, grid, kDispatchThreads, 0, st, T, kk, c.hidden,
                          static_cast<const uint4*>(x), slot_of, static_cast<uint2*>(xe), xe_scale);
    const int nvec = c.hidden * elt_bytes(c.dtype) / 16;
    return launch_pdl(dispatch_copy_kernel, grid, kDispatchThreads, 0, st, T, kk, nvec, static_cast<const uint4*>(x),
                      slot_of, static_cast<uint4*>(xe));
}

}  // namespace moe
