// The low-latency head of a ubatch: plan and dispatch in one launch.
//
// For a batch whose plan is a single chunk (T * (k+S) <= 4096 entries) every CTA derives
// the whole plan in shared memory -- it is small and deterministic, so every CTA gets
// the same slots -- CTA 0 also writes counts / offsets / slot_of for the FFN and the
// combine, and then each CTA dispatches its share of (token, slice) work items with the
// slots it holds.  No CTA waits on another, and the plan -> dispatch round trip through
// global memory and the second launch are gone.  Results are identical to moe_plan
// followed by moe_dispatch (token_of is not produced).
#include "common.cuh"
#include "dispatch_impl.cuh"
#include "kernels.h"
#include "plan_impl.cuh"

namespace moe {

template <bool kFp8>
__global__ void __launch_bounds__(kPlanThreads) plan_dispatch_kernel(
    int T, int k, int S, int E, int capacity, int align, const int32_t* __restrict__ ids,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ slot_of, int32_t* err,
    const uint4* __restrict__ x, void* __restrict__ xe, float* __restrict__ xe_scale, int64_t scale_cs, int nvec) {
    extern __shared__ int head_sm[];
    pdl_begin();
    const int kk = k + S;
    const int n = T * kk;
    int* chunk_e = head_sm;
    int* slot_sm = head_sm + n;
    plan_assign_cta(T, k, S, E, T, 1, 0, capacity, align, ids, nullptr, counts, offsets, slot_of, nullptr, err,
                    chunk_e, slot_sm, blockIdx.x == 0);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int warps = blockDim.x >> 5;
    const int nslices = (nvec + 127) / 128;
    const int items = T * nslices;
    for (int it = blockIdx.x * warps + (threadIdx.x >> 5); it < items; it += gridDim.x * warps) {
        const int t = it / nslices;
        const int vbeg = (it - t * nslices) * 128;
        const int my_slot = lane < kk ? slot_sm[t * kk + lane] : -1;
        if (kFp8)
            dispatch_fp8_item(kk, nvec, x + (size_t)t * nvec, vbeg, min(nvec, vbeg + 128), my_slot,
                              static_cast<uint2*>(xe), xe_scale, scale_cs, lane);
        else
            dispatch_copy_item(kk, nvec, x + (size_t)t * nvec, vbeg, my_slot, static_cast<uint4*>(xe), lane);
    }
}

bool plan_dispatch_fusable(const moe_config& c, int T) { return T > 0 && plan_num_chunks(c, T) == 1; }

template <bool kFp8>
static cudaError_t launch_fused(const moe_config& c, int T, const int32_t* ids, int capacity, int align,
                                int32_t* counts, int32_t* offsets, int32_t* slot_of, int32_t* err, const void* x,
                                void* xe, float* xe_scale, int64_t scale_cs, int grid_cap, cudaStream_t st) {
    const int kk = c.top_k + c.num_shared;
    const size_t smem = 2 * (size_t)T * kk * sizeof(int);
    // the static plan tables plus up to 32 KB of entries exceed the default 48 KB
    cudaError_t e = ensure_max_dynamic_smem(plan_dispatch_kernel<kFp8>, 2 * kPlanEntriesPerChunk * (int)sizeof(int));
    if (e != cudaSuccess) return e;
    const int nvec = kFp8 ? c.hidden / 8 : c.hidden * elt_bytes(c.dtype) / 16;
    const int nvec_io = c.hidden * io_bytes(c.dtype) / 16;
    const long items = (long)T * ((nvec_io + 127) / 128);
    int grid = (int)((items + kPlanWarps - 1) / kPlanWarps);
    if (grid > grid_cap) grid = grid_cap;
    if (grid < 1) grid = 1;
    return launch_pdl(plan_dispatch_kernel<kFp8>, grid, kPlanThreads, smem, st, T, c.top_k, c.num_shared,
                      c.num_experts, capacity, align, ids, counts, offsets, slot_of, err,
                      static_cast<const uint4*>(x), xe, xe_scale, scale_cs, nvec);
}

cudaError_t launch_plan_dispatch(const moe_config& c, int T, const int32_t* ids, int capacity, int align,
                                 int32_t* counts, int32_t* offsets, int32_t* slot_of, int32_t* err, const void* x,
                                 void* xe, float* xe_scale, int64_t scale_cs, int grid_cap, cudaStream_t st) {
    if (c.dtype == MOE_FP8_E4M3)
        return launch_fused<true>(c, T, ids, capacity, align, counts, offsets, slot_of, err, x, xe, xe_scale,
                                  scale_cs, grid_cap, st);
    return launch_fused<false>(c, T, ids, capacity, align, counts, offsets, slot_of, err, x, xe, xe_scale, scale_cs,
                               grid_cap, st);
}

}  // namespace moe
