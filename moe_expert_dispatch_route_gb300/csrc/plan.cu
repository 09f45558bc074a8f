// moe_plan kernels: a deterministic, stable counting sort of the (token, choice)
// entries by expert; slot assignment uses only order-independent integer adds.
//
// A batch of up to 4096 entries is one chunk; a larger one is cut into chunks of whole
// tokens of about 1024 entries each, so that the passes spread over many SMs.
//   pass 1 (plan_count_kernel, skipped when there is one chunk): one CTA per chunk
//           writes the chunk's per-expert histogram to the workspace.
//   pass 2 (plan_assign_kernel): one CTA per chunk re-derives the global counts and
//           its chunk's starting rank per expert from the histograms, scans the
//           (aligned) counts into offsets, then walks its entries in order, 256 at a
//           time: __match_any_sync groups equal experts within a warp (rank = peers
//           below this lane), a per-warp count table in shared memory gives the
//           rank contributed by earlier warps, and a running per-expert base
//           carries the rank across steps.  Slots are therefore the stable
//           (t, j)-order ranks, identical on every run.
#include "common.cuh"
#include "kernels.h"
#include "plan_impl.cuh"

namespace moe {

int plan_tokens_per_chunk(const moe_config& c, int T) {
    const int kk = c.top_k + c.num_shared;
    const int tpc = ((int64_t)T * kk <= kPlanEntriesPerChunk ? kPlanEntriesPerChunk : kPlanEntriesPerChunkMulti) / kk;
    return tpc < 1 ? 1 : tpc;
}

int plan_num_chunks(const moe_config& c, int T) {
    const int tpc = plan_tokens_per_chunk(c, T);
    return (T + tpc - 1) / tpc;
}

__global__ void __launch_bounds__(kPlanThreads) plan_count_kernel(int T, int k, int S, int E, int tpc,
                                                                  const int32_t* __restrict__ ids,
                                                                  int32_t* __restrict__ hist) {
    __shared__ int h[kMaxExperts];
    pdl_begin();
    const int NE = E + S, kk = k + S;
    for (int e = threadIdx.x; e < NE; e += blockDim.x) h[e] = 0;
    __syncthreads();
    const int t0 = blockIdx.x * tpc;
    const int t1 = min(T, t0 + tpc);
    const int n = (t1 - t0) * kk;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        int t = t0 + i / kk, j = i % kk;
        int e = entry_expert(ids, t, j, k, E);
        if (e >= 0) atomicAdd(&h[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < NE; e += blockDim.x) hist[(size_t)blockIdx.x * NE + e] = h[e];
}

__global__ void __launch_bounds__(kPlanThreads) plan_assign_kernel(
    int T, int k, int S, int E, int tpc, int nchunks, int capacity, int align,
    const int32_t* __restrict__ ids, const int32_t* __restrict__ hist, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ slot_of, int32_t* __restrict__ token_of,
    int32_t* err) {
    extern __shared__ int chunk_e[];  // this chunk's entry experts (-1 = bad id)
    pdl_begin();
    plan_assign_cta(T, k, S, E, tpc, nchunks, blockIdx.x, capacity, align, ids, hist, counts, offsets, slot_of,
                    token_of, err, chunk_e, nullptr, true);
}

cudaError_t launch_plan(const moe_config& c, int T, const int32_t* ids, int capacity, int align,
                        int32_t* counts, int32_t* offsets, int32_t* slot_of, int32_t* token_of,
                        int32_t* err, int32_t* hist_ws, int grid_cap, cudaStream_t st) {
    (void)grid_cap;  // one CTA per chunk: the plan is latency-bound and needs few CTAs
    const int tpc = plan_tokens_per_chunk(c, T);
    int nchunks = (T + tpc - 1) / tpc;
    if (nchunks < 1) nchunks = 1;  // T == 0 still writes counts and offsets
    if (nchunks > 1) {
        cudaError_t e = launch_pdl(plan_count_kernel, nchunks, kPlanThreads, 0, st, T, c.top_k, c.num_shared,
                                   c.num_experts, tpc, ids, hist_ws);
        if (e != cudaSuccess) return e;
    }
    const size_t ids_smem = (size_t)tpc * (c.top_k + c.num_shared) * sizeof(int);
    return launch_pdl(plan_assign_kernel, nchunks, kPlanThreads, ids_smem, st, T, c.top_k, c.num_shared,
                      c.num_experts, tpc, nchunks, capacity, align, ids, (const int32_t*)hist_ws, counts, offsets,
                      slot_of, token_of, err);
}

}  // namespace moe
