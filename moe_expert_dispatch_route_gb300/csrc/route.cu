// moe_route kernels: one warp per token.
//
// Softmax gate and grouped-sigmoid gate as stated in moe.h.  Logits are read with
// coalesced 128-byte warp loads (lane l holds experts l, l+32, ...); the top-k
// selection is k rounds of a warp arg-max on (score desc, id asc); weights use
// warp reductions in a fixed butterfly order (deterministic).
#include "common.cuh"
#include "kernels.h"
#include "route_impl.cuh"

namespace moe {

template <int NPER>
__global__ void __launch_bounds__(256) route_softmax_kernel(int T, int E, int k, int renorm,
                                                            const float* __restrict__ logits,
                                                            int32_t* __restrict__ ids,
                                                            float* __restrict__ w) {
    pdl_begin();
    const int lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += nwarps) {
        int id;
        float wt;
        route_token_softmax<NPER>(t, E, k, renorm, logits, id, wt);
        if (lane < k) {
            ids[(size_t)t * k + lane] = id;
            w[(size_t)t * k + lane] = wt;
        }
    }
}

template <int NPER, bool kSqrtSoftplus>
__global__ void __launch_bounds__(256) route_grouped_kernel(int T, int E, int k, int n_group,
                                                            int topk_group, int renorm, float scale,
                                                            const float* __restrict__ logits,
                                                            const float* __restrict__ bias,
                                                            int32_t* __restrict__ ids,
                                                            float* __restrict__ w) {
    extern __shared__ float route_smem[];
    pdl_begin();
    float* cs = route_smem + (threadIdx.x >> 5) * E;  // this warp's choice scores
    const int lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += nwarps) {
        int id;
        float wt;
        route_token_grouped<NPER, kSqrtSoftplus>(t, E, k, n_group, topk_group, renorm, scale, logits, bias, cs, id,
                                                 wt);
        if (lane < k) {
            ids[(size_t)t * k + lane] = id;
            w[(size_t)t * k + lane] = wt;
        }
    }
}

template <int NPER>
static cudaError_t launch_route_n(const moe_config& c, int T, const float* logits, const float* bias,
                                  int32_t* ids, float* w, int grid, cudaStream_t st) {
    if (c.gate == MOE_GATE_SOFTMAX)
        return launch_pdl(route_softmax_kernel<NPER>, grid, 256, 0, st, T, c.num_experts, c.top_k, c.renormalize,
                          logits, ids, w);
    const size_t smem = sizeof(float) * 8 * c.num_experts;
    if (c.gate == MOE_GATE_SQRT_SOFTPLUS)
        return launch_pdl(route_grouped_kernel<NPER, true>, grid, 256, smem, st, T, c.num_experts, c.top_k, c.n_group,
                          c.topk_group, c.renormalize, c.routed_scale, logits, bias, ids, w);
    return launch_pdl(route_grouped_kernel<NPER, false>, grid, 256, smem, st, T, c.num_experts, c.top_k, c.n_group,
                      c.topk_group, c.renormalize, c.routed_scale, logits, bias, ids, w);
}

// Hash routing (DeepSeek-V4-shaped layers): one warp per token; lane j < k takes expert
// table[token_ids[t]][j] and its sqrt-softplus weight, renormalised over the k and
// scaled.  A token id outside [0, vocab) gives ids -1 and weights 0; a table entry
// outside [0, E) is passed on (the plan flags it) with weight 0.
__global__ void __launch_bounds__(256) route_hash_kernel(int T, int E, int k, int renorm, float scale, int vocab,
                                                         const float* __restrict__ logits,
                                                         const int32_t* __restrict__ token_ids,
                                                         const int32_t* __restrict__ table, int32_t* __restrict__ ids,
                                                         float* __restrict__ w) {
    pdl_begin();
    const int lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += nwarps) {
        const int tid = __ldg(token_ids + t);
        int e = -1;
        float s = 0.0f;
        if (lane < k && tid >= 0 && tid < vocab) {
            e = __ldg(table + (size_t)tid * k + lane);
            if (e >= 0 && e < E) s = sqrt_softplus(__ldg(logits + (size_t)t * E + e));
        }
        const float sum = warp_sum(s);
        if (lane < k) {
            ids[(size_t)t * k + lane] = e;
            w[(size_t)t * k + lane] = ((renorm && sum > 0.0f) ? s / sum : s) * scale;
        }
    }
}

cudaError_t launch_route_hash(const moe_config& c, int T, const float* logits, const int32_t* token_ids,
                              const int32_t* table, int vocab, int32_t* ids, float* w, int grid_cap, cudaStream_t st) {
    if (T <= 0) return cudaSuccess;
    int grid = (T + 7) / 8;
    if (grid > grid_cap) grid = grid_cap;
    return launch_pdl(route_hash_kernel, grid, 256, 0, st, T, c.num_experts, c.top_k, c.renormalize, c.routed_scale,
                      vocab, logits, token_ids, table, ids, w);
}

cudaError_t launch_route(const moe_config& c, int T, const float* logits, const float* bias,
                         int32_t* ids, float* w, int grid_cap, cudaStream_t st) {
    if (T <= 0) return cudaSuccess;
    int grid = (T + 7) / 8;
    if (grid > grid_cap) grid = grid_cap;
    int E = c.num_experts;
    if (E <= 32) return launch_route_n<1>(c, T, logits, bias, ids, w, grid, st);
    if (E <= 64) return launch_route_n<2>(c, T, logits, bias, ids, w, grid, st);
    if (E <= 128) return launch_route_n<4>(c, T, logits, bias, ids, w, grid, st);
    if (E <= 256) return launch_route_n<8>(c, T, logits, bias, ids, w, grid, st);
    return launch_route_n<16>(c, T, logits, bias, ids, w, grid, st);
}

}  // namespace moe
