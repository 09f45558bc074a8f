// The low-latency head of a ubatch: plan and dispatch in one launch, and for small
// batches route, plan and dispatch in one launch.
//
// For a batch whose plan is a single chunk (T * (k+S) <= 4096 entries) every CTA derives
// the whole plan in shared memory -- it is small and deterministic, so every CTA gets
// the same slots -- CTA 0 also writes counts / offsets / slot_of for the FFN and the
// combine, and then each CTA dispatches its share of (token, slice) work items with the
// slots it holds.  No CTA waits on another, and the plan -> dispatch round trip through
// global memory and the second launch are gone.  Results are identical to moe_plan
// followed by moe_dispatch (token_of is not produced).
#include <stdlib.h>
#include <string.h>

#include "common.cuh"
#include "dispatch_impl.cuh"
#include "kernels.h"
#include "plan_impl.cuh"
#include "route_impl.cuh"

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

// ---------------------------------------------------------------- route + plan + dispatch
//
// For a small batch (single-chunk plan, at most two tokens per warp of a cluster) the
// gate runs in the same launch.  The grid is made of thread-block clusters of up to 8
// CTAs: the warps of each cluster share out the tokens and route them into their own
// CTA's shared memory; after a cluster barrier (hardware, no polling) every CTA reads
// all the ids from their routing CTAs' shared memory, derives the whole plan as the
// fused plan + dispatch kernel does, and dispatches its share of (token, slice) items.
// The first cluster writes ids and weights, CTA 0 the plan.  Results are identical to
// moe_route, moe_plan and moe_dispatch in sequence (token_of is not produced).
constexpr int kHeadClusterMax = 8;
constexpr int kHeadTokensPerWarp = 2;

__device__ __forceinline__ uint32_t cluster_nctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The int at the same shared-memory offset as p in CTA `rank` of the cluster.
__device__ __forceinline__ int ld_peer_smem(const int* p, uint32_t rank) {
    uint32_t a, v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"((uint32_t)__cvta_generic_to_shared(p)), "r"(rank));
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
    return (int)v;
}

struct HeadArgs {
    int T, E, k, S, n_group, topk_group, renorm;
    float scale;
    const float* logits;
    const float* bias;
    int32_t* ids;
    float* w;
    int capacity, align;
    int32_t* counts;
    int32_t* offsets;
    int32_t* slot_of;
    int32_t* err;
    const uint4* x;
    void* xe;
    float* xe_scale;
    int64_t scale_cs;
    int nvec;
};

// kGate: the gate (moe_gate): softmax, group-limited sigmoid or sqrt-softplus.
template <int NPER, int kGate, bool kFp8>
__global__ void __launch_bounds__(kPlanThreads) route_plan_dispatch_kernel(const __grid_constant__ HeadArgs a) {
    constexpr bool kGrouped = kGate != MOE_GATE_SOFTMAX;
    extern __shared__ int head_sm[];
    pdl_begin();
    const int T = a.T, k = a.k, kk = a.k + a.S, n = T * kk;
    int* rid = head_sm;           // [T][k] routed ids: this CTA's tokens, then all
    int* chunk_e = rid + T * k;   // [T * kk]
    int* slot_sm = chunk_e + n;   // [T * kk]
    float* cs = reinterpret_cast<float*>(slot_sm + n);  // grouped gate: E floats a warp
    const uint32_t crank = cluster_ctarank(), csize = cluster_nctarank();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const bool writer = blockIdx.x < csize;  // the first cluster writes ids and weights
    for (int t = (int)crank * nw + warp; t < T; t += (int)csize * nw) {
        int id;
        float wt;
        if (kGrouped)
            route_token_grouped<NPER, kGate == MOE_GATE_SQRT_SOFTPLUS>(t, a.E, k, a.n_group, a.topk_group, a.renorm,
                                                                       a.scale, a.logits, a.bias, cs + warp * a.E, id,
                                                                       wt);
        else
            route_token_softmax<NPER>(t, a.E, k, a.renorm, a.logits, id, wt);
        if (lane < k) {
            rid[t * k + lane] = id;
            if (writer) {
                a.ids[(size_t)t * k + lane] = id;
                a.w[(size_t)t * k + lane] = wt;
            }
        }
    }
    cluster_barrier();  // every CTA's tokens are routed
    for (int i = threadIdx.x; i < T * k; i += blockDim.x) {
        const uint32_t owner = (uint32_t)(((i / k) % ((int)csize * nw)) / nw);
        if (owner != crank) rid[i] = ld_peer_smem(rid + i, owner);
    }
    cluster_barrier();  // no CTA reads a peer's shared memory past this point
    plan_assign_cta<true>(T, k, a.S, a.E, T, 1, 0, a.capacity, a.align, rid, nullptr, a.counts, a.offsets,
                          a.slot_of, nullptr, a.err, chunk_e, slot_sm, blockIdx.x == 0);
    __syncthreads();
    const int nslices = (a.nvec + 127) / 128;
    const int items = T * nslices;
    for (int it = blockIdx.x * nw + warp; it < items; it += gridDim.x * nw) {
        const int t = it / nslices;
        const int vbeg = (it - t * nslices) * 128;
        const int my_slot = lane < kk ? slot_sm[t * kk + lane] : -1;
        if (kFp8)
            dispatch_fp8_item(kk, a.nvec, a.x + (size_t)t * a.nvec, vbeg, min(a.nvec, vbeg + 128), my_slot,
                              static_cast<uint2*>(a.xe), a.xe_scale, a.scale_cs, lane);
        else
            dispatch_copy_item(kk, a.nvec, a.x + (size_t)t * a.nvec, vbeg, my_slot, static_cast<uint4*>(a.xe), lane);
    }
}

// MOE_HEAD=separate keeps route as its own launch (for measurement).
static bool head_separate() {
    static int v = -1;
    if (v < 0) {
        const char* e = getenv("MOE_HEAD");
        v = (e && strcmp(e, "separate") == 0) ? 1 : 0;
    }
    return v == 1;
}

bool head_fusable(const moe_config& c, int T) {
    return !head_separate() && plan_dispatch_fusable(c, T) && T <= kHeadClusterMax * kPlanWarps * kHeadTokensPerWarp;
}

template <int NPER, int kGate, bool kFp8>
static cudaError_t launch_head_t(const HeadArgs& a, int E, int grid_cap, cudaStream_t st) {
    constexpr bool kGrouped = kGate != MOE_GATE_SOFTMAX;
    auto kern = route_plan_dispatch_kernel<NPER, kGate, kFp8>;
    const int kk = a.k + a.S;
    const size_t smem = (size_t)a.T * a.k * 4 + 2 * (size_t)a.T * kk * 4 + (kGrouped ? (size_t)kPlanWarps * E * 4 : 0);
    cudaError_t e = ensure_max_dynamic_smem(
        kern, (int)(kPlanEntriesPerChunk * 4 * 3 + kPlanWarps * kMaxExperts * 4));
    if (e != cudaSuccess) return e;
    int cs = kHeadClusterMax;
    while (cs > 1 && cs > grid_cap) cs >>= 1;
    const int items = a.T * ((a.nvec + 127) / 128);
    int ctas = (items + kPlanWarps - 1) / kPlanWarps;
    if (ctas > grid_cap) ctas = grid_cap;
    int clusters = ctas / cs;
    if (clusters < 1) clusters = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(clusters * cs));
    cfg.blockDim = dim3(kPlanThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int kGate, bool kFp8>
static cudaError_t launch_head_g(const HeadArgs& a, int E, int grid_cap, cudaStream_t st) {
    if (E <= 32) return launch_head_t<1, kGate, kFp8>(a, E, grid_cap, st);
    if (E <= 64) return launch_head_t<2, kGate, kFp8>(a, E, grid_cap, st);
    if (E <= 128) return launch_head_t<4, kGate, kFp8>(a, E, grid_cap, st);
    if (E <= 256) return launch_head_t<8, kGate, kFp8>(a, E, grid_cap, st);
    return launch_head_t<16, kGate, kFp8>(a, E, grid_cap, st);
}

cudaError_t launch_route_plan_dispatch(const moe_config& c, int T, const float* logits, const float* bias,
                                       int32_t* ids, float* w, int capacity, int align, int32_t* counts,
                                       int32_t* offsets, int32_t* slot_of, int32_t* err, const void* x, void* xe,
                                       float* xe_scale, int64_t scale_cs, int grid_cap, cudaStream_t st) {
    const bool fp8 = c.dtype == MOE_FP8_E4M3;
    HeadArgs a{};
    a.T = T;
    a.E = c.num_experts;
    a.k = c.top_k;
    a.S = c.num_shared;
    a.n_group = c.n_group;
    a.topk_group = c.topk_group;
    a.renorm = c.renormalize;
    a.scale = c.routed_scale;
    a.logits = logits;
    a.bias = bias;
    a.ids = ids;
    a.w = w;
    a.capacity = capacity;
    a.align = align;
    a.counts = counts;
    a.offsets = offsets;
    a.slot_of = slot_of;
    a.err = err;
    a.x = static_cast<const uint4*>(x);
    a.xe = xe;
    a.xe_scale = xe_scale;
    a.scale_cs = scale_cs;
    a.nvec = fp8 ? c.hidden / 8 : c.hidden * elt_bytes(c.dtype) / 16;
    if (c.gate == MOE_GATE_SIGMOID_GROUPED)
        return fp8 ? launch_head_g<MOE_GATE_SIGMOID_GROUPED, true>(a, a.E, grid_cap, st)
                   : launch_head_g<MOE_GATE_SIGMOID_GROUPED, false>(a, a.E, grid_cap, st);
    if (c.gate == MOE_GATE_SQRT_SOFTPLUS)
        return fp8 ? launch_head_g<MOE_GATE_SQRT_SOFTPLUS, true>(a, a.E, grid_cap, st)
                   : launch_head_g<MOE_GATE_SQRT_SOFTPLUS, false>(a, a.E, grid_cap, st);
    return fp8 ? launch_head_g<MOE_GATE_SOFTMAX, true>(a, a.E, grid_cap, st)
               : launch_head_g<MOE_GATE_SOFTMAX, false>(a, a.E, grid_cap, st);
}

}  // namespace moe
