// Device code of the plan shared by the plan kernels (plan.cu) and the fused
// plan + dispatch kernel (head.cu).
#pragma once

#include "common.cuh"

namespace moe {

constexpr int kPlanThreads = 256;
constexpr int kPlanWarps = kPlanThreads / 32;
constexpr int kPlanEntriesPerChunk = 4096;       // a batch up to this many entries is one chunk
constexpr int kPlanEntriesPerChunkMulti = 1024;  // larger batches: chunks of about this many

// Expert of entry (t, j); -1 for a routed id outside [0, E).  kSharedIds: ids are in
// shared memory (the fused head), else in global memory.
template <bool kSharedIds = false>
__device__ __forceinline__ int entry_expert(const int32_t* ids, int t, int j, int k, int E) {
    if (j >= k) return E + (j - k);
    int e = kSharedIds ? ids[(size_t)t * k + j] : __ldg(ids + (size_t)t * k + j);
    return (e >= 0 && e < E) ? e : -1;
}

// Exclusive block scan of v[0..n) in shared memory (n <= kMaxExperts); writes
// out[0..n], out[n] = total.  All threads of the block must call it.
__device__ __forceinline__ void block_exclusive_scan(const int* v, int* out, int n, int* warp_tot) {
    const int per = (n + blockDim.x - 1) / blockDim.x;  // <= 2 for n <= 512
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int local[4];
    int s = 0;
    for (int i = 0; i < per; ++i) {
        int idx = threadIdx.x * per + i;
        local[i] = idx < n ? v[idx] : 0;
        s += local[i];
    }
    int incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (threadIdx.x == 0) {
        int acc = 0;
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
            int t = warp_tot[w];
            warp_tot[w] = acc;
            acc += t;
        }
        warp_tot[blockDim.x >> 5] = acc;
    }
    __syncthreads();
    int run = warp_tot[warp] + incl - s;
    for (int i = 0; i < per; ++i) {
        int idx = threadIdx.x * per + i;
        if (idx < n) out[idx] = run;
        run += local[i];
    }
    if (threadIdx.x == 0) out[n] = warp_tot[blockDim.x >> 5];
    __syncthreads();
}

// One CTA's share of the plan: chunk `chunk` of `nchunks` (ids in shared memory when
// kSharedIds).  chunk_e: shared memory for
// the chunk's entry experts.  write_outputs: this CTA stores counts / offsets (chunk 0),
// slot_of and token_of; slot_sm (may be null): the chunk's slots are also kept in
// shared memory (the fused plan + dispatch kernel, where every CTA plans the whole batch
// and only CTA 0 writes).  Every thread of the CTA must call it.
template <bool kSharedIds = false>
__device__ __forceinline__ void plan_assign_cta(int T, int k, int S, int E, int tpc, int nchunks, int chunk,
                                                int capacity, int align, const int32_t* __restrict__ ids,
                                                const int32_t* __restrict__ hist, int32_t* __restrict__ counts,
                                                int32_t* __restrict__ offsets, int32_t* __restrict__ slot_of,
                                                int32_t* __restrict__ token_of, int32_t* err, int* chunk_e,
                                                int* slot_sm, bool write_outputs) {
    __shared__ int total[kMaxExperts];
    __shared__ int base[kMaxExperts];
    __shared__ int padded[kMaxExperts];
    __shared__ int off[kMaxExperts + 1];
    __shared__ int wcnt[kPlanWarps][kMaxExperts];
    __shared__ int warp_tot[kPlanWarps + 1];

    const int NE = E + S, kk = k + S;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int t0 = chunk * tpc;
    const int t1 = min(T, t0 + tpc);
    const int n = (t1 - t0) * kk;

    for (int i = threadIdx.x; i < kPlanWarps * NE; i += blockDim.x) (&wcnt[0][0])[(i / NE) * kMaxExperts + i % NE] = 0;
    if (nchunks == 1) {
        for (int e = threadIdx.x; e < NE; e += blockDim.x) {
            total[e] = 0;
            base[e] = 0;
        }
        __syncthreads();
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            int e = entry_expert<kSharedIds>(ids, t0 + i / kk, i % kk, k, E);
            chunk_e[i] = e;
            if (e >= 0) atomicAdd(&total[e], 1);
        }
    } else {
        for (int i = threadIdx.x; i < n; i += blockDim.x)
            chunk_e[i] = entry_expert<kSharedIds>(ids, t0 + i / kk, i % kk, k, E);
        for (int e = threadIdx.x; e < NE; e += blockDim.x) {
            int tot = 0, bef = 0;
            for (int c = 0; c < nchunks; ++c) {
                int v = hist[(size_t)c * NE + e];
                tot += v;
                if (c < chunk) bef += v;
            }
            total[e] = tot;
            base[e] = bef;
        }
    }
    __syncthreads();

    // offsets: exact mode scans the aligned counts; capacity mode is static
    if (capacity > 0) {
        for (int e = threadIdx.x; e <= NE; e += blockDim.x) off[e] = e * capacity;
        __syncthreads();
    } else {
        for (int e = threadIdx.x; e < NE; e += blockDim.x) padded[e] = (total[e] + align - 1) / align * align;
        __syncthreads();
        block_exclusive_scan(padded, off, NE, warp_tot);
    }
    if (chunk == 0 && write_outputs) {
        for (int e = threadIdx.x; e < NE; e += blockDim.x)
            counts[e] = capacity > 0 ? min(total[e], capacity) : total[e];
        for (int e = threadIdx.x; e <= NE; e += blockDim.x) offsets[e] = off[e];
    }
    // padding rows are marked -1 (when the caller wants token_of): one warp per expert,
    // experts dealt round-robin over the CTAs' warps
    if (token_of && write_outputs) {
        for (int e = chunk * kPlanWarps + warp; e < NE; e += nchunks * kPlanWarps) {
            const int used = capacity > 0 ? min(total[e], capacity) : total[e];
            for (int r = off[e] + used + lane; r < off[e + 1]; r += 32) token_of[r] = -1;
        }
    }
    for (int e = threadIdx.x; e < NE; e += blockDim.x) base[e] += off[e];
    __syncthreads();

    for (int it = 0; it < n; it += kPlanThreads) {
        const int i = it + threadIdx.x;
        const bool in = i < n;
        const int t = t0 + (in ? i / kk : 0), j = in ? i % kk : 0;
        int e = in ? chunk_e[i] : -1;
        const bool good = in && e >= 0;
        if (in && !good) {
            if (write_outputs) slot_of[(size_t)t * kk + j] = -1;
            if (slot_sm) slot_sm[i] = -1;
            set_err(err, MOE_ERR_BAD_INDEX);
        }
        const int key = good ? e : (0x40000000 | threadIdx.x);
        const uint32_t peers = __match_any_sync(0xffffffffu, key);
        const int rank_w = __popc(peers & lanemask_lt());
        const bool leader = (__ffs(peers) - 1) == lane;
        if (good && leader) wcnt[warp][e] = __popc(peers);
        __syncthreads();
        if (good) {
            int pre = 0;
            for (int w = 0; w < warp; ++w) pre += wcnt[w][e];
            const int row = base[e] + pre + rank_w;
            int slot = row;
            if (capacity > 0 && row - off[e] >= capacity) {
                slot = -1;
                set_err(err, MOE_ERR_CAPACITY);
            } else if (token_of && write_outputs) {
                token_of[row] = t;
            }
            if (write_outputs) slot_of[(size_t)t * kk + j] = slot;
            if (slot_sm) slot_sm[i] = slot;
        }
        __syncthreads();
        if (good && leader) {  // several warps may hold the same expert: add atomically
            atomicAdd(&base[e], __popc(peers));
            wcnt[warp][e] = 0;
        }
        __syncthreads();
    }
}

}  // namespace moe
