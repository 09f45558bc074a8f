// moe_combine kernels.
//
// Staged (the default; three CTAs per SM): a CTA takes a contiguous range of (token,
// column chunk) units.
// Its producer warp copies the chunk of each of the token's k+S expert-output rows (and
// of the residual row, if any) from HBM into a shared-memory stage with bulk async
// copies (cp.async.bulk, one contiguous request of up to 4 KB per row) while the
// consumer warps reduce earlier stages: y = resid + sum_j w_j * ye_j in fp32 in the
// fixed (j, then s) order, one 16-byte output vector per thread, stored once.  Each
// row chunk is one long DRAM request and several stages are in flight per SM.
//
// Register (one warp per (token, slice of 64 vectors), two vectors a lane): used when
// a stage of the token's rows does not fit the shared-memory budget (k+S above 31).
// Both forms run the same FMA chain, so their results are identical bit for bit.
//
// No atomics: every output element is written by exactly one thread.
#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

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

// ------------------------------------------------------------------ staged form
constexpr int kStageConsumerWarps = 8;
constexpr int kStageThreads = 32 * (1 + kStageConsumerWarps);
constexpr int kStageMaxStages = 16;
// The producer keeps the slots and weights of the next kTokPrefetch tokens in flight
// into a ring of kTokRing shared-memory entries (cp.async: a register never waits on
// an outstanding load, so one token's metadata latency is paid once, not per token).
constexpr int kTokPrefetch = 6;
constexpr int kTokRing = 8;

struct CombineStageMeta {
    float w[32];     // weight of entry j (1 for shared experts)
    uint32_t mask;   // bit j: entry j placed (its row is in the stage)
    int32_t t, cb, len;
};

struct TokenMeta {
    int32_t slot[32];
    float w[32];
};

// barriers (512 bytes), per-stage metadata, the token ring, then the stages
constexpr int kCombineHeaderBytes =
    512 + kStageMaxStages * (int)sizeof(CombineStageMeta) + kTokRing * (int)sizeof(TokenMeta);

struct CombineParams {
    int T, k, kk, rowb, chunk, nchunk, stages, has_res;
    long long units;
    const uint8_t* ye;
    const float* w;
    const int32_t* slot_of;
    uint8_t* y;
    const uint8_t* resid;
    int32_t* err;
    long long inject_ns;
};

template <bool kF32>
__global__ void __launch_bounds__(kStageThreads, 1) combine_staged_kernel(const CombineParams p) {
    extern __shared__ __align__(128) uint8_t csm[];
    uint64_t* full = reinterpret_cast<uint64_t*>(csm);
    uint64_t* empty = full + kStageMaxStages;
    uint64_t* never = empty + kStageMaxStages;
    volatile int* abort = reinterpret_cast<volatile int*>(never + 1);
    CombineStageMeta* meta = reinterpret_cast<CombineStageMeta*>(csm + 512);
    TokenMeta* ring = reinterpret_cast<TokenMeta*>(csm + 512 + kStageMaxStages * sizeof(CombineStageMeta));
    uint8_t* data = csm + kCombineHeaderBytes;
    const int stage_bytes = (p.kk + p.has_res) * p.chunk;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < p.stages; ++i) {
            tc::mbar_init(&full[i], 1);
            tc::mbar_init(&empty[i], kStageConsumerWarps);
        }
        tc::mbar_init(never, 1);
        *abort = 0;
        tc::fence_barrier_init();
    }
    __syncthreads();
    pdl_begin();
    if (p.inject_ns > 0) {  // failure-path test hook: no copy has been issued yet
        if (threadIdx.x == 0) {
            tc::wait_on_nothing(never, (uint64_t)p.inject_ns);
            set_err(p.err, MOE_ERR_TIMEOUT);
        }
        return;
    }
    const long long u0 = (long long)blockIdx.x * p.units / gridDim.x;
    const long long u1 = (long long)(blockIdx.x + 1) * p.units / gridDim.x;
    if (u0 >= u1) return;
    if (warp == 0) {
        // producer
        const int t_first = (int)(u0 / p.nchunk), t_last = (int)((u1 - 1) / p.nchunk);
#pragma unroll
        for (int r = 0; r < kTokRing; ++r) {  // entries no token fills: not placed, weight 1
            ring[r].slot[lane] = -1;
            ring[r].w[lane] = 1.0f;
        }
        __syncwarp();
        auto prefetch = [&](int tt) {  // one cp.async group per token, empty past the range
            if (tt <= t_last) {
                TokenMeta& e = ring[tt % kTokRing];
                if (lane < p.kk) tc::cp_async_4(&e.slot[lane], p.slot_of + (size_t)tt * p.kk + lane);
                if (lane < p.k) tc::cp_async_4(&e.w[lane], p.w + (size_t)tt * p.k + lane);
            }
            tc::cp_async_commit();
        };
#pragma unroll 1
        for (int d = 0; d < kTokPrefetch; ++d) prefetch(t_first + d);
        int cur = t_first - 1;
        int slot = -1;
        float wv = 1.0f;
        long long i = 0;
        bool ok = true;
        for (long long u = u0; u < u1; ++u, ++i) {
            const int t = (int)(u / p.nchunk);
            const int c = (int)(u - (long long)t * p.nchunk);
            if (t != cur) {  // next token: its metadata group is the oldest of kTokPrefetch
                tc::cp_async_wait<kTokPrefetch - 1>();
                const TokenMeta& e = ring[t % kTokRing];
                slot = e.slot[lane];
                wv = e.w[lane];
                prefetch(t + kTokPrefetch);  // into the entry of token t + kTokPrefetch - kTokRing (done)
                cur = t;
            }
            const int s = (int)(i % p.stages);
            const uint32_t n = (uint32_t)(i / p.stages);
            if (n > 0 && !tc::mbar_wait(&empty[s], (n - 1) & 1u, abort)) {
                ok = false;
                break;
            }
            const int cb = c * p.chunk;
            const int len = min(p.chunk, p.rowb - cb);
            const uint32_t valid = __ballot_sync(0xffffffffu, slot >= 0);
            CombineStageMeta& m = meta[s];
            m.w[lane] = wv;
            if (lane == 0) {
                m.mask = valid;
                m.t = t;
                m.cb = cb;
                m.len = len;
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive_expect_tx(&full[s], (uint32_t)((__popc(valid) + p.has_res) * len));
            __syncwarp();
            uint8_t* st = data + (size_t)s * stage_bytes;
            if (slot >= 0) tc::bulk_load(st + lane * p.chunk, p.ye + (size_t)slot * p.rowb + cb, (uint32_t)len, &full[s]);
            if (p.has_res && lane == 0)
                tc::bulk_load(st + p.kk * p.chunk, p.resid + (size_t)t * p.rowb + cb, (uint32_t)len, &full[s]);
        }
        tc::cp_async_wait<0>();
        if (!ok) {
            if (lane == 0) {
                set_err(p.err, MOE_ERR_TIMEOUT);
                *abort = 1;
                // copies still in flight land before the CTA leaves: the last issue of each stage
                for (long long q = i - 1; q >= 0 && q >= i - p.stages; --q)
                    tc::mbar_wait_bounded(&full[q % p.stages], (uint32_t)(q / p.stages) & 1u);
            }
        }
        return;
    }
    // consumers
    constexpr int kPer = kF32 ? 4 : 8;
    const int ct = threadIdx.x - 32;
    long long i = 0;
    for (long long u = u0; u < u1; ++u, ++i) {
        const int s = (int)(i % p.stages);
        const uint32_t n = (uint32_t)(i / p.stages);
        if (!tc::mbar_wait(&full[s], n & 1u, abort)) {
            if (lane == 0) {
                set_err(p.err, MOE_ERR_TIMEOUT);
                *abort = 1;
            }
            return;
        }
        const CombineStageMeta& m = meta[s];
        const uint32_t mask = m.mask;
        const int nv = m.len >> 4;
        const uint8_t* st = data + (size_t)s * stage_bytes;
        uint4* yrow = reinterpret_cast<uint4*>(p.y + (size_t)m.t * p.rowb + m.cb);
        for (int v = ct; v < nv; v += 32 * kStageConsumerWarps) {
            float acc[kPer];
#pragma unroll
            for (int e = 0; e < kPer; ++e) acc[e] = 0.0f;
            if (p.has_res) unpack16<kF32>(reinterpret_cast<const uint4*>(st + p.kk * p.chunk)[v], acc);
            for (int j = 0; j < p.kk; ++j) {
                if (!((mask >> j) & 1u)) continue;
                float f[kPer];
                unpack16<kF32>(reinterpret_cast<const uint4*>(st + j * p.chunk)[v], f);
                const float wj = m.w[j];
#pragma unroll
                for (int e = 0; e < kPer; ++e) acc[e] = fmaf(wj, f[e], acc[e]);
            }
            uint4 out;
            if (kF32)
                out = make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]), __float_as_uint(acc[2]),
                                 __float_as_uint(acc[3]));
            else
                out = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                                 pack_bf16x2(acc[6], acc[7]));
            yrow[v] = out;
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&empty[s]);
    }
}

// Three staged CTAs per SM (each ~74 KB of shared memory: two or more stages of up to
// 4 KB per row) keep more requests in flight than one CTA with the whole shared memory:
// one CTA's producer, consumers and their barrier hand-offs leave gaps that the other
// two fill.  Measured on GB300 against one and two CTAs per SM and 1-4 KB chunks.
constexpr int kStageCtasPerSm = 3;
constexpr int kStageSmemBudget = 233472 / kStageCtasPerSm - 2048;
constexpr int kStageChunkCap = 4096;


int combine_ctas_per_sm() { return kStageCtasPerSm; }

cudaError_t launch_combine(const moe_config& c, int T, const void* ye, const float* w,
                           const int32_t* slot_of, void* y, int grid_cap, cudaStream_t st, const void* resid,
                           int32_t* err) {
    if (T <= 0) return cudaSuccess;
    const int kk = c.top_k + c.num_shared;
    const int rowb = c.hidden * io_bytes(c.dtype);
    const int nvec = rowb / 16;
    const int has_res = resid != nullptr;
    // chunk: the row split into equal pieces of at most kStageChunkCap bytes (multiples
    // of 16), so that a stage of (k+S+resid) chunks fits a few times into the budget
    int nchunk = (rowb + kStageChunkCap - 1) / kStageChunkCap;
    int chunk = (((rowb + nchunk - 1) / nchunk) + 15) & ~15;
    const int meta_bytes = kCombineHeaderBytes;
    int stages = 0;
    if (kk <= 31 || (kk == 32 && !has_res)) {
        while ((long)(kk + has_res) * chunk * 2 > kStageSmemBudget - meta_bytes && chunk > 256) {
            ++nchunk;
            chunk = (((rowb + nchunk - 1) / nchunk) + 15) & ~15;
        }
        stages = (kStageSmemBudget - meta_bytes) / ((kk + has_res) * chunk);
        if (stages > kStageMaxStages) stages = kStageMaxStages;
    }
    if (stages >= 2) {
        nchunk = (rowb + chunk - 1) / chunk;
        CombineParams p;
        p.T = T;
        p.k = c.top_k;
        p.kk = kk;
        p.rowb = rowb;
        p.chunk = chunk;
        p.nchunk = nchunk;
        p.stages = stages;
        p.has_res = has_res;
        p.units = (long long)T * nchunk;
        p.ye = static_cast<const uint8_t*>(ye);
        p.w = w;
        p.slot_of = slot_of;
        p.y = static_cast<uint8_t*>(y);
        p.resid = static_cast<const uint8_t*>(resid);
        p.err = err ? err : comm_error_word();
        if (!p.err) return cudaErrorInvalidValue;
        p.inject_ns = wait_injection_ns();
        const int smem = meta_bytes + stages * (kk + has_res) * chunk;
        long grid = (long)device_info().num_sms * kStageCtasPerSm;
        if (grid > grid_cap) grid = grid_cap;
        if (grid > p.units) grid = (int)p.units;
        auto kern = c.dtype == MOE_F32 ? combine_staged_kernel<true> : combine_staged_kernel<false>;
        cudaError_t e = ensure_max_dynamic_smem(kern, smem);
        if (e != cudaSuccess) return e;
        return launch_pdl(kern, (int)grid, kStageThreads, (size_t)smem, st, p);
    }
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
