// Portable grouped expert FFN on the CUDA cores (fp32 FMA).  It serves the fp32
// layers (the tensor-core path covers bf16 and fp8) and is a second, independent
// GPU implementation the tensor-core kernels can be compared against.
//
// Two persistent kernels: gate/up GEMM with the SwiGLU epilogue (h in the
// activation type, fp8 with 1x128 scales), then the down GEMM.  Tiles are
// (expert, 32-row block, 128-column block); every CTA derives the tile list from
// the device counts/offsets, so no host synchronisation is needed.
#include "common.cuh"
#include "kernels.h"

namespace moe {

namespace {

constexpr int BM = 32, BN = 128, BK = 32, NT = 256;

// tstart[0..NE]: exclusive scan of the tile counts, run by one warp.
__device__ void scan_tiles_warp(int NE, const int32_t* counts, const int32_t* offsets, int64_t max_rows,
                                int ntn, int bm, int* tstart, int32_t* err) {
    const int lane = threadIdx.x & 31;
    const int per = (NE + 31) / 32;
    int s = 0;
    int vals[16];
    for (int i = 0; i < per; ++i) {
        int e = lane * per + i;
        int v = 0;
        if (e < NE) {
            int cnt = __ldg(counts + e);
            int64_t end = (int64_t)__ldg(offsets + e) + cnt;
            if (cnt < 0 || end > max_rows) {
                set_err(err, MOE_ERR_BAD_INDEX);
                cnt = 0;
            }
            v = (cnt + bm - 1) / bm * ntn;
        }
        vals[i] = v;
        s += v;
    }
    int incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    int run = incl - s;
    for (int i = 0; i < per; ++i) {
        int e = lane * per + i;
        if (e < NE) tstart[e] = run;
        run += vals[i];
    }
    if (lane == 31) tstart[NE] = incl;
}

// largest e with tstart[e] <= tile (tiles of empty experts are skipped naturally)
__device__ __forceinline__ int find_expert(const int* tstart, int NE, int tile) {
    int lo = 0, hi = NE - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (tstart[mid] <= tile) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

template <int DT>
// (fp8 scales: row-major [rows][K/128] when sc_cs == 0, else column-major with that stride)
__device__ __forceinline__ float load_act(const void* p, const float* sc, int64_t row, int kx, int K,
                                          int64_t sc_cs = 0) {
    if (DT == MOE_F32) return static_cast<const float*>(p)[row * K + kx];
    if (DT == MOE_BF16) return bf16_bits_to_f(static_cast<const uint16_t*>(p)[row * K + kx]);
    return e4m3_to_f(static_cast<const uint8_t*>(p)[row * K + kx]) *
           sc[sc_cs ? (kx / kQG) * sc_cs + row : row * (K / kQG) + kx / kQG];
}

// weight element (e, n, kx) of a [NE][N][K] tensor with 128x128 block scales
template <int DT>
__device__ __forceinline__ float load_w(const void* p, const float* sc, int e, int n, int kx, int N, int K) {
    const size_t idx = ((size_t)e * N + n) * K + kx;
    if (DT == MOE_F32) return static_cast<const float*>(p)[idx];
    if (DT == MOE_BF16) return bf16_bits_to_f(static_cast<const uint16_t*>(p)[idx]);
    return e4m3_to_f(static_cast<const uint8_t*>(p)[idx]) *
           sc[((size_t)e * (N / kQG) + n / kQG) * (K / kQG) + kx / kQG];
}

template <int DT>
__global__ void __launch_bounds__(NT) ffn_simt_up_kernel(int NE, int H, int I, const int32_t* counts,
                                                         const int32_t* offsets, int64_t max_rows,
                                                         const void* xe, const float* xe_scale, int64_t xs_cs,
                                                         const void* w13, const float* w13_scale,
                                                         void* h, float* h_scale, int32_t* err, int reverse) {
    __shared__ int tstart[kMaxExperts + 1];
    __shared__ float As[BK][BM];
    __shared__ float Bg[BK][BN + 4];
    __shared__ float Bu[BK][BN + 4];
    const int ntn = (I + BN - 1) / BN;
    if (threadIdx.x < 32) scan_tiles_warp(NE, counts, offsets, max_rows, ntn, BM, tstart, err);
    __syncthreads();
    const int total = tstart[NE];
    const int ty = threadIdx.x >> 5, tx = threadIdx.x & 31;
    for (int lin = blockIdx.x; lin < total; lin += gridDim.x) {
        const int tile = reverse ? total - 1 - lin : lin;
        const int e = find_expert(tstart, NE, tile);
        const int local = tile - tstart[e];
        const int mt = local / ntn, nt = local % ntn;
        const int cnt = counts[e];
        const int64_t row0 = (int64_t)offsets[e] + (int64_t)mt * BM;
        const int rows_here = min(BM, cnt - mt * BM);
        const int n0 = nt * BN;
        float ag[4][4], au[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) ag[i][j] = au[i][j] = 0.0f;
        for (int k0 = 0; k0 < H; k0 += BK) {
            {
                const int r = threadIdx.x / 8, kq = (threadIdx.x % 8) * 4;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int kx = k0 + kq + q;
                    As[kq + q][r] = (r < rows_here && kx < H) ? load_act<DT>(xe, xe_scale, row0 + r, kx, H, xs_cs) : 0.0f;
                }
            }
            {
                const int n = threadIdx.x / 2, kq = (threadIdx.x % 2) * 16;
#pragma unroll 4
                for (int q = 0; q < 16; ++q) {
                    const int kx = k0 + kq + q;
                    const bool ok = (n0 + n < I) && kx < H;
                    Bg[kq + q][n] = ok ? load_w<DT>(w13, w13_scale, e, n0 + n, kx, 2 * I, H) : 0.0f;
                    Bu[kq + q][n] = ok ? load_w<DT>(w13, w13_scale, e, I + n0 + n, kx, 2 * I, H) : 0.0f;
                }
            }
            __syncthreads();
#pragma unroll 8
            for (int kx = 0; kx < BK; ++kx) {
                float a[4], bg[4], bu[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) a[i] = As[kx][ty * 4 + i];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    bg[j] = Bg[kx][tx * 4 + j];
                    bu[j] = Bu[kx][tx * 4 + j];
                }
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        ag[i][j] = fmaf(a[i], bg[j], ag[i][j]);
                        au[i][j] = fmaf(a[i], bu[j], au[i][j]);
                    }
            }
            __syncthreads();
        }
        // SwiGLU epilogue
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = ty * 4 + i;
            float hv[4];
            float amax = 0.0f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float g = ag[i][j];
                hv[j] = g / (1.0f + expf(-g)) * au[i][j];
                if (n0 + tx * 4 + j < I) amax = fmaxf(amax, fabsf(hv[j]));
            }
            if (DT == MOE_FP8_E4M3) {
                amax = warp_max(amax);  // the warp holds this row's 128 columns
                const int s = fp8_scale_exp(amax);
                if (r < rows_here) {
                    uint8_t* hq = static_cast<uint8_t*>(h) + (row0 + r) * I + n0 + tx * 4;
                    const Pow2Factors f = pow2_neg(s);
                    const uint16_t p0 = f2_to_e4m3x2(scale_by(hv[0], f), scale_by(hv[1], f));
                    const uint16_t p1 = f2_to_e4m3x2(scale_by(hv[2], f), scale_by(hv[3], f));
                    *reinterpret_cast<uint32_t*>(hq) = (uint32_t)p0 | ((uint32_t)p1 << 16);
                    if (tx == 0) h_scale[(row0 + r) * (I / kQG) + nt] = mul_pow2(1.0f, s);
                }
            } else if (r < rows_here) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int n = n0 + tx * 4 + j;
                    if (n >= I) continue;
                    if (DT == MOE_F32) static_cast<float*>(h)[(row0 + r) * I + n] = hv[j];
                    else static_cast<uint16_t*>(h)[(row0 + r) * I + n] = f_to_bf16_bits(hv[j]);
                }
            }
        }
    }
}

template <int DT>
__global__ void __launch_bounds__(NT) ffn_simt_down_kernel(int NE, int H, int I, const int32_t* counts,
                                                           const int32_t* offsets, int64_t max_rows,
                                                           const void* h, const float* h_scale,
                                                           const void* w2, const float* w2_scale, void* ye,
                                                           int reverse) {
    __shared__ int tstart[kMaxExperts + 1];
    __shared__ float As[BK][BM];
    __shared__ float Bs[BK][BN + 4];
    const int ntn = (H + BN - 1) / BN;
    if (threadIdx.x < 32) scan_tiles_warp(NE, counts, offsets, max_rows, ntn, BM, tstart, nullptr);
    __syncthreads();
    const int total = tstart[NE];
    const int ty = threadIdx.x >> 5, tx = threadIdx.x & 31;
    for (int lin = blockIdx.x; lin < total; lin += gridDim.x) {
        const int tile = reverse ? total - 1 - lin : lin;
        const int e = find_expert(tstart, NE, tile);
        const int local = tile - tstart[e];
        const int mt = local / ntn, nt = local % ntn;
        const int cnt = counts[e];
        const int64_t row0 = (int64_t)offsets[e] + (int64_t)mt * BM;
        const int rows_here = min(BM, cnt - mt * BM);
        const int n0 = nt * BN;
        float acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
        for (int k0 = 0; k0 < I; k0 += BK) {
            {
                const int r = threadIdx.x / 8, kq = (threadIdx.x % 8) * 4;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int kx = k0 + kq + q;
                    As[kq + q][r] = (r < rows_here && kx < I) ? load_act<DT>(h, h_scale, row0 + r, kx, I) : 0.0f;
                }
            }
            {
                const int n = threadIdx.x / 2, kq = (threadIdx.x % 2) * 16;
#pragma unroll 4
                for (int q = 0; q < 16; ++q) {
                    const int kx = k0 + kq + q;
                    Bs[kq + q][n] = (n0 + n < H && kx < I) ? load_w<DT>(w2, w2_scale, e, n0 + n, kx, H, I) : 0.0f;
                }
            }
            __syncthreads();
#pragma unroll 8
            for (int kx = 0; kx < BK; ++kx) {
                float a[4], b[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) a[i] = As[kx][ty * 4 + i];
#pragma unroll
                for (int j = 0; j < 4; ++j) b[j] = Bs[kx][tx * 4 + j];
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
            }
            __syncthreads();
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = ty * 4 + i;
            if (r >= rows_here) continue;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int n = n0 + tx * 4 + j;
                if (n >= H) continue;
                if (DT == MOE_F32) static_cast<float*>(ye)[(row0 + r) * H + n] = acc[i][j];
                else static_cast<uint16_t*>(ye)[(row0 + r) * H + n] = f_to_bf16_bits(acc[i][j]);
            }
        }
    }
}

template <int DT>
cudaError_t launch_simt_dt(const moe_config& c, const FfnArgs& a, int grid, cudaStream_t st) {
    const int NE = c.num_experts + c.num_shared;
    const int H = c.hidden, I = c.inter;
    void* h = a.ws;
    float* h_scale = nullptr;
    if (DT == MOE_FP8_E4M3)
        h_scale = reinterpret_cast<float*>(static_cast<char*>(a.ws) + align_up((size_t)a.max_rows * I, 256));
    ffn_simt_up_kernel<DT><<<grid, NT, 0, st>>>(NE, H, I, a.counts, a.offsets, a.max_rows, a.xe, a.xe_scale,
                                                a.xs_cs, a.w13, a.w13_scale, h, h_scale, a.err, a.reverse);
    ffn_simt_down_kernel<DT><<<grid, NT, 0, st>>>(NE, H, I, a.counts, a.offsets, a.max_rows, h, h_scale, a.w2,
                                                  a.w2_scale, a.ye, a.reverse);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ffn_simt(const moe_config& c, const FfnArgs& a, int grid_cap, cudaStream_t st) {
    int grid = device_info().num_sms * 4;
    if (grid > grid_cap) grid = grid_cap;
    if (c.dtype == MOE_F32) return launch_simt_dt<MOE_F32>(c, a, grid, st);
    if (c.dtype == MOE_BF16) return launch_simt_dt<MOE_BF16>(c, a, grid, st);
    return launch_simt_dt<MOE_FP8_E4M3>(c, a, grid, st);
}

}  // namespace moe
