// Grouped expert FFN on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Two persistent, warp-specialised kernels, one CTA per SM:
//   up   : acc[128 x 256] = xe[rows] . [W13 gate rows n0..n0+127 | up rows I+n0..]^T,
//          epilogue h = silu(g) * u -> bf16 h[rows][n0..n0+127]
//   down : acc[128 x 256] = h[rows] . W2[e][n0..n0+255]^T, epilogue -> bf16 ye
// A tile = 128 rows of one expert's segment (rows past the segment are computed and
// discarded), B tile = 256 weight rows; k-blocks of 64 bf16 (one 128-byte swizzle
// row).  Tiles (expert, n-block, m-block) are derived on the device from counts and
// offsets, so no host synchronisation is needed and the launch is graph-capturable.
//
// Roles (192 threads):
//   warp 0 (one lane)  TMA producer: 4-stage ring of {A 16 KB, B 32 KB}
//   warp 1 (one lane)  MMA issuer: tcgen05.mma M=128 N=256 K=16 into a TMEM
//                      accumulator, double buffered (2 x 256 of 512 columns)
//   warps 2..5         epilogue: tcgen05.ld of the warp's 32 TMEM lanes (one row per
//                      thread), activation, stores of the row's columns
// Every wait is bounded: after kWaitTimeoutNs a role raises a CTA-wide abort flag,
// stores MOE_ERR_TIMEOUT, drains its own outstanding copies / MMAs, and the CTA frees
// its TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdlib.h>
#include <string.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kBN = 256;
constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr int kABytes = kBM * kBK * 2;
constexpr int kBBytes = kBN * kBK * 2;
constexpr int kStageBytes = kABytes + kBBytes;
constexpr uint32_t kTmemCols = 2 * kBN;
constexpr int kNumBars = 2 * kStages + 2 + 2 + 1;  // full, empty, tmem full, tmem empty, drain
constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + kNumBars * 8 + 16 +
                              3 * (kMaxExperts + 1) * sizeof(int) + 512 * sizeof(float) + 256 * sizeof(int);
constexpr int kF8Threads = 320;  // warp 0 TMA, warp 1 MMA, warps 2..9 promotion + epilogue
constexpr int kF8BK = 128;       // e4m3 elements per k-block = one 128-wide scale block

// A tiles are loaded with the smallest box of 16 / 32 / 64 / 128 rows that covers the
// tile's rows: at decode an expert has a handful of rows, and fetching 128 would
// re-read other experts' rows (and, once the weight stream has evicted them from L2,
// from DRAM).  The MMA still reads 128 rows of the stage; the rows past the box hold
// stale data whose results land in accumulator rows that are never stored.
constexpr int kNumABoxes = 4;
__host__ __device__ constexpr int a_box_rows(int i) { return 16 << i; }

struct TcParams {
    CUtensorMap tmA[kNumABoxes];  // activations [max_rows][K], box heights 16, 32, 64, 128
    CUtensorMap tmB;              // weights [NE * NB][K]
    const int32_t* counts;
    const int32_t* offsets;
    int NE, K, kblocks;
    int NB;   // weight rows per expert
    int ntn;  // n-blocks per expert
    int I, H;
    int64_t max_rows;
    void* out;
    int32_t* err;
    int reverse;
    const float* a_scale;  // fp8: [max_rows][K/128] row-group scales of A
    const float* b_scale;  // fp8: [NE][NB/128][K/128] block scales of B
    float* out_scale;      // fp8 up: [max_rows][I/128] scales of the quantised h
    int dense_rows;        // counts == nullptr: one dense matrix of this many rows
    const void* resid;     // bf16 down: added to the product before rounding ([rows][H])
};

struct Smem {
    uint8_t* stages;
    uint64_t* full;
    uint64_t* empty;
    uint64_t* tfull;
    uint64_t* tempty;
    uint64_t* drain;
    uint32_t* tmem_base;
    volatile int* abort;
    int* tstart;
    int* cnt;
    int* off;
    float* xval;         // fp8 up epilogue: [2 parities][2 halves][128 rows] partial amax
    volatile int* xseq;  // [2 halves][128 rows] tile sequence number of the value
};

__device__ __forceinline__ Smem carve(uint8_t* raw) {
    Smem s;
    uint8_t* p = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    s.stages = p;
    p += (size_t)kStages * kStageBytes;
    s.full = reinterpret_cast<uint64_t*>(p);
    s.empty = s.full + kStages;
    s.tfull = s.empty + kStages;
    s.tempty = s.tfull + 2;
    s.drain = s.tempty + 2;
    s.tmem_base = reinterpret_cast<uint32_t*>(s.drain + 1);
    s.abort = reinterpret_cast<volatile int*>(s.tmem_base + 1);
    s.tstart = reinterpret_cast<int*>(s.tmem_base + 4);
    s.cnt = s.tstart + (kMaxExperts + 1);
    s.off = s.cnt + (kMaxExperts + 1);
    s.xval = reinterpret_cast<float*>(s.off + (kMaxExperts + 1));
    s.xseq = reinterpret_cast<volatile int*>(s.xval + 512);
    return s;
}

__device__ __forceinline__ void fail(const Smem& s, int32_t* err) {
    set_err(err, MOE_ERR_TIMEOUT);
    *s.abort = 1;
}

struct Tile {
    int e, mt, nt, rows;
    int row0;
};

__device__ __forceinline__ Tile decode_tile(const TcParams& p, const Smem& s, int total, int lin) {
    const int tile = p.reverse ? total - 1 - lin : lin;
    int lo = 0, hi = p.NE - 1;
    while (lo < hi) {  // largest e with tstart[e] <= tile
        const int mid = (lo + hi + 1) >> 1;
        if (s.tstart[mid] <= tile) lo = mid;
        else hi = mid - 1;
    }
    Tile t;
    t.e = lo;
    const int local = tile - s.tstart[lo];
    const int cnt = s.cnt[lo];
    const int mtiles = (cnt + kBM - 1) / kBM;
    t.nt = local / mtiles;  // n-major within an expert: consecutive CTAs share B
    t.mt = local % mtiles;
    t.row0 = s.off[lo] + t.mt * kBM;
    t.rows = min(kBM, cnt - t.mt * kBM);
    return t;
}

// One warp: copies counts/offsets into shared memory and scans the tile counts.
__device__ void scan_tiles(const TcParams& p, const Smem& s) {
    const int lane = threadIdx.x & 31;
    const int per = (p.NE + 31) / 32;
    int vals[16];
    int sum = 0;
    for (int i = 0; i < per; ++i) {
        const int e = lane * per + i;
        int v = 0;
        if (e < p.NE) {
            int cnt = p.counts ? __ldg(p.counts + e) : p.dense_rows;
            const int off = p.counts ? __ldg(p.offsets + e) : 0;
            if (cnt < 0 || off < 0 || (int64_t)off + cnt > p.max_rows) {
                set_err(p.err, MOE_ERR_BAD_INDEX);
                cnt = 0;
            }
            s.cnt[e] = cnt;
            s.off[e] = off;
            v = (cnt + kBM - 1) / kBM * p.ntn;
        }
        vals[i] = v;
        sum += v;
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    int run = incl - sum;
    for (int i = 0; i < per; ++i) {
        const int e = lane * per + i;
        if (e < p.NE) s.tstart[e] = run;
        run += vals[i];
    }
    if (lane == 31) s.tstart[p.NE] = incl;
}

// kKElems: elements per k-block (one 128-byte swizzle row): 64 bf16 or 128 e4m3.
template <bool kUp, int kKElems>
__device__ void producer(const TcParams& p, const Smem& s, int total) {
    int stage = 0;
    uint32_t phase = 0;
    uint32_t pending = 0, pend_par = 0;  // per stage: a load in flight, and its phase parity
    bool ok = true;
    for (int lin = blockIdx.x; lin < total && ok; lin += gridDim.x) {
        const Tile t = decode_tile(p, s, total, lin);
        int b0, b1;
        if (kUp) {
            b0 = t.e * p.NB + t.nt * 128;
            b1 = t.e * p.NB + p.I + t.nt * 128;
        } else {
            b0 = t.e * p.NB + t.nt * kBN;
            b1 = b0 + 128;
        }
        int abox = 0;
        while (abox < kNumABoxes - 1 && a_box_rows(abox) < t.rows) ++abox;
        const int abox_rows = a_box_rows(abox);
        for (int kb = 0; kb < p.kblocks; ++kb) {
            if (!tc::mbar_wait(&s.empty[stage], phase ^ 1u, s.abort)) {
                ok = false;
                break;
            }
            uint8_t* a = s.stages + (size_t)stage * kStageBytes;
            uint8_t* b = a + kABytes;
            tc::mbar_arrive_expect_tx(&s.full[stage], (uint32_t)(abox_rows * 128 + kBBytes));
            tc::tma_load_2d(a, &p.tmA[abox], &s.full[stage], kb * kKElems, t.row0);
            tc::tma_load_2d(b, &p.tmB, &s.full[stage], kb * kKElems, b0);
            tc::tma_load_2d(b + kBBytes / 2, &p.tmB, &s.full[stage], kb * kKElems, b1);
            pending |= 1u << stage;
            pend_par = (pend_par & ~(1u << stage)) | (phase << stage);
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    if (!ok) {
        fail(s, p.err);
        // let the copies already issued land before the CTA exits
        for (int st = 0; st < kStages; ++st)
            if ((pending >> st) & 1u) {
                const uint64_t t0 = tc::globaltimer();
                while (!tc::mbar_try_wait(&s.full[st], (pend_par >> st) & 1u) &&
                       tc::globaltimer() - t0 < tc::kWaitTimeoutNs) {
                }
            }
    }
}

__device__ void mma_issuer(const TcParams& p, const Smem& s, int total, uint32_t tmem_base) {
    int stage = 0;
    uint32_t phase = 0;
    int buf = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    constexpr uint32_t idesc = tc::idesc_bf16_f32(kBM, kBN);
    for (int lin = blockIdx.x; lin < total && ok; lin += gridDim.x) {
        if (!tc::mbar_wait(&s.tempty[buf], acc_phase ^ 1u, s.abort)) {
            ok = false;
            break;
        }
        tc::tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(buf * kBN);
        for (int kb = 0; kb < p.kblocks; ++kb) {
            if (!tc::mbar_wait(&s.full[stage], phase, s.abort)) {
                ok = false;
                break;
            }
            tc::tc_fence_after();
            const uint32_t a_addr = tc::smem_u32(s.stages + (size_t)stage * kStageBytes);
            const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
                tc::mma_bf16(d, tc::desc_sw128_kmajor(a_addr + kk * 32), tc::desc_sw128_kmajor(b_addr + kk * 32),
                             idesc, (kb | kk) != 0 ? 1u : 0u);
            }
            tc::mma_commit(&s.empty[stage]);  // frees the smem stage once these MMAs finish
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok) break;
        tc::mma_commit(&s.tfull[buf]);  // accumulator ready for the epilogue
        buf ^= 1;
        if (buf == 0) acc_phase ^= 1u;
    }
    if (!ok) fail(s, p.err);
    // drain: every MMA issued above has completed before TMEM is released
    tc::mma_commit(s.drain);
    const uint64_t t0 = tc::globaltimer();
    while (!tc::mbar_try_wait(s.drain, 0) && tc::globaltimer() - t0 < tc::kWaitTimeoutNs) {
    }
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

template <bool kUp>
__device__ void epilogue(const TcParams& p, const Smem& s, int total, uint32_t tmem_base) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;
    int buf = 0;
    uint32_t acc_phase = 0;
    for (int lin = blockIdx.x; lin < total; lin += gridDim.x) {
        const Tile t = decode_tile(p, s, total, lin);
        if (!tc::mbar_wait(&s.tfull[buf], acc_phase, s.abort)) {
            fail(s, p.err);
            break;
        }
        tc::tc_fence_after();
        const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * kBN);
        const bool valid = r < t.rows;
        const int64_t row = (int64_t)t.row0 + r;
        if (kUp) {
            uint16_t* hrow = static_cast<uint16_t*>(p.out) + row * p.I + t.nt * 128;
#pragma unroll 1
            for (int c = 0; c < 128; c += 32) {
                uint32_t g[32], u[32];
                tc::tmem_ld32(tb + c, g);
                tc::tmem_ld32(tb + 128 + c, u);
                tc::tmem_wait_ld();
                if (valid) {
                    uint4 v[4];
                    uint32_t* w = reinterpret_cast<uint32_t*>(v);
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        w[i] = pack_bf16x2(silu_mul(__uint_as_float(g[2 * i]), __uint_as_float(u[2 * i])),
                                           silu_mul(__uint_as_float(g[2 * i + 1]), __uint_as_float(u[2 * i + 1])));
                    uint4* dst = reinterpret_cast<uint4*>(hrow + c);
#pragma unroll
                    for (int i = 0; i < 4; ++i) dst[i] = v[i];
                }
            }
        } else {
            uint16_t* yrow = static_cast<uint16_t*>(p.out) + row * p.H + t.nt * kBN;
            const uint16_t* rrow = p.resid ? static_cast<const uint16_t*>(p.resid) + row * p.H + t.nt * kBN : nullptr;
#pragma unroll 1
            for (int c = 0; c < kBN; c += 32) {
                uint32_t a[32];
                tc::tmem_ld32(tb + c, a);
                tc::tmem_wait_ld();
                if (valid) {
                    if (rrow) {  // residual: out = resid + product, one rounding
                        const uint4* rr = reinterpret_cast<const uint4*>(rrow + c);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const uint4 q = rr[i];
                            const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                a[8 * i + 2 * j] = __float_as_uint(__uint_as_float(a[8 * i + 2 * j]) +
                                                                   bf16_bits_to_f((uint16_t)(wd[j] & 0xffffu)));
                                a[8 * i + 2 * j + 1] = __float_as_uint(__uint_as_float(a[8 * i + 2 * j + 1]) +
                                                                       bf16_bits_to_f((uint16_t)(wd[j] >> 16)));
                            }
                        }
                    }
                    uint4 v[4];
                    uint32_t* w = reinterpret_cast<uint32_t*>(v);
#pragma unroll
                    for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(__uint_as_float(a[2 * i]), __uint_as_float(a[2 * i + 1]));
                    uint4* dst = reinterpret_cast<uint4*>(yrow + c);
#pragma unroll
                    for (int i = 0; i < 4; ++i) dst[i] = v[i];
                }
            }
        }
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&s.tempty[buf]);
        buf ^= 1;
        if (buf == 0) acc_phase ^= 1u;
    }
}

template <bool kUp>
__global__ void __launch_bounds__(kThreads, 1) ffn_tc_bf16_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    const Smem s = carve(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            tc::mbar_init(&s.full[i], 1);
            tc::mbar_init(&s.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&s.tfull[i], 1);
            tc::mbar_init(&s.tempty[i], 4);
        }
        tc::mbar_init(s.drain, 1);
        *s.abort = 0;
        tc::fence_barrier_init();
        for (int i = 0; i < kNumABoxes; ++i) tc::prefetch_tmap(&p.tmA[i]);
        tc::prefetch_tmap(&p.tmB);
    }
    if (warp == 1) {
        tc::tmem_alloc(s.tmem_base, kTmemCols);
        tc::tmem_relinquish();
    }
    // Everything above overlaps the previous kernel's tail.  Nothing produced upstream
    // (counts, offsets, xe, h) is read before this wait: with a chain of such
    // launches an earlier kernel than the immediate predecessor may still be running.
    tc::pdl_launch_dependents();
    tc::pdl_wait();
    if (warp == 2) scan_tiles(p, s);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem_base = *s.tmem_base;
    const int total = s.tstart[p.NE];

    if (warp == 0) {
        if (lane == 0) producer<kUp, kBK>(p, s, total);
    } else if (warp == 1) {
        if (lane == 0) mma_issuer(p, s, total, tmem_base);
    } else {
        epilogue<kUp>(p, s, total, tmem_base);
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ---------------------------------------------------------------- FP8 (e4m3) kernels
//
// Same tiles and TMA ring as the bf16 kernels, with k-blocks of 128 e4m3 elements (one
// 128-byte row), which is exactly one 128-wide scale block.  Each k-block's four
// kind::f8f6f4 MMAs (K = 32) write a fresh partial product into one of two TMEM
// buffers; eight promotion warps read it back, multiply by a_scale[row][kb] *
// b_scale[n-block][kb] (both powers of two) and accumulate in fp32 registers (each
// thread: one row, 128 of the 256 columns), while the MMAs of the next k-block fill
// the other buffer.  The up kernel's epilogue forms h = silu(g) * u, finds the 1x128
// group amax of its row with its partner thread (the other half of the columns)
// through shared memory, and stores h as e4m3 with its power-of-two scale; the down
// kernel stores ye as bf16.

__device__ void mma_issuer_f8(const TcParams& p, const Smem& s, int total, uint32_t tmem_base) {
    int stage = 0;
    uint32_t phase = 0;
    int pb = 0;
    uint32_t pph = 0;
    bool ok = true;
    constexpr uint32_t idesc = tc::idesc_e4m3_f32(kBM, kBN);
    for (int lin = blockIdx.x; lin < total && ok; lin += gridDim.x) {
        for (int kb = 0; kb < p.kblocks; ++kb) {
            if (!tc::mbar_wait(&s.tempty[pb], pph ^ 1u, s.abort) || !tc::mbar_wait(&s.full[stage], phase, s.abort)) {
                ok = false;
                break;
            }
            tc::tc_fence_after();
            const uint32_t d = tmem_base + (uint32_t)(pb * kBN);
            const uint32_t a_addr = tc::smem_u32(s.stages + (size_t)stage * kStageBytes);
            const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
            for (int kk = 0; kk < kF8BK / 32; ++kk)
                tc::mma_e4m3(d, tc::desc_sw128_kmajor(a_addr + kk * 32), tc::desc_sw128_kmajor(b_addr + kk * 32),
                             idesc, kk != 0 ? 1u : 0u);
            tc::mma_commit(&s.empty[stage]);
            tc::mma_commit(&s.tfull[pb]);
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
            }
            pb ^= 1;
            if (pb == 0) pph ^= 1u;
        }
    }
    if (!ok) fail(s, p.err);
    tc::mma_commit(s.drain);
    const uint64_t t0 = tc::globaltimer();
    while (!tc::mbar_try_wait(s.drain, 0) && tc::globaltimer() - t0 < tc::kWaitTimeoutNs) {
    }
}

// acc += partial * sc for 32 columns of this thread's TMEM lane, as packed two-wide
// fp32 FMAs (acc[i] holds columns 2i, 2i+1).  Loaded 16 columns at a time: with 10
// warps per SM a thread has at most 168 registers, 128 of which are accumulators.
__device__ __forceinline__ void promote32(uint32_t taddr, float sc, float2* acc) {
    const float2 s2 = make_float2(sc, sc);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t v[16];
        tc::tmem_ld16(taddr + 16 * h, v);
        tc::tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 8; ++i)
            acc[8 * h + i] =
                __ffma2_rn(make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])), s2, acc[8 * h + i]);
    }
}

template <bool kUp>
__device__ void epilogue_f8(const TcParams& p, const Smem& s, int total, uint32_t tmem_base) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3;           // TMEM lane quarter
    const int half = (warp - 2) >> 2;  // which half of the 256 columns
    const int r = q * 32 + lane;
    const int ksb = p.K / kF8BK;      // scale blocks along K
    int pb = 0;
    uint32_t pph = 0;
    int seq = 0;
    bool ok = true;
    for (int lin = blockIdx.x; lin < total && ok; lin += gridDim.x) {
        const Tile t = decode_tile(p, s, total, lin);
        const int64_t row = (int64_t)t.row0 + r;
        const bool in_rows = row < p.max_rows;
        const float* asc = p.a_scale + (in_rows ? row : 0) * ksb;
        const float* bsc = p.b_scale + (size_t)t.e * (p.NB / kF8BK) * ksb;
        const int nb0 = kUp ? t.nt : 2 * t.nt + half;  // gate (up kernel) or output block
        const int nb1 = kUp ? p.I / kF8BK + t.nt : nb0;  // up block (up kernel)
        float2 acc[64];  // up: gate columns in acc[0..31], up columns in acc[32..63]
#pragma unroll
        for (int i = 0; i < 64; ++i) acc[i] = make_float2(0.0f, 0.0f);
        // a warp whose 32 rows are all past the tile's rows has nothing to promote (at
        // decode most tiles hold fewer than 32 rows)
        const bool busy = q * 32 < t.rows;
        const float* bs0 = bsc + (size_t)nb0 * ksb;
        const float* bs1 = bsc + (size_t)nb1 * ksb;
        // scales of the next k-block are loaded while the current one is promoted
        float sa_n = (busy && in_rows) ? __ldg(asc) : 0.0f;
        float sb0_n = busy ? __ldg(bs0) : 0.0f;
        float sb1_n = (busy && kUp) ? __ldg(bs1) : 0.0f;
        for (int kb = 0; kb < p.kblocks; ++kb) {
            const float s0 = sa_n * sb0_n, s1 = sa_n * sb1_n;
            if (busy && kb + 1 < p.kblocks) {
                sa_n = in_rows ? __ldg(asc + kb + 1) : 0.0f;
                sb0_n = __ldg(bs0 + kb + 1);
                if (kUp) sb1_n = __ldg(bs1 + kb + 1);
            }
            if (!tc::mbar_wait(&s.tfull[pb], pph, s.abort)) {
                ok = false;
                break;
            }
            tc::tc_fence_after();
            const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(pb * kBN);
            if (busy) {
                if (kUp) {
                    promote32(tb + 64 * half, s0, acc);
                    promote32(tb + 64 * half + 32, s0, acc + 16);
                    promote32(tb + 128 + 64 * half, s1, acc + 32);
                    promote32(tb + 128 + 64 * half + 32, s1, acc + 48);
                } else {
#pragma unroll
                    for (int c = 0; c < 4; ++c) promote32(tb + 128 * half + 32 * c, s0, acc + 16 * c);
                }
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&s.tempty[pb]);
            pb ^= 1;
            if (pb == 0) pph ^= 1u;
        }
        if (!ok) break;
        const bool valid = r < t.rows;
        if (kUp) {
            // h for this thread's 64 columns (written over the gate pairs)
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float g0 = acc[i].x, g1 = acc[i].y;
                acc[i].x = g0 / (1.0f + expf(-g0)) * acc[32 + i].x;
                acc[i].y = g1 / (1.0f + expf(-g1)) * acc[32 + i].y;
                amax = fmaxf(amax, fmaxf(fabsf(acc[i].x), fabsf(acc[i].y)));
            }
            // the row's other 64 columns belong to the partner thread: exchange amax
            ++seq;
            const int par = seq & 1;
            s.xval[(par * 2 + half) * 128 + r] = amax;
            __threadfence_block();
            s.xseq[half * 128 + r] = seq;
            const uint64_t t0 = tc::globaltimer();
            while (s.xseq[(1 - half) * 128 + r] < seq) {
                if (*s.abort || tc::globaltimer() - t0 > tc::kWaitTimeoutNs) {
                    ok = false;
                    break;
                }
            }
            if (!ok) break;
            __threadfence_block();
            amax = fmaxf(amax, s.xval[(par * 2 + 1 - half) * 128 + r]);
            const int se = fp8_scale_exp(amax);
            if (valid) {
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const uint16_t lo = f2_to_e4m3x2(scalbnf(acc[2 * i].x, -se), scalbnf(acc[2 * i].y, -se));
                    const uint16_t hi = f2_to_e4m3x2(scalbnf(acc[2 * i + 1].x, -se), scalbnf(acc[2 * i + 1].y, -se));
                    w[i] = (uint32_t)lo | ((uint32_t)hi << 16);
                }
                uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) + row * p.I + t.nt * 128 + 64 * half);
#pragma unroll
                for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                if (half == 0) p.out_scale[row * (p.I / kF8BK) + t.nt] = scalbnf(1.0f, se);
            }
        } else if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + row * p.H + t.nt * kBN + 128 * half);
#pragma unroll
            for (int i = 0; i < 16; ++i)
                dst[i] = make_uint4(pack_bf16x2(acc[4 * i].x, acc[4 * i].y), pack_bf16x2(acc[4 * i + 1].x, acc[4 * i + 1].y),
                                    pack_bf16x2(acc[4 * i + 2].x, acc[4 * i + 2].y),
                                    pack_bf16x2(acc[4 * i + 3].x, acc[4 * i + 3].y));
        }
    }
    if (!ok) fail(s, p.err);
}

template <bool kUp>
__global__ void __launch_bounds__(kF8Threads, 1) ffn_tc_fp8_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    const Smem s = carve(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            tc::mbar_init(&s.full[i], 1);
            tc::mbar_init(&s.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&s.tfull[i], 1);
            tc::mbar_init(&s.tempty[i], 8);
        }
        tc::mbar_init(s.drain, 1);
        *s.abort = 0;
        tc::fence_barrier_init();
        for (int i = 0; i < kNumABoxes; ++i) tc::prefetch_tmap(&p.tmA[i]);
        tc::prefetch_tmap(&p.tmB);
    }
    for (int i = threadIdx.x; i < 256; i += blockDim.x) s.xseq[i] = 0;
    if (warp == 1) {
        tc::tmem_alloc(s.tmem_base, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::pdl_launch_dependents();
    tc::pdl_wait();  // see the bf16 kernel: nothing from upstream is read before this
    if (warp == 2) scan_tiles(p, s);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem_base = *s.tmem_base;
    const int total = s.tstart[p.NE];

    if (warp == 0) {
        if (lane == 0) producer<kUp, kF8BK>(p, s, total);
    } else if (warp == 1) {
        if (lane == 0) mma_issuer_f8(p, s, total, tmem_base);
    } else {
        epilogue_f8<kUp>(p, s, total, tmem_base);
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

// 2-D K-major matrix [rows][inner] with the 128-byte swizzle and a box of one
// 128-byte row (64 bf16 or 128 e4m3) by box_rows rows.
bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, bool fp8, int box_rows = 128) {
    auto enc = encode_fn();
    if (!enc) return false;
    const uint64_t elt = fp8 ? 1 : 2;
    cuuint64_t dims[2] = {inner, rows};
    cuuint64_t strides[1] = {inner * elt};
    cuuint32_t box[2] = {(cuuint32_t)(128 / elt), (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    return enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
               dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kUp, bool kFp8>
cudaError_t launch_one(const TcParams& p, int grid, cudaStream_t st) {
    static int configured_dev = -1;
    const int dev = device_info().device;
    auto kern = kFp8 ? ffn_tc_fp8_kernel<kUp> : ffn_tc_bf16_kernel<kUp>;
    if (configured_dev != dev) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        configured_dev = dev;
    }
    // programmatic dependent launch: this kernel's prologue may overlap the tail of the
    // previous kernel on the stream; it waits (griddepcontrol.wait) before reading
    // anything that kernel wrote
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kFp8 ? kF8Threads : kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

bool ffn_tc_supported(const moe_config& c) {
    const DeviceInfo& d = device_info();
    return (c.dtype == MOE_BF16 || c.dtype == MOE_FP8_E4M3) && d.cc_major == 10 && c.hidden % kBN == 0 &&
           c.inter % 128 == 0 && d.smem_optin >= kSmemBytes && encode_fn() != nullptr;
}

cudaError_t launch_ffn_tc(const moe_config& c, const FfnArgs& a, int grid_cap, cudaStream_t st) {
    const int NE = c.num_experts + c.num_shared;
    const int H = c.hidden, I = c.inter;
    const bool fp8 = c.dtype == MOE_FP8_E4M3;
    int grid = device_info().num_sms;
    if (grid > grid_cap) grid = grid_cap;
    if (grid < 1) grid = 1;
    void* h = a.ws;
    float* h_scale =
        fp8 ? reinterpret_cast<float*>(static_cast<char*>(a.ws) + align_up((size_t)a.max_rows * I, 256)) : nullptr;
    const int kelems = fp8 ? kF8BK : kBK;
    TcParams up{};
    for (int i = 0; i < kNumABoxes; ++i)
        if (!make_map(&up.tmA[i], a.xe, (uint64_t)H, (uint64_t)a.max_rows, fp8, a_box_rows(i)))
            return cudaErrorInvalidValue;
    if (!make_map(&up.tmB, a.w13, (uint64_t)H, (uint64_t)NE * 2 * I, fp8)) return cudaErrorInvalidValue;
    up.counts = a.counts;
    up.offsets = a.offsets;
    up.NE = NE;
    up.K = H;
    up.kblocks = H / kelems;
    up.NB = 2 * I;
    up.ntn = I / 128;
    up.I = I;
    up.H = H;
    up.max_rows = a.max_rows;
    up.out = h;
    up.err = a.err;
    up.reverse = a.reverse;
    up.a_scale = a.xe_scale;
    up.b_scale = a.w13_scale;
    up.out_scale = h_scale;
    TcParams dn = up;
    for (int i = 0; i < kNumABoxes; ++i)
        if (!make_map(&dn.tmA[i], h, (uint64_t)I, (uint64_t)a.max_rows, fp8, a_box_rows(i)))
            return cudaErrorInvalidValue;
    if (!make_map(&dn.tmB, a.w2, (uint64_t)I, (uint64_t)NE * H, fp8)) return cudaErrorInvalidValue;
    dn.K = I;
    dn.kblocks = I / kelems;
    dn.NB = H;
    dn.ntn = H / kBN;
    dn.out = a.ye;
    dn.a_scale = h_scale;
    dn.b_scale = a.w2_scale;
    dn.out_scale = nullptr;
    cudaError_t e = fp8 ? launch_one<true, true>(up, grid, st) : launch_one<true, false>(up, grid, st);
    if (e != cudaSuccess) return e;
    return fp8 ? launch_one<false, true>(dn, grid, st) : launch_one<false, false>(dn, grid, st);
}

bool standin_tc_supported(const moe_config& c) {
    const DeviceInfo& d = device_info();
    return c.dtype != MOE_F32 && d.cc_major == 10 && c.hidden % kBN == 0 && d.smem_optin >= kSmemBytes &&
           encode_fn() != nullptr;
}

// out[rows][H] = x + x . Wa^T (bf16, fp32 accumulation): the down kernel on one dense
// "expert" with a residual epilogue.
cudaError_t launch_standin(const moe_config& c, int rows, const void* x, const void* wa, void* out, int grid_cap,
                           cudaStream_t st) {
    if (rows <= 0) return cudaSuccess;
    const int H = c.hidden;
    int grid = device_info().num_sms;
    if (grid > grid_cap) grid = grid_cap;
    if (grid < 1) grid = 1;
    TcParams p{};
    for (int i = 0; i < kNumABoxes; ++i)
        if (!make_map(&p.tmA[i], x, (uint64_t)H, (uint64_t)rows, false, a_box_rows(i))) return cudaErrorInvalidValue;
    if (!make_map(&p.tmB, wa, (uint64_t)H, (uint64_t)H, false)) return cudaErrorInvalidValue;
    p.counts = nullptr;
    p.offsets = nullptr;
    p.dense_rows = rows;
    p.NE = 1;
    p.K = H;
    p.kblocks = H / kBK;
    p.NB = H;
    p.ntn = H / kBN;
    p.I = H;
    p.H = H;
    p.max_rows = rows;
    p.out = out;
    p.resid = x;
    return launch_one<false, false>(p, grid, st);
}

}  // namespace moe
