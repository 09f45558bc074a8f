// Grouped expert FFN on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Two persistent, warp-specialised kernels per layer type, one CTA per SM (the bf16
// kernels are described here, the block-scaled FP8 ones with their code below):
//   up   : acc[128 x 256] = xe[rows] . [W13 gate rows n0..n0+127 | up rows I+n0..]^T,
//          epilogue h = silu(g) * u -> bf16 h[rows][n0..n0+127]
//   down : acc[128 x 256] = h[rows] . W2[e][n0..n0+255]^T, epilogue -> bf16 ye
// A tile = 128 rows of one expert's segment (rows past the segment are computed and
// discarded), B tile = 256 weight rows, one TMA box (W13 is addressed as a 3-D tensor
// so that the gate and up n-blocks come in one box); k-blocks of 64 bf16 (one 128-byte
// swizzle row).  Tiles (expert, n-block, m-block) are derived on the device from counts
// and offsets, so no host synchronisation is needed and the launch is graph-capturable.
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
constexpr int kF8BK = 128;  // e4m3 elements per k-block = one 128-wide scale block

// FP8 tile geometry: 128 x 256 tiles (up: gate 128 | up 128 columns, so that a whole
// 1x128 group of h is formed in one tile; down: two 128-row n-blocks of W2), one
// accumulator (the scale slots take the rest of TMEM), 4 stages of 48 KB.  Scale factors
// of each stage are staged in shared memory (kSfStageBytes) and copied into TMEM slot
// kSfCol + 16 * stage.  (128 x 128 down tiles with two accumulators and 6 stages of
// 32 KB measured slower.)
template <bool kUp>
struct F8 {
    static constexpr int N = 256;
    static constexpr int AccBufs = 1;
    static constexpr int Stages = 4;
    static constexpr int StageBytes = kBM * kF8BK + N * kF8BK;
};
constexpr int kSfCol = 256;
constexpr int kSfStageBytes = 1536;  // A scales, B scales of rows 0-127, of rows 128-255 (512 B each)
constexpr int kMaxStages = 6;
constexpr int kNumBars = 2 * kMaxStages + 2 + 2 + 2;  // full, empty, tmem full, tmem empty, drain, never
constexpr int kOutSlotBytes = 2048;  // per epilogue warp: 32 rows x 64 bytes of output staging
constexpr size_t kSmemTail = kNumBars * 8 + 16 + 3 * (kMaxExperts + 1) * sizeof(int) + 512 * sizeof(float) +
                             256 * sizeof(int) + 128 + 8 * kOutSlotBytes;
constexpr size_t smem_bytes(int stages, int stage_bytes, int sf_bytes) {
    return 1024 + (size_t)stages * (stage_bytes + sf_bytes) + kSmemTail;
}
constexpr size_t kSmemBytes = smem_bytes(kStages, kStageBytes, 0);
template <bool kUp>
constexpr size_t kF8SmemBytes = smem_bytes(F8<kUp>::Stages, F8<kUp>::StageBytes, kSfStageBytes);
constexpr int kF8Stagers = 1;    // scale-staging warps (round-robin over the steps; two measured slower)
constexpr int kF8Threads = 32 * (2 + kF8Stagers + 8);  // TMA, MMA, staging, 8 epilogue warps
constexpr int kF8FirstEpiWarp = 2 + kF8Stagers;
constexpr int kScGroup = 8;      // fp8: k-blocks of scales loaded at once

// A tiles are loaded with the smallest box of 16 / 32 / 64 / 128 rows that covers the
// tile's rows: at decode an expert has a handful of rows, and fetching 128 would
// re-read other experts' rows (and, once the weight stream has evicted them from L2,
// from DRAM).  The MMA still reads 128 rows of the stage; the rows past the box hold
// stale data whose results land in accumulator rows that are never stored.
constexpr int kNumABoxes = 4;
__host__ __device__ constexpr int a_box_rows(int i) { return 16 << i; }

struct TcParams {
    CUtensorMap tmA[kNumABoxes];  // activations [max_rows][K], box heights 16, 32, 64, 128
    CUtensorMap tmB;  // up: W13 viewed as [2 NE halves][I][K], box = one n-block of gate and of up rows;
                      // down: W2 [NE * H][K], box = the tile's N rows
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
    const float* a_scale;  // fp8: row-group scales of A, (row r, group g) at r * a_rs + g * a_cs
    int64_t a_rs, a_cs;
    const float* b_scale;  // fp8: [NE][NB/128][K/128] block scales of B
    float* out_scale;      // fp8 up: scales of the quantised h, column-major [I/128][max_rows]
    int dense_rows;        // counts == nullptr: one dense matrix of this many rows
    const void* resid;     // bf16 down: added to the product before rounding ([rows][H])
    int64_t inject_ns;     // test hook: > 0 = the producer's first wait runs out after this long
    // Fused gather (up kernels): A row r is row gather[r] (its token) of tmG -- x, or x_q
    // for fp8, with a box one row high -- fetched with tile::gather4; null: A rows are
    // rows of the dispatched xe (tmA).  zero / zero_n: the combine counters, cleared here.
    const int32_t* gather;
    CUtensorMap tmG;
    int32_t* zero;
    int64_t zero_n;
    // Fused combine (down kernels): see combine_slab.  comb_token: token of each row;
    // comb_slot / comb_w: slot_of [T][kk] / topk_w [T][k]; comb_y: y [T][H]; comb_cnt:
    // per (token, slab of comb_cols columns) arrival counters, zero at launch.
    const int32_t* comb_token;
    const int32_t* comb_slot;
    const float* comb_w;
    void* comb_y;
    int32_t* comb_cnt;
    int comb_k, comb_kk, comb_cols;
};

struct Smem {
    uint8_t* stages;
    uint8_t* sf;  // fp8: per stage, the scale factors staged for tcgen05.cp
    uint64_t* full;
    uint64_t* empty;
    uint64_t* tfull;
    uint64_t* tempty;
    uint64_t* drain;
    uint64_t* never;  // test hook: a barrier nothing ever arrives on
    uint32_t* tmem_base;
    volatile int* abort;
    int* tstart;
    int* cnt;
    int* off;
    float* xval;         // fp8 up epilogue: [2 parities][2 halves][128 rows] partial amax
    volatile int* xseq;  // [2 halves][128 rows] tile sequence number of the value
    uint4* oslot;        // epilogue output staging: kOutSlotBytes per epilogue warp
};

__device__ __forceinline__ Smem carve(uint8_t* raw, int stages, int stage_bytes, int sf_bytes) {
    Smem s;
    uint8_t* p = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    s.stages = p;
    p += (size_t)stages * stage_bytes;
    s.sf = p;
    p += (size_t)stages * sf_bytes;
    s.full = reinterpret_cast<uint64_t*>(p);
    s.empty = s.full + stages;
    s.tfull = s.empty + stages;
    s.tempty = s.tfull + 2;
    s.drain = s.tempty + 2;
    s.never = s.drain + 1;
    s.tmem_base = reinterpret_cast<uint32_t*>(s.drain + 2);
    s.abort = reinterpret_cast<volatile int*>(s.tmem_base + 1);
    s.tstart = reinterpret_cast<int*>(s.tmem_base + 4);
    s.cnt = s.tstart + (kMaxExperts + 1);
    s.off = s.cnt + (kMaxExperts + 1);
    s.xval = reinterpret_cast<float*>(s.off + (kMaxExperts + 1));
    s.xseq = reinterpret_cast<volatile int*>(s.xval + 512);
    s.oslot = reinterpret_cast<uint4*>((reinterpret_cast<uintptr_t>(s.xseq + 256) + 127) & ~uintptr_t(127));
    return s;
}

// Stores 64 bytes of each of a warp's 32 rows (lane i holds row i's words w[0..15],
// registers: every index is a constant after unrolling)
// through the warp's shared slot: written with the 16-byte chunks XOR-swizzled by row
// (no bank conflicts either way), read back so that lane l holds chunk l % 4 of row
// l / 4 + 8j, then stored 8 rows x 64 contiguous bytes per instruction instead of 32
// rows x 16 bytes.  base: the warp's first row's destination; pitch: bytes between
// rows; nrows: rows of the 32 to write.  Whole warp; 16-byte aligned base and pitch.
__device__ __forceinline__ void store_rows64(uint4* slot, const uint32_t* w, uint8_t* base, int64_t pitch,
                                             int nrows, int lane) {
    const int f = (lane >> 1) & 3;
#pragma unroll
    for (int i = 0; i < 4; ++i) slot[lane * 4 + (i ^ f)] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int rr = (lane >> 2) + 8 * j;
        const uint4 v = slot[rr * 4 + ((lane & 3) ^ ((rr >> 1) & 3))];
        if (rr < nrows) reinterpret_cast<uint4*>(base + rr * pitch)[lane & 3] = v;
    }
    __syncwarp();
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
// The failure-path test hook: the producer's first wait (on a barrier nothing arrives
// on) runs out before it issues any copy; the CTA reports MOE_ERR_TIMEOUT and every
// role leaves through its abort check.
__device__ __forceinline__ bool injected_failure(const TcParams& p, const Smem& s) {
    if (p.inject_ns <= 0) return false;
    tc::wait_on_nothing(s.never, (uint64_t)p.inject_ns);
    fail(s, p.err);
    return true;
}

template <bool kUp, int kKElems>
__device__ void producer(const TcParams& p, const Smem& s, int total) {
    if (injected_failure(p, s)) return;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t pending = 0, pend_par = 0;  // per stage: a load in flight, and its phase parity
    bool ok = true;
    for (int lin = blockIdx.x; lin < total && ok; lin += gridDim.x) {
        const Tile t = decode_tile(p, s, total, lin);
        const int b0 = t.e * p.NB + t.nt * kBN;  // down: first weight row of the tile
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
            if (kUp)  // gate rows n0..n0+127 then up rows I+n0.. in one box
                tc::tma_load_3d(b, &p.tmB, &s.full[stage], kb * kKElems, t.nt * 128, 2 * t.e);
            else
                tc::tma_load_2d(b, &p.tmB, &s.full[stage], kb * kKElems, b0);
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

// Clears the fused combine's counters (up kernel; the down kernel reads them only after
// its dependency wait, i.e. after this whole grid has finished).
__device__ __forceinline__ void zero_counters(const TcParams& p) {
    if (!p.zero) return;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < p.zero_n; i += (int64_t)gridDim.x * blockDim.x)
        p.zero[i] = 0;
}

// Fused gather (up kernels of both types: 48 KB stages of A 16 KB + B 32 KB), whole
// warp: lane 0 waits for the stage, announces its bytes and loads B; lane i gathers A
// rows 4i .. 4i+3 of the tile -- the rows of x (or x_q) of their tokens -- with one
// tile::gather4 copy into 512 bytes of the stage at 512 i.  Rows past the tile's count
// read token 0 (their results are never stored).
template <int kKElems>
__device__ void producer_gather(const TcParams& p, const Smem& s, int total) {
    const int lane = threadIdx.x & 31;
    int inj = lane == 0 ? (int)injected_failure(p, s) : 0;
    if (__shfl_sync(0xffffffffu, inj, 0)) return;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t pending = 0, pend_par = 0;  // lane 0: per stage, a load in flight and its parity
    bool ok = true;
    for (int lin = blockIdx.x; lin < total && ok; lin += gridDim.x) {
        const Tile t = decode_tile(p, s, total, lin);
        int tok[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = 4 * lane + i;
            const int v = r < t.rows ? __ldg(p.gather + t.row0 + r) : 0;
            tok[i] = v < 0 ? 0 : v;
        }
        const int ngather = (t.rows + 3) >> 2;
        const uint32_t tx = (uint32_t)(ngather * 512 + kBBytes);
        for (int kb = 0; kb < p.kblocks; ++kb) {
            int good = 1;
            if (lane == 0) good = tc::mbar_wait(&s.empty[stage], phase ^ 1u, s.abort);
            if (!__shfl_sync(0xffffffffu, good, 0)) {
                ok = false;
                break;
            }
            uint8_t* a = s.stages + (size_t)stage * kStageBytes;
            if (lane == 0) {
                tc::mbar_arrive_expect_tx(&s.full[stage], tx);
                tc::tma_load_3d(a + kABytes, &p.tmB, &s.full[stage], kb * kKElems, t.nt * 128, 2 * t.e);
                pending |= 1u << stage;
                pend_par = (pend_par & ~(1u << stage)) | (phase << stage);
            }
            __syncwarp();
            if (lane < ngather)
                tc::tma_gather4(a + 512 * lane, &p.tmG, &s.full[stage], kb * kKElems, tok[0], tok[1], tok[2], tok[3]);
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    if (!ok && lane == 0) {
        fail(s, p.err);
        for (int st = 0; st < kStages; ++st)  // every lane's copies complete on full[st]
            if ((pending >> st) & 1u) {
                const uint64_t t0 = tc::globaltimer();
                while (!tc::mbar_try_wait(&s.full[st], (pend_par >> st) & 1u) &&
                       tc::globaltimer() - t0 < tc::kWaitTimeoutNs) {
                }
            }
    }
}

// Fused combine, whole warp, after this thread's row has stored slab `slab` (p.comb_cols
// columns, the same for the warp) of its ye row: the row is counted for its token, and
// the last of the token's k+S rows to store the slab forms that slab of y[token] exactly
// as moe_combine does -- sum over j in order of w_j * ye[slot_of[token][j]] (weight 1
// for the shared experts) with fp32 fused multiply-adds, one rounding.  An entry the
// plan did not place never arrives, so its token's slab is left unwritten (the plan has
// raised MOE_ERR_CAPACITY / MOE_ERR_BAD_INDEX).
__device__ __forceinline__ void combine_slab(const TcParams& p, bool valid, int64_t row, int slab) {
    const int lane = threadIdx.x & 31;
    const int nslab = p.H / p.comb_cols;
    int tok = -1;
    bool last = false;
    if (valid) {
        tok = __ldg(p.comb_token + row);
        if (tok >= 0) {
            __threadfence();  // this row's slab is visible before it is counted
            last = atomicAdd(p.comb_cnt + (int64_t)tok * nslab + slab, 1) == p.comb_kk - 1;
        }
    }
    uint32_t m = __ballot_sync(0xffffffffu, last);
    if (!m) return;
    __threadfence();  // the other rows' slabs, counted before, are visible to the warp
    __syncwarp();
    const int kk = p.comb_kk, k = p.comb_k;
    const int nv = p.comb_cols / 8;  // 16-byte vectors of the slab (8 bf16 each)
    const int64_t hv = p.H / 8;
    const uint4* ye = static_cast<const uint4*>(p.out);
    while (m) {
        const int l = __ffs(m) - 1;
        m &= m - 1;
        const int t = __shfl_sync(0xffffffffu, tok, l);
        const int my_slot = lane < kk ? __ldg(p.comb_slot + (int64_t)t * kk + lane) : -1;
        const float my_w = lane < k ? __ldg(p.comb_w + (int64_t)t * k + lane) : 1.0f;
        const int64_t v = (int64_t)slab * nv + lane;
        const bool act = lane < nv;
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        for (int j0 = 0; j0 < kk; j0 += 8) {
            uint4 val[8];
            int r[8];
            float wj[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int j = j0 + u;
                r[u] = __shfl_sync(0xffffffffu, my_slot, j & 31);
                wj[u] = __shfl_sync(0xffffffffu, my_w, j & 31);
                if (j >= kk) r[u] = -1;
                if (r[u] >= 0 && act) val[u] = __ldcg(ye + (int64_t)r[u] * hv + v);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (r[u] < 0 || !act) continue;
                const uint32_t wd[4] = {val[u].x, val[u].y, val[u].z, val[u].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[2 * i] = fmaf(wj[u], bf16_bits_to_f((uint16_t)(wd[i] & 0xffffu)), acc[2 * i]);
                    acc[2 * i + 1] = fmaf(wj[u], bf16_bits_to_f((uint16_t)(wd[i] >> 16)), acc[2 * i + 1]);
                }
            }
        }
        if (act)
            static_cast<uint4*>(p.comb_y)[(int64_t)t * hv + v] =
                make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                           pack_bf16x2(acc[6], acc[7]));
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



template <bool kUp, bool kComb>
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
        // this warp's 32 rows: those of the tile, for the staged stores
        const int nrows = min(32, max(0, t.rows - q * 32));
        uint4* slot = s.oslot + (size_t)(warp - 2) * (kOutSlotBytes / 16);
        if (kUp) {
            uint8_t* hbase = reinterpret_cast<uint8_t*>(static_cast<uint16_t*>(p.out) +
                                                        ((int64_t)t.row0 + q * 32) * p.I + t.nt * 128);
#pragma unroll 1
            for (int c = 0; c < 128; c += 32) {
                uint32_t g[32], u[32];
                tc::tmem_ld32(tb + c, g);
                tc::tmem_ld32(tb + 128 + c, u);
                tc::tmem_wait_ld();
                if (nrows > 0) {
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        w[i] = pack_bf16x2(silu_mul_fast(__uint_as_float(g[2 * i]), __uint_as_float(u[2 * i])),
                                           silu_mul_fast(__uint_as_float(g[2 * i + 1]), __uint_as_float(u[2 * i + 1])));
                    store_rows64(slot, w, hbase + c * 2, (int64_t)p.I * 2, nrows, lane);
                }
            }
        } else {
            uint8_t* ybase = reinterpret_cast<uint8_t*>(static_cast<uint16_t*>(p.out) +
                                                        ((int64_t)t.row0 + q * 32) * p.H + t.nt * kBN);
            const uint16_t* rrow = p.resid ? static_cast<const uint16_t*>(p.resid) + row * p.H + t.nt * kBN : nullptr;
#pragma unroll 1
            for (int c = 0; c < kBN; c += 32) {
                uint32_t a[32];
                tc::tmem_ld32(tb + c, a);
                tc::tmem_wait_ld();
                if (valid && rrow) {  // residual: out = resid + product, one rounding
                    {
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
                }
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(__uint_as_float(a[2 * i]), __uint_as_float(a[2 * i + 1]));
                if (kComb) {  // each lane its own row: the fused combine fences and counts that row
                    if (valid) {
                        uint4* dst = reinterpret_cast<uint4*>(ybase + (int64_t)lane * p.H * 2 + c * 2);
#pragma unroll
                        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                    }
                } else if (nrows > 0) {
                    store_rows64(slot, w, ybase + c * 2, (int64_t)p.H * 2, nrows, lane);
                }
            }
        }
        tc::tc_fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&s.tempty[buf]);
        if (kComb) combine_slab(p, valid, row, t.nt);  // slabs of the tile's 256 columns
        buf ^= 1;
        if (buf == 0) acc_phase ^= 1u;
    }
}

// kComb (down kernels): the fused combine in the epilogue (a separate instantiation, so
// the plain kernels keep their registers)
template <bool kUp, bool kComb>
__global__ void __launch_bounds__(kThreads, 1) ffn_tc_bf16_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    const Smem s = carve(smem_raw, kStages, kStageBytes, 0);
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
        tc::mbar_init(s.never, 1);
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
    zero_counters(p);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem_base = *s.tmem_base;
    const int total = s.tstart[p.NE];

    if (warp == 0) {
        if (kUp && p.gather) producer_gather<kBK>(p, s, total);
        else if (lane == 0) producer<kUp, kBK>(p, s, total);
    } else if (warp == 1) {
        if (lane == 0) mma_issuer(p, s, total, tmem_base);
    } else {
        epilogue<kUp, kComb>(p, s, total, tmem_base);
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
// Same persistent tile loop and TMA ring as the bf16 kernels, with k-blocks of 128
// e4m3 elements (one 128-byte row), which is exactly one 128-wide scale block.  The
// scales are powers of two, so they are exact UE8M0 scale factors and the tensor core
// applies them itself: per k-block, four kind::mxf8f6f4 MMAs (K = 32) accumulate
// (A * a_scale[row][kb]) . (B * b_scale[n-block][kb])^T straight into a TMEM
// accumulator.  A staging warp writes each k-block's scale factors into shared memory
// next to the stage's operand tiles (the TMA producer only issues copies); the MMA
// thread copies them into the stage's TMEM scale slot (tcgen05.cp) right before the
// stage's MMAs, which execute in order after it.
// Epilogues: up forms h = silu(g) * u, finds the 1x128 group amax of its row with its
// partner thread (the other half of the columns) through shared memory and stores h
// as e4m3 with its power-of-two scale; down stores ye as bf16.  Each kernel's single
// accumulator is moved into registers and released before any of that arithmetic.

__device__ __forceinline__ uint32_t ue8m0x4(float pow2) {  // the biased exponent, in all four bytes
    const uint32_t e = (__float_as_uint(pow2) >> 23) & 0xffu;
    return e * 0x01010101u;
}

// One thread: the stage's TMA loads (the A box and the tile's 256-row B box).
template <bool kUp>
__device__ void producer_f8(const TcParams& p, const Smem& s, int total) {
    using G = F8<kUp>;
    if (injected_failure(p, s)) return;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t pending = 0, pend_par = 0;
    bool ok = true;
    for (int lin = blockIdx.x; lin < total && ok; lin += gridDim.x) {
        const Tile t = decode_tile(p, s, total, lin);
        const int b0 = t.e * p.NB + t.nt * G::N;  // down: first weight row of the tile
        int abox = 0;
        while (abox < kNumABoxes - 1 && a_box_rows(abox) < t.rows) ++abox;
        const uint32_t tx = (uint32_t)(a_box_rows(abox) * kF8BK + G::N * kF8BK);
        for (int kb = 0; kb < p.kblocks; ++kb) {
            if (!tc::mbar_wait(&s.empty[stage], phase ^ 1u, s.abort)) {
                ok = false;
                break;
            }
            uint8_t* a = s.stages + (size_t)stage * G::StageBytes;
            uint8_t* b = a + kBM * kF8BK;
            tc::mbar_arrive_expect_tx(&s.full[stage], tx);
            tc::tma_load_2d(a, &p.tmA[abox], &s.full[stage], kb * kF8BK, t.row0);
            if (kUp)  // gate rows n0..n0+127 then up rows I+n0.. in one box
                tc::tma_load_3d(b, &p.tmB, &s.full[stage], kb * kF8BK, t.nt * 128, 2 * t.e);
            else
                tc::tma_load_2d(b, &p.tmB, &s.full[stage], kb * kF8BK, b0);
            pending |= 1u << stage;
            pend_par = (pend_par & ~(1u << stage)) | (phase << stage);
            if (++stage == G::Stages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    if (!ok) {
        fail(s, p.err);
        // let the copies already issued land before the CTA exits
        for (int st = 0; st < G::Stages; ++st)
            if ((pending >> st) & 1u) {
                const uint64_t t0 = tc::globaltimer();
                while (!tc::mbar_try_wait(&s.full[st], (pend_par >> st) & 1u) &&
                       tc::globaltimer() - t0 < tc::kWaitTimeoutNs) {
                }
            }
    }
}

// Position of the scale stager's loads in the CTA's sequence of (tile, k-block) steps,
// with the tile's scale rows for this lane.
struct ScaleCursor {
    int lin, kb;
    const float* arow[4];  // A scale rows of tile rows 32c + lane (null past the tile)
    const float* bs0;      // B scales of the tile's first 128 weight rows
    const float* bs1;      // up kernel: of the up rows
};

template <bool kUp>
__device__ __forceinline__ void cursor_tile(const TcParams& p, const Smem& s, int total, ScaleCursor& c) {
    const int lane = threadIdx.x & 31;
    const int ksb = p.K / kF8BK;
    c.kb = 0;
    if (c.lin >= total) return;
    const Tile t = decode_tile(p, s, total, c.lin);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int rr = 32 * i + lane;
        const int64_t row = (int64_t)t.row0 + rr;
        int64_t src = -1;  // the scale row: the row itself, or its token when gathering
        if (rr < t.rows && row < p.max_rows) src = p.gather ? (int64_t)__ldg(p.gather + row) : row;
        c.arow[i] = src >= 0 ? p.a_scale + src * p.a_rs : nullptr;
    }
    // B rows 0-127 and 128-255 of the tile: up, the gate and the up n-block; down, two
    // consecutive 128-row blocks of W2
    const float* bsc = p.b_scale + (size_t)t.e * (p.NB / kF8BK) * ksb;
    const int nb0 = kUp ? t.nt : t.nt * (F8<kUp>::N / 128);
    const int nb1 = kUp ? p.I / kF8BK + t.nt : nb0 + 1;
    c.bs0 = bsc + (size_t)nb0 * ksb;
    c.bs1 = bsc + (size_t)nb1 * ksb;
}

template <bool kUp>
__device__ __forceinline__ void cursor_next(const TcParams& p, const Smem& s, int total, ScaleCursor& c) {
    if (c.lin < total && ++c.kb == p.kblocks) {
        c.lin += gridDim.x;
        cursor_tile<kUp>(p, s, total, c);
    }
}

// Loads the scales of the cursor's step (1.0 past the end), then moves the cursor to
// this warp's next step (kF8Stagers steps on).
template <bool kUp>
__device__ __forceinline__ void cursor_fetch(const TcParams& p, const Smem& s, int total, ScaleCursor& c,
                                             float (&va)[4], float& v0, float& v1) {
    const bool in = c.lin < total;
#pragma unroll
    for (int i = 0; i < 4; ++i) va[i] = (in && c.arow[i]) ? __ldg(c.arow[i] + c.kb * p.a_cs) : 1.0f;
    v0 = in ? __ldg(c.bs0 + c.kb) : 1.0f;
    v1 = (in && F8<kUp>::N == 256) ? __ldg(c.bs1 + c.kb) : 1.0f;
#pragma unroll
    for (int k = 0; k < kF8Stagers; ++k) cursor_next<kUp>(p, s, total, c);
}

// Whole warp: for each stage, its row of the stage's three 32 x 16-byte scale blocks:
// A (word c of row i = the scale of tile row 32c + i, the layout the MMA reads after
// the replicating copy), B rows 0-127 and B rows 128-255 (one value each), then the
// second arrival on full[stage].  The CTA's (tile, k-block) steps form one sequence,
// shared out round-robin among the kF8Stagers staging warps (`which` = this warp's
// turn); each loads its scales kScGroup of its steps ahead of their use, across tile
// boundaries, so a load's latency stays hidden even for tiles of a few k-blocks.
template <bool kUp>
__device__ void scale_stager_f8(const TcParams& p, const Smem& s, int total, int which) {
    using G = F8<kUp>;
    const int lane = threadIdx.x & 31;
    const int tiles = blockIdx.x < (unsigned)total ? (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int steps = tiles * p.kblocks;
    ScaleCursor cur;
    cur.lin = blockIdx.x;
    cursor_tile<kUp>(p, s, total, cur);
    for (int k = 0; k < which; ++k) cursor_next<kUp>(p, s, total, cur);
    float ca[kScGroup][4], c0[kScGroup], c1[kScGroup];
#pragma unroll
    for (int j = 0; j < kScGroup; ++j) cursor_fetch<kUp>(p, s, total, cur, ca[j], c0[j], c1[j]);
    bool ok = true;
    for (int i0 = 0; i0 * kF8Stagers + which < steps && ok; i0 += kScGroup) {
        float na[kScGroup][4], n0[kScGroup], n1[kScGroup];
#pragma unroll
        for (int j = 0; j < kScGroup; ++j) cursor_fetch<kUp>(p, s, total, cur, na[j], n0[j], n1[j]);
#pragma unroll
        for (int j = 0; j < kScGroup; ++j) {
            const int step = (i0 + j) * kF8Stagers + which;
            if (step >= steps) break;
            const int stage = step % G::Stages;
            const uint32_t phase = (uint32_t)(step / G::Stages) & 1u;
            if (!tc::mbar_wait(&s.empty[stage], phase ^ 1u, s.abort)) {
                ok = false;
                break;
            }
            uint4* sf = reinterpret_cast<uint4*>(s.sf + (size_t)stage * kSfStageBytes);
            sf[lane] = make_uint4(ue8m0x4(ca[j][0]), ue8m0x4(ca[j][1]), ue8m0x4(ca[j][2]), ue8m0x4(ca[j][3]));
            const uint32_t w0 = ue8m0x4(c0[j]), w1 = ue8m0x4(c1[j]);
            sf[32 + lane] = make_uint4(w0, w0, w0, w0);
            if (G::N == 256) sf[64 + lane] = make_uint4(w1, w1, w1, w1);
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&s.full[stage]);
        }
#pragma unroll
        for (int j = 0; j < kScGroup; ++j) {
#pragma unroll
            for (int i = 0; i < 4; ++i) ca[j][i] = na[j][i];
            c0[j] = n0[j];
            c1[j] = n1[j];
        }
    }
    if (!ok) fail(s, p.err);
}

template <bool kUp>
__device__ void mma_issuer_f8(const TcParams& p, const Smem& s, int total, uint32_t tmem_base) {
    using G = F8<kUp>;
    int stage = 0, buf = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true;
    constexpr uint32_t idesc = tc::idesc_mx_e4m3(kBM, G::N);
    for (int lin = blockIdx.x; lin < total && ok; lin += gridDim.x) {
        if (!tc::mbar_wait(&s.tempty[buf], acc_phase ^ 1u, s.abort)) {
            ok = false;
            break;
        }
        tc::tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(buf * G::N);
        for (int kb = 0; kb < p.kblocks; ++kb) {
            if (!tc::mbar_wait(&s.full[stage], phase, s.abort)) {
                ok = false;
                break;
            }
            tc::tc_fence_after();
            const uint32_t a_addr = tc::smem_u32(s.stages + (size_t)stage * G::StageBytes);
            const uint32_t b_addr = a_addr + kBM * kF8BK;
            const uint32_t sf_smem = tc::smem_u32(s.sf + (size_t)stage * kSfStageBytes);
            const uint32_t sf = tmem_base + (uint32_t)(kSfCol + 16 * stage);
            tc::tmem_cp_32x128b_x4(sf, tc::desc_rows16(sf_smem));                // A: columns sf .. sf+3
            tc::tmem_cp_32x128b_x4(sf + 8, tc::desc_rows16(sf_smem + 512));       // B rows 0-127
            if (G::N == 256) tc::tmem_cp_32x128b_x4(sf + 12, tc::desc_rows16(sf_smem + 1024));  // B rows 128-255
#pragma unroll
            for (int kk = 0; kk < kF8BK / 32; ++kk)
                tc::mma_mx_e4m3(d, tc::desc_sw128_kmajor(a_addr + kk * 32), tc::desc_sw128_kmajor(b_addr + kk * 32),
                                idesc, sf, sf + 8, (kb | kk) != 0 ? 1u : 0u);
            tc::mma_commit(&s.empty[stage]);  // stage (tiles and scales) free once these finish
            if (++stage == G::Stages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok) break;
        tc::mma_commit(&s.tfull[buf]);
        if (++buf == G::AccBufs) {
            buf = 0;
            acc_phase ^= 1u;
        }
    }
    if (!ok) fail(s, p.err);
    tc::mma_commit(s.drain);
    const uint64_t t0 = tc::globaltimer();
    while (!tc::mbar_try_wait(s.drain, 0) && tc::globaltimer() - t0 < tc::kWaitTimeoutNs) {
    }
}

__device__ __forceinline__ void release_acc(const Smem& s, int buf) {
    tc::tc_fence_before();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) tc::mbar_arrive(&s.tempty[buf]);
}

// Eight warps, two per TMEM lane quarter; `half` selects half of the tile's columns.
template <bool kUp, bool kComb>
__device__ void epilogue_f8(const TcParams& p, const Smem& s, int total, uint32_t tmem_base) {
    using G = F8<kUp>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3;
    const int half = (warp - kF8FirstEpiWarp) >> 2;
    const int r = q * 32 + lane;
    int buf = 0;
    uint32_t acc_phase = 0;
    int seq = 0;
    bool ok = true;
    for (int lin = blockIdx.x; lin < total && ok; lin += gridDim.x) {
        const Tile t = decode_tile(p, s, total, lin);
        const int64_t row = (int64_t)t.row0 + r;
        const bool valid = r < t.rows;
        // a warp whose 32 rows are all past the tile's rows has nothing to read (at
        // decode most tiles hold fewer than 32 rows)
        const bool busy = q * 32 < t.rows;
        if (!tc::mbar_wait(&s.tfull[buf], acc_phase, s.abort)) {
            ok = false;
            break;
        }
        tc::tc_fence_after();
        const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * G::N);
        if (kUp) {
            uint32_t g0[32], g1[32], u0[32], u1[32];  // gate / up columns 64*half .. +63
            if (busy) {
                tc::tmem_ld32(tb + 64 * half, g0);
                tc::tmem_ld32(tb + 64 * half + 32, g1);
                tc::tmem_ld32(tb + 128 + 64 * half, u0);
                tc::tmem_ld32(tb + 128 + 64 * half + 32, u1);
                tc::tmem_wait_ld();
            }
            release_acc(s, buf);
            float amax = 0.0f;
            if (busy) {
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float ga = __uint_as_float(g0[i]), gb = __uint_as_float(g1[i]);
                    const float ha = silu_mul_fast(ga, __uint_as_float(u0[i]));
                    const float hb = silu_mul_fast(gb, __uint_as_float(u1[i]));
                    g0[i] = __float_as_uint(ha);
                    g1[i] = __float_as_uint(hb);
                    amax = fmaxf(amax, fmaxf(fabsf(ha), fabsf(hb)));
                }
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
            ok = __all_sync(0xffffffffu, ok);  // a wait that ran out ends the tile for the whole warp
            if (!ok) break;
            __threadfence_block();
            amax = fmaxf(amax, s.xval[(par * 2 + 1 - half) * 128 + r]);
            if (busy) {
                const int se = fp8_scale_exp(amax);
                const Pow2Factors f = pow2_neg(se);
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const uint32_t* src = i < 8 ? g0 + 4 * i : g1 + 4 * (i - 8);
                    const uint16_t lo = f2_to_e4m3x2(scale_by(__uint_as_float(src[0]), f),
                                                     scale_by(__uint_as_float(src[1]), f));
                    const uint16_t hi = f2_to_e4m3x2(scale_by(__uint_as_float(src[2]), f),
                                                     scale_by(__uint_as_float(src[3]), f));
                    w[i] = (uint32_t)lo | ((uint32_t)hi << 16);
                }
                // this warp's 32 rows x 64 bytes of h, staged for row-contiguous stores
                uint8_t* hbase = static_cast<uint8_t*>(p.out) + ((int64_t)t.row0 + q * 32) * p.I + t.nt * 128 + 64 * half;
                store_rows64(s.oslot + (size_t)(warp - kF8FirstEpiWarp) * (kOutSlotBytes / 16), w, hbase, p.I,
                             min(32, t.rows - q * 32), lane);
                if (valid && half == 0) p.out_scale[(int64_t)t.nt * p.max_rows + row] = mul_pow2(1.0f, se);
            }
        } else if (kComb) {
            // fused combine: the accumulator in two passes of 64 columns (registers for the
            // combine), released after the second
            uint16_t* yrow = static_cast<uint16_t*>(p.out) + row * p.H + t.nt * G::N + 128 * half;
#pragma unroll 1
            for (int pass = 0; pass < 2; ++pass) {
                uint32_t a[2][32];
                if (busy) {
                    tc::tmem_ld32(tb + 128 * half + 64 * pass, a[0]);
                    tc::tmem_ld32(tb + 128 * half + 64 * pass + 32, a[1]);
                    tc::tmem_wait_ld();
                }
                if (pass == 1) release_acc(s, buf);
                if (valid) {
                    uint4* dst = reinterpret_cast<uint4*>(yrow + 64 * pass);
#pragma unroll
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[4 * c + i] = make_uint4(
                                pack_bf16x2(__uint_as_float(a[c][8 * i]), __uint_as_float(a[c][8 * i + 1])),
                                pack_bf16x2(__uint_as_float(a[c][8 * i + 2]), __uint_as_float(a[c][8 * i + 3])),
                                pack_bf16x2(__uint_as_float(a[c][8 * i + 4]), __uint_as_float(a[c][8 * i + 5])),
                                pack_bf16x2(__uint_as_float(a[c][8 * i + 6]), __uint_as_float(a[c][8 * i + 7])));
                }
            }
            combine_slab(p, valid, row, t.nt * 2 + half);  // this warp's 128 columns
        } else {
            uint32_t a[4][32];  // columns 128*half .. +127 of the 256-wide tile
            if (busy) {
#pragma unroll
                for (int c = 0; c < 4; ++c) tc::tmem_ld32(tb + 128 * half + 32 * c, a[c]);
                tc::tmem_wait_ld();
            }
            release_acc(s, buf);
            if (busy) {  // this warp's 32 rows, 32 columns (64 bytes) a pass, staged stores
                uint8_t* ybase = reinterpret_cast<uint8_t*>(static_cast<uint16_t*>(p.out) +
                                                            ((int64_t)t.row0 + q * 32) * p.H + t.nt * G::N + 128 * half);
                uint4* slot = s.oslot + (size_t)(warp - kF8FirstEpiWarp) * (kOutSlotBytes / 16);
                const int nrows = min(32, t.rows - q * 32);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
#pragma unroll
                    for (int i = 0; i < 16; ++i)  // packed in place: word i from words 2i, 2i+1
                        a[c][i] = pack_bf16x2(__uint_as_float(a[c][2 * i]), __uint_as_float(a[c][2 * i + 1]));
                    store_rows64(slot, a[c], ybase + 64 * c, (int64_t)p.H * 2, nrows, lane);
                }
            }
        }
        if (++buf == G::AccBufs) {
            buf = 0;
            acc_phase ^= 1u;
        }
    }
    if (!ok) fail(s, p.err);
}

template <bool kUp, bool kComb>
__global__ void __launch_bounds__(kF8Threads, 1) ffn_tc_fp8_kernel(const __grid_constant__ TcParams p) {
    using G = F8<kUp>;
    extern __shared__ uint8_t smem_raw[];
    const Smem s = carve(smem_raw, G::Stages, G::StageBytes, kSfStageBytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < G::Stages; ++i) {
            tc::mbar_init(&s.full[i], 2);
            tc::mbar_init(&s.empty[i], 1);
        }
        for (int i = 0; i < G::AccBufs; ++i) {
            tc::mbar_init(&s.tfull[i], 1);
            tc::mbar_init(&s.tempty[i], 8);
        }
        tc::mbar_init(s.drain, 1);
        tc::mbar_init(s.never, 1);
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
    zero_counters(p);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem_base = *s.tmem_base;
    const int total = s.tstart[p.NE];

    if (warp == 0) {
        if (kUp && p.gather) producer_gather<kF8BK>(p, s, total);
        else if (lane == 0) producer_f8<kUp>(p, s, total);
    } else if (warp == 1) {
        if (lane == 0) mma_issuer_f8<kUp>(p, s, total, tmem_base);
    } else if (warp < kF8FirstEpiWarp) {
        scale_stager_f8<kUp>(p, s, total, warp - 2);
    } else {
        epilogue_f8<kUp, kComb>(p, s, total, tmem_base);
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() { return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tma_encode_fn()); }

bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, bool fp8, int box_rows = 128) {
    return make_tma_map_2d(m, base, inner, rows, fp8, box_rows);
}

// W13 [NE][2I][K] as a 3-D tensor [2 NE][I][K] (gate half 2e, up half 2e + 1) with a
// box of one 128-byte row x 128 rows x both halves: one copy brings the up tile's B.
bool make_map_w13(CUtensorMap* m, const void* base, uint64_t K, uint64_t I, uint64_t NE, bool fp8) {
    auto enc = encode_fn();
    if (!enc) return false;
    const uint64_t elt = fp8 ? 1 : 2;
    cuuint64_t dims[3] = {K, I, 2 * NE};
    cuuint64_t strides[2] = {K * elt, I * K * elt};
    cuuint32_t box[3] = {(cuuint32_t)(128 / elt), 128, 2};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base),
               dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kUp, bool kFp8, bool kComb = false>
cudaError_t launch_one(const TcParams& p, int grid, cudaStream_t st) {
    auto kern = kFp8 ? ffn_tc_fp8_kernel<kUp, kComb> : ffn_tc_bf16_kernel<kUp, kComb>;
    const size_t smem = kFp8 ? kF8SmemBytes<kUp> : kSmemBytes;
    cudaError_t e = ensure_max_dynamic_smem(kern, (int)smem);
    if (e != cudaSuccess) return e;
    // programmatic dependent launch: this kernel's prologue may overlap the tail of the
    // previous kernel on the stream; it waits (griddepcontrol.wait) before reading
    // anything that kernel wrote
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kFp8 ? kF8Threads : kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

void* tma_encode_fn() {
    static void* fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = f;
    }
    return fn;
}

// 2-D K-major matrix [rows][inner] with the 128-byte swizzle and a box of one
// 128-byte row (64 bf16 or 128 e4m3) by box_rows rows.
bool make_tma_map_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, bool fp8, int box_rows) {
    auto enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(tma_encode_fn());
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

bool ffn_tc_supported(const moe_config& c) {
    const DeviceInfo& d = device_info();
    const size_t smem = c.dtype == MOE_FP8_E4M3 ? (kF8SmemBytes<true> > kF8SmemBytes<false> ? kF8SmemBytes<true>
                                                                                              : kF8SmemBytes<false>)
                                                : kSmemBytes;
    return (c.dtype == MOE_BF16 || c.dtype == MOE_FP8_E4M3) && d.cc_major == 10 && c.hidden % kBN == 0 &&
           c.inter % 128 == 0 && d.smem_optin >= smem && encode_fn() != nullptr;
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
    if (!make_map_w13(&up.tmB, a.w13, (uint64_t)H, (uint64_t)I, (uint64_t)NE, fp8)) return cudaErrorInvalidValue;
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
    up.a_rs = a.xs_cs ? 1 : H / kF8BK;  // see FfnArgs::xs_cs
    up.a_cs = a.xs_cs ? a.xs_cs : 1;
    up.b_scale = a.w13_scale;
    up.out_scale = h_scale;
    up.inject_ns = wait_injection_ns();
    if (a.token_of && a.gx) {  // fused gather: A rows straight from x / x_q by token
        if (!make_tma_map_2d(&up.tmG, a.gx, (uint64_t)H, (uint64_t)a.gT, fp8, 1)) return cudaErrorInvalidValue;
        up.gather = a.token_of;
        up.a_scale = a.gx_scale;
        up.a_rs = 1;
        up.a_cs = a.gT;
    }
    if (a.token_of && a.y) {  // the fused combine's counters start at zero
        up.zero = a.cnt;
        up.zero_n = (int64_t)a.gT * (H / 128);
    }
    TcParams dn = up;
    dn.gather = nullptr;
    dn.zero = nullptr;
    dn.zero_n = 0;
    if (a.y) {  // fused combine in the down kernel's epilogue
        dn.comb_token = a.token_of;
        dn.comb_slot = a.slot_of;
        dn.comb_w = a.topk_w;
        dn.comb_y = a.y;
        dn.comb_cnt = a.cnt;
        dn.comb_k = c.top_k;
        dn.comb_kk = c.top_k + c.num_shared;
        dn.comb_cols = fp8 ? 128 : kBN;
    }
    for (int i = 0; i < kNumABoxes; ++i)
        if (!make_map(&dn.tmA[i], h, (uint64_t)I, (uint64_t)a.max_rows, fp8, a_box_rows(i)))
            return cudaErrorInvalidValue;
    if (!make_map(&dn.tmB, a.w2, (uint64_t)I, (uint64_t)NE * H, fp8, fp8 ? F8<false>::N : kBN))
        return cudaErrorInvalidValue;
    dn.K = I;
    dn.kblocks = I / kelems;
    dn.NB = H;
    dn.ntn = H / (fp8 ? F8<false>::N : kBN);
    dn.out = a.ye;
    dn.a_scale = h_scale;  // written column-major by the up kernel
    dn.a_rs = 1;
    dn.a_cs = a.max_rows;
    dn.b_scale = a.w2_scale;
    dn.out_scale = nullptr;
    cudaError_t e = fp8 ? launch_one<true, true>(up, grid, st) : launch_one<true, false>(up, grid, st);
    if (e != cudaSuccess) return e;
    if (a.y)
        return fp8 ? launch_one<false, true, true>(dn, grid, st) : launch_one<false, false, true>(dn, grid, st);
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
    if (!make_map(&p.tmB, wa, (uint64_t)H, (uint64_t)H, false, kBN)) return cudaErrorInvalidValue;
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
