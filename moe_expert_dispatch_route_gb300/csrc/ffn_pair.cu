// Grouped expert FFN on CTA pairs (tcgen05.mma.cta_group::2), for batches where most
// experts hold a few hundred rows (prefill).
//
// A cluster of two CTAs on the two SMs of a TPC computes one 256 x 256 tile: CTA r
// (r = cluster rank) loads rows 128r .. 128r+127 of the tile's A rows and B rows
// 128r .. 128r+127 of the 256 weight rows, each with its own plain TMA copies (no
// multicast); one thread of the leader (r = 0) issues the pair MMAs, which read A from
// both CTAs' shared memory and both halves of B, and leave rows 128r.. of the 256 x
// 256 fp32 accumulator in CTA r's TMEM.  Per SM and k-block that is 32 KB of operands
// for a 128 x 256 x K product (the one-CTA kernels move 48 KB for the same work), so
// six stages fit in shared memory where the one-CTA kernels hold four.
//   up   : acc = xe[rows] . [W13 gate rows n0.. (CTA 0's half) | up rows I+n0.. (CTA 1's)]^T,
//          epilogue h = silu(g) * u  (fp8: e4m3 + 1x128 power-of-two scale; bf16: bf16)
//   down : acc = h[rows] . W2[e][n0 .. n0+255]^T, epilogue -> bf16 ye
// Tiles (expert, n-block, 256-row m-block) come from the device counts, as in the
// one-CTA kernels; both CTAs of a pair walk the same tile sequence.
//
// Synchronisation (all waits bounded, see tc_ptx.cuh).  Waits and the leader's own
// arrivals are CTA-scoped: the phases that carry data complete through the async proxy
// (TMA complete_tx, tcgen05.commit), which orders the data by itself.  Only the peer's
// remote arrivals (its epilogue's, once per tile) are released at cluster scope.
//   full[s]   leader only: the leader producer's arrive.expect_tx (both CTAs' bytes),
//             both CTAs' copies complete on it, and (fp8) the scale stager arrives;
//   empty[s]  in both CTAs: the leader's MMA commit, multicast to the pair;
//   tfull     in both CTAs: the leader's commit after a tile's last k-block;
//   tempty    leader only: every epilogue warp of both CTAs arrives once its rows are
//             in registers (the peer's warps arrive remotely);
//   drain     in both CTAs: the leader's final commit; nobody frees TMEM before it.
// FP8 scale factors: one warp of the leader stages, per step, each CTA's A rows' scales
// and the 256 B rows' scales into that CTA's shared memory (the peer's through
// distributed shared memory); the leader copies them into TMEM with the pair form of
// tcgen05.cp (each CTA's shared memory into its own TMEM at the same address).
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

constexpr int kRows = 128;        // A rows per CTA (the pair tile has 256)
constexpr int kPairRows = 256;
constexpr int kN = 256;           // accumulator columns
constexpr int kStages = 6;
constexpr int kABytes = kRows * 128;  // one 128-byte k-row of 128 A rows
constexpr int kBBytes = 128 * 128;    // this CTA's 128 B rows
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kSfBytes = 1536;    // fp8: A scales, B rows 0-127, B rows 128-255 (32 x 16 B each)
constexpr int kSfCol = 256;       // fp8: TMEM column of stage 0's scale slot (16 columns a stage)
constexpr uint32_t kTmemCols = 512;
constexpr int kNumABoxes = 4;     // A boxes of 16 / 32 / 64 / 128 rows
constexpr int kEpiWarps = 8;      // two per TMEM lane quarter, each half of the columns
constexpr int kFirstEpiWarp = 3;  // warp 0 TMA, 1 MMA, 2 scale stager (fp8) / idle (bf16)
constexpr int kThreads = 32 * (kFirstEpiWarp + kEpiWarps);
constexpr int kScGroup = 4;       // fp8: k-blocks of scales loaded ahead (8 A values a lane per step)
__host__ __device__ constexpr int a_box_rows(int i) { return 16 << i; }

template <bool kFp8>
struct Cfg {
    static constexpr int KElems = kFp8 ? 128 : 64;  // elements per k-block (one 128-byte row)
    static constexpr int AccBufs = kFp8 ? 1 : 2;    // fp8 keeps TMEM columns for the scales
    static constexpr int SfBytes = kFp8 ? kSfBytes : 0;
};

constexpr size_t kTail = 64 * 8 + 16 + 3 * (kMaxExperts + 1) * sizeof(int) + 512 * sizeof(float) + 256 * sizeof(int);
// bf16: per epilogue warp, 32 rows x 64 bytes of output staging (the fp8 kernels have no
// room left for it and store row by row)
constexpr int kOutSlotBytes = 2048;
template <bool kFp8>
constexpr size_t smem_bytes() {
    return 1024 + (size_t)kStages * (kStageBytes + Cfg<kFp8>::SfBytes) + kTail +
           (kFp8 ? 0 : 128 + (size_t)kEpiWarps * kOutSlotBytes);
}

struct PairParams {
    CUtensorMap tmA[kNumABoxes];  // activations [max_rows][K]
    CUtensorMap tmB;              // weights as [NE * NB][K] (up: W13, down: W2), box = 128 rows
    const int32_t* counts;
    const int32_t* offsets;
    int NE, K, kblocks;
    int NB;   // weight rows per expert (up 2I, down H)
    int ntn;  // n-blocks of 256 columns per expert
    int I, H;
    int64_t max_rows;
    void* out;
    int32_t* err;
    int reverse;
    const float* a_scale;  // fp8: (row r, group g) at r * a_rs + g * a_cs
    int64_t a_rs, a_cs;
    const float* b_scale;  // fp8: [NE][NB/128][K/128]
    float* out_scale;      // fp8 up: h scales, column-major [I/128][max_rows]
    int64_t inject_ns;     // test hook: > 0 = the producer's first wait runs out after this long
};

struct Smem {
    uint8_t* stages;
    uint8_t* sf;
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
    float* xval;
    volatile int* xseq;
    uint4* oslot;  // bf16: kOutSlotBytes per epilogue warp
};

__device__ __forceinline__ Smem carve(uint8_t* raw, int sf_bytes) {
    Smem s;
    uint8_t* p = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
    s.stages = p;
    p += (size_t)kStages * kStageBytes;
    s.sf = p;
    p += (size_t)kStages * sf_bytes;
    s.full = reinterpret_cast<uint64_t*>(p);
    s.empty = s.full + kStages;
    s.tfull = s.empty + kStages;  // [2]
    s.tempty = s.tfull + 2;       // [2]
    s.drain = s.tempty + 2;
    s.never = s.drain + 1;
    s.tmem_base = reinterpret_cast<uint32_t*>(s.full + 64);
    s.abort = reinterpret_cast<volatile int*>(s.tmem_base + 1);
    s.tstart = reinterpret_cast<int*>(s.tmem_base + 4);
    s.cnt = s.tstart + (kMaxExperts + 1);
    s.off = s.cnt + (kMaxExperts + 1);
    s.xval = reinterpret_cast<float*>(s.off + (kMaxExperts + 1));
    s.xseq = reinterpret_cast<volatile int*>(s.xval + 512);
    s.oslot = reinterpret_cast<uint4*>((reinterpret_cast<uintptr_t>(s.xseq + 256) + 127) & ~uintptr_t(127));
    return s;
}

// Stores 64 bytes of each of a warp's 32 rows (lane i holds row i's words w[0..15])
// through the warp's shared slot, 16-byte chunks XOR-swizzled by row, so that each
// global store instruction covers 8 rows x 64 contiguous bytes.  Whole warp.
__device__ __forceinline__ void store_rows64(uint4* slot, const uint32_t* w, uint8_t* base, int64_t pitch, int nrows,
                                             int lane) {
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
    int e, nt, rows, row0;  // rows / row0 of the whole 256-row pair tile
};

__device__ __forceinline__ int pair_index() { return (int)(blockIdx.x >> 1); }
__device__ __forceinline__ int num_pairs() { return (int)(gridDim.x >> 1); }

__device__ __forceinline__ Tile decode_tile(const PairParams& p, const Smem& s, int total, int lin) {
    const int tile = p.reverse ? total - 1 - lin : lin;
    int lo = 0, hi = p.NE - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s.tstart[mid] <= tile) lo = mid;
        else hi = mid - 1;
    }
    Tile t;
    t.e = lo;
    const int local = tile - s.tstart[lo];
    const int cnt = s.cnt[lo];
    const int mtiles = (cnt + kPairRows - 1) / kPairRows;
    t.nt = local / mtiles;  // n-major within an expert: neighbouring pairs share B
    const int mt = local % mtiles;
    t.row0 = s.off[lo] + mt * kPairRows;
    t.rows = min(kPairRows, cnt - mt * kPairRows);
    return t;
}

// rows of the pair tile that belong to CTA `rank`
__device__ __forceinline__ int cta_rows(const Tile& t, uint32_t rank) {
    return max(0, min(kRows, t.rows - (int)rank * kRows));
}

__device__ __forceinline__ int box_for(int rows) {
    int b = 0;
    while (b < kNumABoxes - 1 && a_box_rows(b) < rows) ++b;
    return b;
}

// One warp: counts/offsets into shared memory and the scan of the pair-tile counts.
__device__ void scan_tiles(const PairParams& p, const Smem& s) {
    const int lane = threadIdx.x & 31;
    const int per = (p.NE + 31) / 32;
    int vals[16];
    int sum = 0;
    for (int i = 0; i < per; ++i) {
        const int e = lane * per + i;
        int v = 0;
        if (e < p.NE) {
            int cnt = __ldg(p.counts + e);
            const int off = __ldg(p.offsets + e);
            if (cnt < 0 || off < 0 || (int64_t)off + cnt > p.max_rows) {
                set_err(p.err, MOE_ERR_BAD_INDEX);
                cnt = 0;
            }
            s.cnt[e] = cnt;
            s.off[e] = off;
            v = (cnt + kPairRows - 1) / kPairRows * p.ntn;
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

// ---------------------------------------------------------------- TMA producer (both CTAs)
template <bool kUp, bool kFp8>
__device__ void producer(const PairParams& p, const Smem& s, int total, uint32_t rank) {
    using C = Cfg<kFp8>;
    if (p.inject_ns > 0) {  // test hook: the first wait runs out before any copy is issued
        tc::wait_on_nothing(s.never, (uint64_t)p.inject_ns);
        fail(s, p.err);
        return;
    }
    const uint32_t leader_full = tc::map_to_rank(s.full, 0);  // leader's full[0]
    int stage = 0;
    uint32_t phase = 0;
    uint32_t pending = 0, pend_par = 0;
    bool ok = true;
    for (int lin = pair_index(); lin < total && ok; lin += num_pairs()) {
        const Tile t = decode_tile(p, s, total, lin);
        const int abox = box_for(cta_rows(t, rank)), pbox = box_for(cta_rows(t, rank ^ 1u));
        const uint32_t tx = (uint32_t)((a_box_rows(abox) + a_box_rows(pbox)) * 128 + 2 * kBBytes);
        const int arow = t.row0 + (int)rank * kRows;  // past the tensor: zero-filled, never stored
        const int brow = kUp ? t.e * p.NB + (int)rank * p.I + t.nt * 128 : t.e * p.NB + t.nt * kN + (int)rank * 128;
        for (int kb = 0; kb < p.kblocks; ++kb) {
            if (!tc::mbar_wait(&s.empty[stage], phase ^ 1u, s.abort)) {
                ok = false;
                break;
            }
            uint8_t* a = s.stages + (size_t)stage * kStageBytes;
            if (rank == 0) tc::mbar_arrive_expect_tx(&s.full[stage], tx);
            const uint32_t bar = leader_full + (uint32_t)(stage * 8);
            tc::tma_load_2d_pair(a, &p.tmA[abox], bar, kb * C::KElems, arow);
            tc::tma_load_2d_pair(a + kABytes, &p.tmB, bar, kb * C::KElems, brow);
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
        // let the copies already issued land before the CTA can exit: the leader sees
        // them on its full barriers; the peer's complete on the leader's, so it waits a
        // fixed time far above any copy's latency
        if (rank == 0) {
            for (int st = 0; st < kStages; ++st)
                if ((pending >> st) & 1u) {
                    const uint64_t t0 = tc::globaltimer();
                    while (!tc::mbar_try_wait(&s.full[st], (pend_par >> st) & 1u) &&
                           tc::globaltimer() - t0 < tc::kWaitTimeoutNs) {
                    }
                }
        } else if (pending) {
            const uint64_t t0 = tc::globaltimer();
            while (tc::globaltimer() - t0 < 2000000ull) {
            }
        }
    }
}

// ---------------------------------------------------------------- FP8 scale stager (leader only)
struct ScaleCursor {
    int lin, kb;
    const float* arow[8];  // A scale rows of pair-tile rows 32c + lane (c < 4: leader, c >= 4: peer)
    const float* bs0;
    const float* bs1;
};

template <bool kUp>
__device__ __forceinline__ void cursor_tile(const PairParams& p, const Smem& s, int total, ScaleCursor& c) {
    const int lane = threadIdx.x & 31;
    const int ksb = p.K / 128;
    c.kb = 0;
    if (c.lin >= total) return;
    const Tile t = decode_tile(p, s, total, c.lin);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int rr = 32 * i + lane;
        const int64_t row = (int64_t)t.row0 + rr;
        c.arow[i] = (rr < t.rows && row < p.max_rows) ? p.a_scale + row * p.a_rs : nullptr;
    }
    // B rows 0-127 and 128-255 of the tile (the same for both CTAs): up, the gate and the
    // up n-block; down, two consecutive 128-row blocks of W2
    const float* bsc = p.b_scale + (size_t)t.e * (p.NB / 128) * ksb;
    const int nb0 = kUp ? t.nt : t.nt * 2;
    const int nb1 = kUp ? p.I / 128 + t.nt : nb0 + 1;
    c.bs0 = bsc + (size_t)nb0 * ksb;
    c.bs1 = bsc + (size_t)nb1 * ksb;
}

template <bool kUp>
__device__ __forceinline__ void cursor_fetch(const PairParams& p, const Smem& s, int total, ScaleCursor& c,
                                             float (&va)[8], float& v0, float& v1) {
    const bool in = c.lin < total;
#pragma unroll
    for (int i = 0; i < 8; ++i) va[i] = (in && c.arow[i]) ? __ldg(c.arow[i] + c.kb * p.a_cs) : 1.0f;
    v0 = in ? __ldg(c.bs0 + c.kb) : 1.0f;
    v1 = in ? __ldg(c.bs1 + c.kb) : 1.0f;
    if (in && ++c.kb == p.kblocks) {
        c.lin += num_pairs();
        cursor_tile<kUp>(p, s, total, c);
    }
}

__device__ __forceinline__ uint32_t ue8m0x4(float pow2) {
    const uint32_t e = (__float_as_uint(pow2) >> 23) & 0xffu;
    return e * 0x01010101u;
}

// Whole warp of the leader: per step, the three 32 x 16-byte scale blocks of both CTAs
// (A: word c of row i = scale of the CTA's tile row 32c + i; B rows 0-127 and 128-255:
// word c of row i = scale of B row 32c + i, all equal within the tile's 128-row block),
// the leader's in its own shared memory, the peer's written into the peer's shared
// memory at the same offset; then one proxy fence and an arrival on full[stage].  The
// writer and the MMA thread that copies the blocks into both TMEMs are in the same
// CTA, so no cross-CTA release is needed per step.  Scales are loaded kScGroup steps
// ahead, across tile boundaries.
template <bool kUp>
__device__ void scale_stager(const PairParams& p, const Smem& s, int total) {
    const int lane = threadIdx.x & 31;
    const int tiles = pair_index() < total ? (total - 1 - pair_index()) / num_pairs() + 1 : 0;
    const int steps = tiles * p.kblocks;
    const uint32_t peer_sf = tc::map_to_rank(s.sf, 1);
    ScaleCursor cur;
    cur.lin = pair_index();
    cursor_tile<kUp>(p, s, total, cur);
    float ca[kScGroup][8], c0[kScGroup], c1[kScGroup];
#pragma unroll
    for (int j = 0; j < kScGroup; ++j) cursor_fetch<kUp>(p, s, total, cur, ca[j], c0[j], c1[j]);
    bool ok = true;
    for (int i0 = 0; i0 < steps && ok; i0 += kScGroup) {
        float na[kScGroup][8], n0[kScGroup], n1[kScGroup];
#pragma unroll
        for (int j = 0; j < kScGroup; ++j) cursor_fetch<kUp>(p, s, total, cur, na[j], n0[j], n1[j]);
#pragma unroll
        for (int j = 0; j < kScGroup; ++j) {
            const int step = i0 + j;
            if (step >= steps) break;
            const int stage = step % kStages;
            const uint32_t phase = (uint32_t)(step / kStages) & 1u;
            if (!tc::mbar_wait(&s.empty[stage], phase ^ 1u, s.abort)) {
                ok = false;
                break;
            }
            uint4* sf = reinterpret_cast<uint4*>(s.sf + (size_t)stage * kSfBytes);
            const uint32_t psf = peer_sf + (uint32_t)(stage * kSfBytes);
            const uint32_t w0 = ue8m0x4(c0[j]), w1 = ue8m0x4(c1[j]);
            const uint4 b0 = make_uint4(w0, w0, w0, w0), b1 = make_uint4(w1, w1, w1, w1);
            sf[lane] = make_uint4(ue8m0x4(ca[j][0]), ue8m0x4(ca[j][1]), ue8m0x4(ca[j][2]), ue8m0x4(ca[j][3]));
            sf[32 + lane] = b0;
            sf[64 + lane] = b1;
            tc::st_cluster_v4(psf + 16u * lane, make_uint4(ue8m0x4(ca[j][4]), ue8m0x4(ca[j][5]),
                                                           ue8m0x4(ca[j][6]), ue8m0x4(ca[j][7])));
            tc::st_cluster_v4(psf + 16u * (32 + lane), b0);
            tc::st_cluster_v4(psf + 16u * (64 + lane), b1);
            tc::fence_proxy_async_cluster_smem();  // both CTAs' blocks -> the leader's tcgen05.cp
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&s.full[stage]);
        }
#pragma unroll
        for (int j = 0; j < kScGroup; ++j) {
#pragma unroll
            for (int i = 0; i < 8; ++i) ca[j][i] = na[j][i];
            c0[j] = n0[j];
            c1[j] = n1[j];
        }
    }
    if (!ok) fail(s, p.err);
}

// ---------------------------------------------------------------- MMA issuer (leader only)
template <bool kFp8>
__device__ void mma_issuer(const PairParams& p, const Smem& s, int total, uint32_t tmem_base) {
    using C = Cfg<kFp8>;
    int stage = 0, buf = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true;
    const uint32_t idesc = kFp8 ? tc::idesc_mx_e4m3(kPairRows, kN) : tc::idesc_bf16_f32(kPairRows, kN);
    for (int lin = pair_index(); lin < total && ok; lin += num_pairs()) {
        if (!tc::mbar_wait(&s.tempty[buf], acc_phase ^ 1u, s.abort)) {
            ok = false;
            break;
        }
        tc::tc_fence_after();
        const uint32_t d = tmem_base + (uint32_t)(buf * kN);
        for (int kb = 0; kb < p.kblocks; ++kb) {
            if (!tc::mbar_wait(&s.full[stage], phase, s.abort)) {
                ok = false;
                break;
            }
            tc::tc_fence_after();
            const uint32_t a_addr = tc::smem_u32(s.stages + (size_t)stage * kStageBytes);
            const uint32_t b_addr = a_addr + kABytes;
            if (kFp8) {
                const uint32_t sf_smem = tc::smem_u32(s.sf + (size_t)stage * kSfBytes);
                const uint32_t sf = tmem_base + (uint32_t)(kSfCol + 16 * stage);
                tc::tmem_cp_32x128b_x4_pair(sf, tc::desc_rows16(sf_smem));              // A rows
                tc::tmem_cp_32x128b_x4_pair(sf + 8, tc::desc_rows16(sf_smem + 512));    // B rows 0-127
                tc::tmem_cp_32x128b_x4_pair(sf + 12, tc::desc_rows16(sf_smem + 1024));  // B rows 128-255
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc::mma_mx_e4m3_pair(d, tc::desc_sw128_kmajor(a_addr + kk * 32),
                                         tc::desc_sw128_kmajor(b_addr + kk * 32), idesc, sf, sf + 8,
                                         (kb | kk) != 0 ? 1u : 0u);
            } else {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc::mma_bf16_pair(d, tc::desc_sw128_kmajor(a_addr + kk * 32),
                                      tc::desc_sw128_kmajor(b_addr + kk * 32), idesc, (kb | kk) != 0 ? 1u : 0u);
            }
            tc::mma_commit_pair(&s.empty[stage], 3);  // both CTAs' stage free once these finish
            if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok) break;
        tc::mma_commit_pair(&s.tfull[buf], 3);
        if (++buf == C::AccBufs) {
            buf = 0;
            acc_phase ^= 1u;
        }
    }
    if (!ok) fail(s, p.err);
    tc::mma_commit_pair(s.drain, 3);
}

// ---------------------------------------------------------------- epilogue (both CTAs)
__device__ __forceinline__ void release_acc(const Smem& s, int buf, uint32_t rank, uint32_t leader_tempty) {
    tc::tc_fence_before();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
        if (rank == 0) tc::mbar_arrive(&s.tempty[buf]);
        else tc::mbar_arrive_remote(leader_tempty + (uint32_t)(buf * 8));
    }
}



// Eight warps, two per TMEM lane quarter; `half` selects half of the tile's columns
// (up: 64 gate + the matching 64 up columns; down: 128 of the 256).
template <bool kUp, bool kFp8>
__device__ void epilogue(const PairParams& p, const Smem& s, int total, uint32_t tmem_base, uint32_t rank) {
    using C = Cfg<kFp8>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3;
    const int half = (warp - kFirstEpiWarp) >> 2;
    const int r = q * 32 + lane;  // this thread's row within the CTA's 128
    const uint32_t leader_tempty = tc::map_to_rank(s.tempty, 0);
    int buf = 0;
    uint32_t acc_phase = 0;
    int seq = 0;
    bool ok = true;
    for (int lin = pair_index(); lin < total && ok; lin += num_pairs()) {
        const Tile t = decode_tile(p, s, total, lin);
        const int my_rows = cta_rows(t, rank);
        const int64_t row = (int64_t)t.row0 + (int)rank * kRows + r;
        const bool valid = r < my_rows;
        const bool busy = q * 32 < my_rows;  // a warp whose 32 rows are all empty reads nothing
        if (!tc::mbar_wait(&s.tfull[buf], acc_phase, s.abort)) {
            ok = false;
            break;
        }
        tc::tc_fence_after();
        const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * kN);
        if (kUp) {
            uint32_t g0[32], g1[32], u0[32], u1[32];  // gate / up columns 64*half .. +63
            if (busy) {
                tc::tmem_ld32(tb + 64 * half, g0);
                tc::tmem_ld32(tb + 64 * half + 32, g1);
                tc::tmem_ld32(tb + 128 + 64 * half, u0);
                tc::tmem_ld32(tb + 128 + 64 * half + 32, u1);
                tc::tmem_wait_ld();
            }
            release_acc(s, buf, rank, leader_tempty);
            float amax = 0.0f;
            if (busy) {
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float ha = silu_mul_fast(__uint_as_float(g0[i]), __uint_as_float(u0[i]));
                    const float hb = silu_mul_fast(__uint_as_float(g1[i]), __uint_as_float(u1[i]));
                    g0[i] = __float_as_uint(ha);
                    g1[i] = __float_as_uint(hb);
                    amax = fmaxf(amax, fmaxf(fabsf(ha), fabsf(hb)));
                }
            }
            if (kFp8) {
                // the row's other 64 columns of the 1x128 group belong to the partner thread
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
                if (valid) {
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
                    uint4* dst =
                        reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) + row * p.I + t.nt * 128 + 64 * half);
#pragma unroll
                    for (int i = 0; i < 4; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                    if (half == 0) p.out_scale[(int64_t)t.nt * p.max_rows + row] = mul_pow2(1.0f, se);
                }
            } else if (busy) {  // this warp's 32 rows x 64 columns of h, staged stores
                uint8_t* hbase = reinterpret_cast<uint8_t*>(static_cast<uint16_t*>(p.out) +
                                                            ((int64_t)t.row0 + (int)rank * kRows + q * 32) * p.I +
                                                            t.nt * 128 + 64 * half);
                uint4* slot = s.oslot + (size_t)(warp - kFirstEpiWarp) * (kOutSlotBytes / 16);
                const int nrows = min(32, my_rows - q * 32);
#pragma unroll
                for (int i = 0; i < 16; ++i) {  // packed in place
                    g0[i] = pack_bf16x2(__uint_as_float(g0[2 * i]), __uint_as_float(g0[2 * i + 1]));
                    g1[i] = pack_bf16x2(__uint_as_float(g1[2 * i]), __uint_as_float(g1[2 * i + 1]));
                }
                store_rows64(slot, g0, hbase, (int64_t)p.I * 2, nrows, lane);
                store_rows64(slot, g1, hbase + 64, (int64_t)p.I * 2, nrows, lane);
            }
        } else {
            uint32_t a[4][32];  // columns 128*half .. +127
            if (busy) {
#pragma unroll
                for (int c = 0; c < 4; ++c) tc::tmem_ld32(tb + 128 * half + 32 * c, a[c]);
                tc::tmem_wait_ld();
            }
            release_acc(s, buf, rank, leader_tempty);
            if (!kFp8 && busy) {  // this warp's 32 rows x 128 columns, staged stores
                uint8_t* ybase = reinterpret_cast<uint8_t*>(static_cast<uint16_t*>(p.out) +
                                                            ((int64_t)t.row0 + (int)rank * kRows + q * 32) * p.H +
                                                            t.nt * kN + 128 * half);
                uint4* slot = s.oslot + (size_t)(warp - kFirstEpiWarp) * (kOutSlotBytes / 16);
                const int nrows = min(32, my_rows - q * 32);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
#pragma unroll
                    for (int i = 0; i < 16; ++i)  // packed in place
                        a[c][i] = pack_bf16x2(__uint_as_float(a[c][2 * i]), __uint_as_float(a[c][2 * i + 1]));
                    store_rows64(slot, a[c], ybase + 64 * c, (int64_t)p.H * 2, nrows, lane);
                }
            } else if (valid) {
                uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + row * p.H + t.nt * kN + 128 * half);
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[4 * c + i] =
                            make_uint4(pack_bf16x2(__uint_as_float(a[c][8 * i]), __uint_as_float(a[c][8 * i + 1])),
                                       pack_bf16x2(__uint_as_float(a[c][8 * i + 2]), __uint_as_float(a[c][8 * i + 3])),
                                       pack_bf16x2(__uint_as_float(a[c][8 * i + 4]), __uint_as_float(a[c][8 * i + 5])),
                                       pack_bf16x2(__uint_as_float(a[c][8 * i + 6]), __uint_as_float(a[c][8 * i + 7])));
            }
        }
        if (++buf == C::AccBufs) {
            buf = 0;
            acc_phase ^= 1u;
        }
    }
    if (!ok) fail(s, p.err);
}

template <bool kUp, bool kFp8>
__global__ void __launch_bounds__(kThreads, 1) ffn_pair_kernel(const __grid_constant__ PairParams p) {
    using C = Cfg<kFp8>;
    extern __shared__ uint8_t smem_raw[];
    const Smem s = carve(smem_raw, C::SfBytes);
    const uint32_t rank = tc::cluster_rank();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            tc::mbar_init(&s.full[i], kFp8 ? 2 : 1);  // leader producer (+ the leader's scale stager)
            tc::mbar_init(&s.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&s.tfull[i], 1);
            tc::mbar_init(&s.tempty[i], 2 * kEpiWarps);
        }
        tc::mbar_init(s.drain, 1);
        tc::mbar_init(s.never, 1);
        *s.abort = 0;
        tc::fence_barrier_init();
        for (int i = 0; i < kNumABoxes; ++i) tc::prefetch_tmap(&p.tmA[i]);
        tc::prefetch_tmap(&p.tmB);
    }
    for (int i = threadIdx.x; i < 256; i += blockDim.x) s.xseq[i] = 0;
    // both CTAs' barriers are initialised before any remote arrival or copy, and both
    // CTAs are running before the pair allocates TMEM
    tc::cluster_sync();
    if (warp == 1) {
        tc::tmem_alloc_pair(s.tmem_base, kTmemCols);
        tc::tmem_relinquish_pair();
    }
    tc::pdl_launch_dependents();
    tc::pdl_wait();  // nothing produced upstream is read before this
    if (warp == 2) scan_tiles(p, s);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem_base = *s.tmem_base;
    const int total = s.tstart[p.NE];

    if (warp == 0) {
        if (lane == 0) producer<kUp, kFp8>(p, s, total, rank);
    } else if (warp == 1) {
        if (lane == 0) {
            if (rank == 0) mma_issuer<kFp8>(p, s, total, tmem_base);
            // every pair MMA (they write both CTAs' TMEM) has completed before TMEM is freed
            const uint64_t t0 = tc::globaltimer();
            while (!tc::mbar_try_wait(s.drain, 0) && tc::globaltimer() - t0 < tc::kWaitTimeoutNs) {
            }
        }
    } else if (warp == 2) {
        if (kFp8 && rank == 0) scale_stager<kUp>(p, s, total);
    } else {
        epilogue<kUp, kFp8>(p, s, total, tmem_base, rank);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::cluster_sync();  // neither CTA's TMEM or shared memory is in use by the pair any more
    tc::tc_fence_after();
    if (warp == 1) tc::tmem_dealloc_pair(tmem_base, kTmemCols);
}

template <bool kUp, bool kFp8>
cudaError_t launch_pair(const PairParams& p, int pairs, cudaStream_t st) {
    auto kern = ffn_pair_kernel<kUp, kFp8>;
    const size_t smem = smem_bytes<kFp8>();
    cudaError_t e = ensure_max_dynamic_smem(kern, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * pairs));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

// MOE_FFN_TILE=pair / single forces one kernel family (tests, measurements).
int tile_override() {
    static int v = -1;
    if (v < 0) {
        const char* e = getenv("MOE_FFN_TILE");
        v = (e && strcmp(e, "pair") == 0) ? 1 : (e && strcmp(e, "single") == 0) ? 2 : 0;
    }
    return v;
}

}  // namespace

bool ffn_pair_supported(const moe_config& c) {
    const DeviceInfo& d = device_info();
    const size_t smem = c.dtype == MOE_FP8_E4M3 ? smem_bytes<true>() : smem_bytes<false>();
    return (c.dtype == MOE_BF16 || c.dtype == MOE_FP8_E4M3) && d.cc_major == 10 && c.hidden % kN == 0 &&
           c.inter % 128 == 0 && d.smem_optin >= smem && tma_encode_fn() != nullptr;
}

// bf16 layers averaging >= 128 rows per expert take the pair tiles (measured 0.90x the
// one-CTA kernel's time on the DeepSeek-V2-Lite-shaped prefill layer).  FP8 layers stay
// on the one-CTA kernels unless forced: the pair kernel must stage each k-block's scale
// factors of both CTAs from one CTA (the proxy fence on the peer's shared memory costs
// ~0.4 us a step), and even without any scale work it only matched the one-CTA kernel on
// the DeepSeek-V3 prefill layer (3.49 vs 3.58 ms), both keeping ~192 KB in flight per SM.
bool ffn_pair_preferred(const moe_config& c, int64_t rows_hint) {
    if (!ffn_pair_supported(c)) return false;
    const int o = tile_override();
    if (o == 1) return true;
    if (o == 2) return false;
    const int64_t NE = c.num_experts + c.num_shared;
    return c.dtype == MOE_BF16 && rows_hint >= 128 * NE;
}

cudaError_t launch_ffn_pair(const moe_config& c, const FfnArgs& a, int grid_cap, cudaStream_t st) {
    const int NE = c.num_experts + c.num_shared;
    const int H = c.hidden, I = c.inter;
    const bool fp8 = c.dtype == MOE_FP8_E4M3;
    int ctas = device_info().num_sms;
    if (ctas > grid_cap) ctas = grid_cap;
    const int pairs = ctas / 2 > 0 ? ctas / 2 : 1;
    void* h = a.ws;
    float* h_scale =
        fp8 ? reinterpret_cast<float*>(static_cast<char*>(a.ws) + align_up((size_t)a.max_rows * I, 256)) : nullptr;
    const int kelems = fp8 ? 128 : 64;
    PairParams up{};
    for (int i = 0; i < kNumABoxes; ++i)
        if (!make_tma_map_2d(&up.tmA[i], a.xe, (uint64_t)H, (uint64_t)a.max_rows, fp8, a_box_rows(i)))
            return cudaErrorInvalidValue;
    if (!make_tma_map_2d(&up.tmB, a.w13, (uint64_t)H, (uint64_t)NE * 2 * I, fp8, 128)) return cudaErrorInvalidValue;
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
    up.a_rs = a.xs_cs ? 1 : H / 128;
    up.a_cs = a.xs_cs ? a.xs_cs : 1;
    up.b_scale = a.w13_scale;
    up.out_scale = h_scale;
    up.inject_ns = wait_injection_ns();
    PairParams dn = up;
    for (int i = 0; i < kNumABoxes; ++i)
        if (!make_tma_map_2d(&dn.tmA[i], h, (uint64_t)I, (uint64_t)a.max_rows, fp8, a_box_rows(i)))
            return cudaErrorInvalidValue;
    if (!make_tma_map_2d(&dn.tmB, a.w2, (uint64_t)I, (uint64_t)NE * H, fp8, 128)) return cudaErrorInvalidValue;
    dn.K = I;
    dn.kblocks = I / kelems;
    dn.NB = H;
    dn.ntn = H / kN;
    dn.out = a.ye;
    dn.a_scale = h_scale;  // written column-major by the up kernel
    dn.a_rs = 1;
    dn.a_cs = a.max_rows;
    dn.b_scale = a.w2_scale;
    dn.out_scale = nullptr;
    cudaError_t e = fp8 ? launch_pair<true, true>(up, pairs, st) : launch_pair<true, false>(up, pairs, st);
    if (e != cudaSuccess) return e;
    return fp8 ? launch_pair<false, true>(dn, pairs, st) : launch_pair<false, false>(dn, pairs, st);
}

}  // namespace moe
