// moe_layer_dbo: the MoE layer on two micro-batches (ubatches) overlapped on a
// compute stream and a comm stream.
//
// The Dual-Batch Overlap mechanism ("[Core/DBO][1/N] Add Dual-Batch Overlap
// mechanism to VLLM", Purpose) runs two host threads that hand the CPU to each
// other at every "yield" and switch streams, so that one ubatch's dispatch /
// combine kernels are enqueued on the comm stream while the other ubatch's expert
// kernels are on the compute stream.  For one layer on one GPU the interleaving
// those yields produce is a fixed order, so a single host thread enqueues it
// directly (the schedule below); the CUDA events between the streams play the part
// of the GPU events of that mechanism.  The dependency rule of "[Perf] Fix DBO
// overlap: capture DeepEP event before yield" (Purpose) is kept by construction:
// every event a comm step waits on is recorded on the compute stream immediately
// after the kernel it stands for, before the other ubatch's compute is enqueued,
// so it covers that ubatch's compute tail only.  The comm stream is joined back to
// the compute stream at the end ("DeepEP HT: full decode CUDA graphs via
// worst-token dispatch", commit messages: dispatch and combine are joined to the
// compute stream), so the whole call is one capturable fork/join.
#include <cuda_runtime.h>

#include <stdint.h>

#include <vector>

#include "kernels.h"
#include "moe.h"

namespace moe {
namespace {

enum { kEvStart = 0, kEvDisp0, kEvFfn0, kEvDisp1, kEvFfn1, kEvDone,
       // stack of layers: stand-in done, dispatch done, FFN done, combine done, per ubatch
       kSevA0, kSevA1, kSevD0, kSevD1, kSevF0, kSevF1, kSevC0, kSevC1, kNumEvents };

struct Op {
    int stream;  // 0 compute, 1 comm
    int op;      // MOE_OP_*
    int ub;      // ubatch or -1
    int ev;      // event id for RECORD / WAIT, else -1
};

// fused (the combine inside the expert FFN's down kernel): there is no combine step, so
// a ubatch's comm side is route, plan (with token_of) and its DISPATCH step (the gather,
// or with the gather fused too, for fp8 the per-token quantisation).
std::vector<Op> make_schedule(bool two, bool fused = false) {
    std::vector<Op> s;
    auto add = [&](int st, int op, int ub, int ev) { s.push_back(Op{st, op, ub, ev}); };
    if (!two) {
        add(0, MOE_OP_ROUTE, 0, -1);
        add(0, MOE_OP_PLAN, 0, -1);
        add(0, MOE_OP_DISPATCH, 0, -1);
        add(0, MOE_OP_FFN, 0, -1);
        if (!fused) add(0, MOE_OP_COMBINE, 0, -1);
        return s;
    }
    if (fused) {
        add(0, MOE_OP_RECORD, -1, kEvStart);
        add(1, MOE_OP_WAIT, -1, kEvStart);
        for (int u = 0; u < 2; ++u) {
            add(1, MOE_OP_ROUTE, u, -1);  // ubatch 1's overlaps the experts of ubatch 0
            add(1, MOE_OP_PLAN, u, -1);
            add(1, MOE_OP_DISPATCH, u, -1);
            add(1, MOE_OP_RECORD, u, u ? kEvDisp1 : kEvDisp0);
            add(0, MOE_OP_WAIT, u, u ? kEvDisp1 : kEvDisp0);
            add(0, MOE_OP_FFN, u, -1);
        }
        add(1, MOE_OP_RECORD, -1, kEvDone);
        add(0, MOE_OP_WAIT, -1, kEvDone);
        return s;
    }
    add(0, MOE_OP_RECORD, -1, kEvStart);  // fork: the comm stream starts after the inputs
    add(1, MOE_OP_WAIT, -1, kEvStart);
    add(1, MOE_OP_ROUTE, 0, -1);          // ubatch 0: dispatch side
    add(1, MOE_OP_PLAN, 0, -1);
    add(1, MOE_OP_DISPATCH, 0, -1);
    add(1, MOE_OP_RECORD, 0, kEvDisp0);
    add(0, MOE_OP_WAIT, 0, kEvDisp0);     // ubatch 0: experts
    add(0, MOE_OP_FFN, 0, -1);
    add(0, MOE_OP_RECORD, 0, kEvFfn0);    // recorded before ubatch 1's compute is enqueued
    add(1, MOE_OP_ROUTE, 1, -1);          // ubatch 1: dispatch side, overlaps FFN(0)
    add(1, MOE_OP_PLAN, 1, -1);
    add(1, MOE_OP_DISPATCH, 1, -1);
    add(1, MOE_OP_RECORD, 1, kEvDisp1);
    add(0, MOE_OP_WAIT, 1, kEvDisp1);     // ubatch 1: experts
    add(0, MOE_OP_FFN, 1, -1);
    add(0, MOE_OP_RECORD, 1, kEvFfn1);
    add(1, MOE_OP_WAIT, 0, kEvFfn0);      // ubatch 0: combine, overlaps FFN(1)
    add(1, MOE_OP_COMBINE, 0, -1);
    add(1, MOE_OP_WAIT, 1, kEvFfn1);      // ubatch 1: combine
    add(1, MOE_OP_COMBINE, 1, -1);
    add(1, MOE_OP_RECORD, -1, kEvDone);
    add(0, MOE_OP_WAIT, -1, kEvDone);     // join: nothing of the layer stays on the comm stream
    return s;
}

// A stack of layers, each = stand-in non-MoE block (A) then the MoE layer: dispatch
// side D (route, plan, dispatch), experts F, combine C.  Compute stream: A0 A1 F0 F1 per
// layer; comm stream: D0 D1 C0 C1.  D(u) waits for A(u), F(u) for D(u), C(u) for F(u),
// A(u) of the next layer for C(u).  With event_before_yield the event a comm step
// waits on is recorded right after the compute kernel it stands for, so D0 overlaps A1,
// D1 overlaps F0, C0 overlaps F1 and C1 overlaps the next layer's A0.  Without it (the
// placement before "[Perf] Fix DBO overlap: capture DeepEP event before yield") the
// event is recorded only after the other ubatch's compute has been enqueued too, so
// D0 also waits for A1 and C0 for F1.
std::vector<Op> make_stack_schedule(int L, bool two, bool before_yield) {
    std::vector<Op> s;
    auto add = [&](int st, int op, int ub, int ev) { s.push_back(Op{st, op, ub, ev}); };
    if (!two) {
        for (int l = 0; l < L; ++l) {
            add(0, MOE_OP_STANDIN, 0, -1);
            add(0, MOE_OP_ROUTE, 0, -1);
            add(0, MOE_OP_PLAN, 0, -1);
            add(0, MOE_OP_DISPATCH, 0, -1);
            add(0, MOE_OP_FFN, 0, -1);
            add(0, MOE_OP_COMBINE, 0, -1);
        }
        return s;
    }
    add(0, MOE_OP_RECORD, -1, kEvStart);
    add(1, MOE_OP_WAIT, -1, kEvStart);
    for (int l = 0; l < L; ++l) {
        if (l > 0) add(0, MOE_OP_WAIT, 0, kSevC0);
        add(0, MOE_OP_STANDIN, 0, -1);
        if (before_yield) add(0, MOE_OP_RECORD, 0, kSevA0);
        if (l > 0) add(0, MOE_OP_WAIT, 1, kSevC1);
        add(0, MOE_OP_STANDIN, 1, -1);
        if (!before_yield) add(0, MOE_OP_RECORD, 0, kSevA0);
        add(0, MOE_OP_RECORD, 1, kSevA1);
        for (int u = 0; u < 2; ++u) {
            add(1, MOE_OP_WAIT, u, u ? kSevA1 : kSevA0);
            add(1, MOE_OP_ROUTE, u, -1);
            add(1, MOE_OP_PLAN, u, -1);
            add(1, MOE_OP_DISPATCH, u, -1);
            add(1, MOE_OP_RECORD, u, u ? kSevD1 : kSevD0);
        }
        add(0, MOE_OP_WAIT, 0, kSevD0);
        add(0, MOE_OP_FFN, 0, -1);
        if (before_yield) add(0, MOE_OP_RECORD, 0, kSevF0);
        add(0, MOE_OP_WAIT, 1, kSevD1);
        add(0, MOE_OP_FFN, 1, -1);
        if (!before_yield) add(0, MOE_OP_RECORD, 0, kSevF0);
        add(0, MOE_OP_RECORD, 1, kSevF1);
        for (int u = 0; u < 2; ++u) {
            add(1, MOE_OP_WAIT, u, u ? kSevF1 : kSevF0);
            add(1, MOE_OP_COMBINE, u, -1);
            add(1, MOE_OP_RECORD, u, u ? kSevC1 : kSevC0);
        }
    }
    add(1, MOE_OP_RECORD, -1, kEvDone);
    add(0, MOE_OP_WAIT, -1, kEvDone);
    return s;
}

// Byte layout of one ubatch's slice of the layer workspace.
struct UbLayout {
    size_t counts, offsets, slot_of, hist, xe, xe_scale, ye, ffn;
    size_t token_of, xq, xq_scale, comb_cnt;  // the fused gather / combine
    size_t total;
    int64_t rows;
};

UbLayout ub_layout(const moe_config& c, int T, int capacity, int align) {
    UbLayout L{};
    const size_t NE = (size_t)c.num_experts + c.num_shared;
    const size_t kk = (size_t)c.top_k + c.num_shared;
    const size_t H = c.hidden;
    L.rows = (int64_t)moe_plan_rows(&c, T, capacity, align);
    size_t o = 0;
    auto take = [&](size_t bytes) {
        size_t at = o;
        o = align_up(o + bytes, 256);
        return at;
    };
    L.counts = take(NE * 4);
    L.offsets = take((NE + 1) * 4);
    L.slot_of = take((size_t)T * kk * 4);
    L.hist = take(moe_plan_workspace_size(&c, T));
    L.xe = take((size_t)L.rows * H * elt_bytes(c.dtype));
    L.xe_scale = take(c.dtype == MOE_FP8_E4M3 ? (size_t)L.rows * (H / 128) * 4 : 0);
    L.ye = take((size_t)L.rows * H * io_bytes(c.dtype));
    L.ffn = take(ffn_scratch_bytes(c, L.rows));
    const bool fp8 = c.dtype == MOE_FP8_E4M3;
    L.token_of = take((size_t)L.rows * 4);
    L.xq = take(fp8 ? (size_t)T * H : 0);
    L.xq_scale = take(fp8 ? (size_t)T * (H / 128) * 4 : 0);
    L.comb_cnt = take((size_t)T * (H / 128) * 4);
    L.total = o;
    return L;
}

}  // namespace
}  // namespace moe

using namespace moe;

struct moe_dbo_handle {
    cudaEvent_t ev[kNumEvents];
    int device;
};

namespace {
// An enqueue failed after the comm stream was forked from the compute stream: join it
// back anyway, so that the comm work already queued (which may still write the
// caller's buffers) is ordered before later work on the compute stream and a capture
// is not left with an unjoined fork.  Best effort: the call reports MOE_ERR_CUDA.
void join_after_failure(moe_dbo_handle* h, cudaStream_t compute, cudaStream_t comm) {
    if (cudaEventRecord(h->ev[kEvDone], comm) == cudaSuccess) cudaStreamWaitEvent(compute, h->ev[kEvDone], 0);
}
}  // namespace

extern "C" {

moe_status moe_dbo_create(moe_dbo_handle** out) {
    if (!out) return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    moe_dbo_handle* h = new moe_dbo_handle();
    cudaGetDevice(&h->device);
    for (int i = 0; i < kNumEvents; ++i) {
        if (cudaEventCreateWithFlags(&h->ev[i], cudaEventDisableTiming) != cudaSuccess) {
            for (int j = 0; j < i; ++j) cudaEventDestroy(h->ev[j]);
            delete h;
            return MOE_ERR_CUDA;
        }
    }
    *out = h;
    return MOE_OK;
}

void moe_dbo_destroy(moe_dbo_handle* h) {
    if (!h) return;
    for (int i = 0; i < kNumEvents; ++i) cudaEventDestroy(h->ev[i]);
    delete h;
}

int32_t moe_dbo_schedule(int32_t two_ubatches, int32_t* ops, int32_t max_ops) {
    return moe_dbo_schedule_ex(two_ubatches, 0, ops, max_ops);
}

int32_t moe_dbo_schedule_ex(int32_t two_ubatches, int32_t flags, int32_t* ops, int32_t max_ops) {
    std::vector<Op> s = make_schedule(two_ubatches != 0, (flags & MOE_LAYER_FUSED_COMBINE) != 0);
    if (ops)
        for (int i = 0; i < (int)s.size() && i < max_ops; ++i) {
            ops[4 * i + 0] = s[i].stream;
            ops[4 * i + 1] = s[i].op;
            ops[4 * i + 2] = s[i].ub;
            ops[4 * i + 3] = s[i].ev;
        }
    return (int32_t)s.size();
}

size_t moe_layer_workspace_size(const moe_config* cfg, int32_t T, int32_t capacity, int32_t align) {
    if (check_config(cfg) != MOE_OK || T < 0 || capacity < 0 || align < 1) return 0;
    // each ubatch slot is sized for all T tokens, so any split fits
    return 256 + 2 * ub_layout(*cfg, T, capacity, align).total;
}

moe_status moe_layer_dbo(moe_dbo_handle* h, const moe_config* cfg, const moe_layer_args* a, int32_t T,
                         int32_t split, int32_t min_tokens, int32_t capacity, int32_t align,
                         int32_t comm_sms, moe_stream_t compute_s, moe_stream_t comm_s) {
    return moe_layer_dbo_ex(h, cfg, a, T, split, min_tokens, capacity, align, comm_sms, 0, compute_s, comm_s);
}

moe_status moe_layer_dbo_ex(moe_dbo_handle* h, const moe_config* cfg, const moe_layer_args* a, int32_t T,
                            int32_t split, int32_t min_tokens, int32_t capacity, int32_t align, int32_t comm_sms,
                            int32_t flags, moe_stream_t compute_s, moe_stream_t comm_s) {
    if (!h || !cfg || !a) return MOE_ERR_INVALID_ARG;
    if (T < 0 || split < 0 || capacity < 0 || align < 1 || comm_sms < 0) return MOE_ERR_INVALID_ARG;
    if (flags & ~MOE_LAYER_FUSED) return MOE_ERR_INVALID_ARG;  // the two fusion bits only
    const moe_status cs_ok = check_config(cfg);
    if (cs_ok != MOE_OK) return cs_ok;
    if (T == 0) return MOE_OK;
    if (!a->logits || !a->x || !a->w13 || !a->w2 || !a->y || !a->topk_ids || !a->topk_w)
        return MOE_ERR_INVALID_ARG;
    if (cfg->dtype == MOE_FP8_E4M3 && (!a->w13_scale || !a->w2_scale)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(a->x) || !aligned16(a->y) || !aligned16(a->w13) || !aligned16(a->w2))
        return MOE_ERR_ALIGNMENT;
    if ((int64_t)moe_plan_rows(cfg, T, capacity, align) > (int64_t)INT32_MAX) return MOE_ERR_INVALID_ARG;
    const size_t need = moe_layer_workspace_size(cfg, T, capacity, align);
    if (!a->workspace || a->workspace_bytes < need) return MOE_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(a->workspace) & 255u) return MOE_ERR_ALIGNMENT;

    const moe_config& c = *cfg;
    cudaStream_t cs = (cudaStream_t)compute_s, ms = (cudaStream_t)comm_s;
    int s = split == 0 ? (T + 1) / 2 : split;
    const bool two = T >= (min_tokens > 2 ? min_tokens : 2) && s > 0 && s < T;
    if (!two) s = T;
    const int t0[2] = {0, s};
    const int tn[2] = {s, T - s};

    const int sms = device_info().num_sms;
    // comm_sms is an SM budget: a comm-side kernel beside an FFN gets as many CTAs as fit
    // on that many SMs (kCommCtasPerSm for the 256-thread kernels, the staged combine's
    // own count), the FFN one CTA on each remaining SM
    // (only when the two streams differ: serialised on one stream nothing runs beside an
    // FFN, and every kernel gets the whole GPU)
    const bool budget = comm_sms > 0 && cs != ms;
    const int comm_cap = budget ? comm_sms * kCommCtasPerSm : sms * 8;
    const int comb_cap = budget ? comm_sms * combine_ctas_per_sm() : sms * 8;
    const int ffn_cap = budget ? (sms - comm_sms > 1 ? sms - comm_sms : 1) : sms * 8;

    char* ws = static_cast<char*>(a->workspace);
    int32_t* err = a->err_flag ? a->err_flag : reinterpret_cast<int32_t*>(ws);
    const UbLayout L = ub_layout(c, T, capacity, align);
    char* ub_base[2] = {ws + 256, ws + 256 + L.total};

    const size_t H = c.hidden;
    const size_t k = c.top_k;
    moe_status st = MOE_OK;
    cudaError_t ce = cudaMemsetAsync(err, 0, sizeof(int32_t), cs);
    if (ce != cudaSuccess) return MOE_ERR_CUDA;

    // the fused gather / combine is served by the tensor-core FFN (bf16 and fp8 layers);
    // other layers run the steps unfused
    const bool tc = ffn_tc_selected(c);
    const bool fgather = (flags & MOE_LAYER_FUSED_GATHER) && tc;
    const bool fcombine = (flags & MOE_LAYER_FUSED_COMBINE) && tc;
    const bool fused = fgather || fcombine;  // the plan records token_of
    bool forked = false;  // the comm stream has been forked from the compute stream
    for (const Op& op : make_schedule(two, fcombine)) {
        cudaStream_t q = op.stream == 0 ? cs : ms;
        const int u = op.ub < 0 ? 0 : op.ub;
        char* b = ub_base[u];
        int32_t* counts = reinterpret_cast<int32_t*>(b + L.counts);
        int32_t* offsets = reinterpret_cast<int32_t*>(b + L.offsets);
        int32_t* slot_of = reinterpret_cast<int32_t*>(b + L.slot_of);
        void* xe = b + L.xe;
        float* xe_scale = c.dtype == MOE_FP8_E4M3 ? reinterpret_cast<float*>(b + L.xe_scale) : nullptr;
        void* ye = b + L.ye;
        const int Tu = tn[u];
        // the SM budget applies to the comm-side steps that overlap an FFN (ubatch 1's
        // route / plan / dispatch, ubatch 0's combine); ubatch 0's first steps and
        // ubatch 1's combine run alone and get the whole GPU
        const bool overlapped = (u == 1 && op.op != MOE_OP_COMBINE) || (u == 0 && op.op == MOE_OP_COMBINE);
        const int comm_grid = (two && overlapped) ? (op.op == MOE_OP_COMBINE ? comb_cap : comm_cap) : sms * 8;
        const int ffn_grid = two ? ffn_cap : sms * 8;
        // the clustered head (clusters of up to 8 CTAs) only where nothing else runs: beside
        // an FFN the free SMs are scattered over the GPCs and a cluster might not fit
        const bool cluster_head = !fused && !(two && overlapped) && head_fusable(c, Tu);
        int32_t* token_of = reinterpret_cast<int32_t*>(b + L.token_of);
        const char* xu = static_cast<const char*>(a->x) + (size_t)t0[u] * H * io_bytes(c.dtype);
        void* xq = b + L.xq;
        float* xq_scale = reinterpret_cast<float*>(b + L.xq_scale);
        const float* logits_u = a->logits + (size_t)t0[u] * c.num_experts;
        int32_t* ids_u = a->topk_ids + (size_t)t0[u] * k;
        float* w_u = a->topk_w + (size_t)t0[u] * k;
        switch (op.op) {
            case MOE_OP_RECORD: ce = cudaEventRecord(h->ev[op.ev], q); break;
            case MOE_OP_WAIT: ce = cudaStreamWaitEvent(q, h->ev[op.ev], 0); break;
            case MOE_OP_ROUTE:
                if (cluster_head) {  // small batch running alone: route, plan and dispatch in one launch
                    ce = launch_route_plan_dispatch(c, Tu, logits_u, a->bias, ids_u, w_u, capacity, align, counts,
                                                    offsets, slot_of, err, xu, xe, xe_scale, L.rows, comm_grid, q);
                } else {
                    ce = launch_route(c, Tu, logits_u, a->bias, ids_u, w_u, comm_grid, q);
                }
                break;
            case MOE_OP_PLAN:
                if (cluster_head) break;             // done with the route
                if (fused) {                         // the FFN gathers by token: token_of wanted
                    ce = launch_plan(c, Tu, ids_u, capacity, align, counts, offsets, slot_of, token_of, err,
                                     reinterpret_cast<int32_t*>(b + L.hist), comm_grid, q);
                    break;
                }
                if (plan_dispatch_fusable(c, Tu)) {  // single-chunk batch: plan and dispatch in one launch
                    ce = launch_plan_dispatch(c, Tu, ids_u, capacity, align, counts, offsets, slot_of, err, xu, xe,
                                              xe_scale, L.rows, comm_grid, q);
                } else {
                    ce = launch_plan(c, Tu, ids_u, capacity, align, counts, offsets, slot_of, nullptr, err,
                                     reinterpret_cast<int32_t*>(b + L.hist), comm_grid, q);
                }
                break;
            case MOE_OP_DISPATCH: {
                if (fgather) {  // fp8: each token's row quantised once; bf16: nothing to move
                    if (c.dtype == MOE_FP8_E4M3)
                        ce = launch_quantize_rows(c, Tu, xu, xq, xq_scale, Tu, comm_grid, q);
                    break;
                }
                if (!fused && plan_dispatch_fusable(c, Tu)) break;  // done with the plan
                ce = launch_dispatch(c, Tu, xu, slot_of, xe, xe_scale, L.rows, comm_grid, q);
                break;
            }
            case MOE_OP_FFN: {
                FfnArgs fa{counts, offsets, L.rows, xe, xe_scale, a->w13, a->w13_scale, a->w2, a->w2_scale,
                           ye, b + L.ffn, err, two && u == 1 ? 1 : 0, L.rows, (int64_t)Tu * (c.top_k + c.num_shared)};
                if (fused) {
                    fa.token_of = token_of;
                    fa.gT = Tu;
                }
                if (fgather) {
                    fa.gx = c.dtype == MOE_FP8_E4M3 ? static_cast<const void*>(xq) : static_cast<const void*>(xu);
                    fa.gx_scale = c.dtype == MOE_FP8_E4M3 ? xq_scale : nullptr;
                }
                if (fcombine) {
                    fa.slot_of = slot_of;
                    fa.topk_w = w_u;
                    fa.y = static_cast<char*>(a->y) + (size_t)t0[u] * H * io_bytes(c.dtype);
                    fa.cnt = reinterpret_cast<int32_t*>(b + L.comb_cnt);
                    // shared experts first: a token's shared row is then never the last of
                    // its rows, and the slabs completed per tile stay few
                    fa.reverse = 1;
                }
                ce = launch_ffn(c, fa, ffn_grid, q);
                break;
            }
            case MOE_OP_COMBINE: {
                char* yu = static_cast<char*>(a->y) + (size_t)t0[u] * H * io_bytes(c.dtype);
                ce = launch_combine(c, Tu, ye, w_u, slot_of, yu, comm_grid, q, nullptr, err);
                break;
            }
        }
        if (ce != cudaSuccess) {
            st = MOE_ERR_CUDA;
            break;
        }
        if (op.op == MOE_OP_WAIT && op.ev == kEvStart) forked = true;
    }
    if (st != MOE_OK && forked) join_after_failure(h, cs, ms);
    return st;
}


int32_t moe_stack_schedule(int32_t layers, int32_t two_ubatches, int32_t event_before_yield, int32_t* ops,
                           int32_t max_ops) {
    if (layers < 1) return 0;
    std::vector<Op> s = make_stack_schedule(layers, two_ubatches != 0, event_before_yield != 0);
    if (ops)
        for (int i = 0; i < (int)s.size() && i < max_ops; ++i) {
            ops[4 * i + 0] = s[i].stream;
            ops[4 * i + 1] = s[i].op;
            ops[4 * i + 2] = s[i].ub;
            ops[4 * i + 3] = s[i].ev;
        }
    return (int32_t)s.size();
}

namespace {
struct StackLayout {
    UbLayout ub;
    size_t ub_base[2], a[2], ids[2], w[2], pp[2], total;
};
StackLayout stack_layout(const moe_config& c, int T, int capacity, int align) {
    StackLayout S{};
    S.ub = ub_layout(c, T, capacity, align);
    const size_t act = align_up((size_t)T * c.hidden * io_bytes(c.dtype), 256);
    const size_t ids = align_up((size_t)T * c.top_k * 4, 256);
    size_t o = 256;  // error flag
    for (int u = 0; u < 2; ++u) {
        S.ub_base[u] = o;
        o += S.ub.total;
    }
    for (int u = 0; u < 2; ++u) {
        S.a[u] = o;
        o += act;
        S.ids[u] = o;
        o += ids;
        S.w[u] = o;
        o += ids;
        S.pp[u] = o;
        o += act;
    }
    S.total = o;
    return S;
}
}  // namespace

size_t moe_stack_workspace_size(const moe_config* cfg, int32_t T, int32_t capacity, int32_t align) {
    if (check_config(cfg) != MOE_OK || T < 0 || capacity < 0 || align < 1) return 0;
    return stack_layout(*cfg, T, capacity, align).total;
}

moe_status moe_stack_dbo(moe_dbo_handle* h, const moe_config* cfg, const moe_stack_args* a, int32_t L, int32_t T,
                         int32_t split, int32_t min_tokens, int32_t capacity, int32_t align, int32_t comm_sms,
                         int32_t event_before_yield, moe_stream_t compute_s, moe_stream_t comm_s) {
    if (!h || !cfg || !a) return MOE_ERR_INVALID_ARG;
    if (L < 1 || T < 0 || split < 0 || capacity < 0 || align < 1 || comm_sms < 0) return MOE_ERR_INVALID_ARG;
    const moe_status cs_ok = check_config(cfg);
    if (cs_ok != MOE_OK) return cs_ok;
    if (!standin_tc_supported(*cfg)) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    if (!a->x || !a->out || !a->logits || !a->wa || !a->w13 || !a->w2) return MOE_ERR_INVALID_ARG;
    const bool fp8 = cfg->dtype == MOE_FP8_E4M3;
    for (int l = 0; l < L; ++l) {
        if (!a->logits[l] || !a->wa[l] || !a->w13[l] || !a->w2[l]) return MOE_ERR_INVALID_ARG;
        if (fp8 && (!a->w13_scale || !a->w2_scale || !a->w13_scale[l] || !a->w2_scale[l])) return MOE_ERR_INVALID_ARG;
        if (!aligned16(a->wa[l]) || !aligned16(a->w13[l]) || !aligned16(a->w2[l])) return MOE_ERR_ALIGNMENT;
    }
    if (!aligned16(a->x) || !aligned16(a->out)) return MOE_ERR_ALIGNMENT;
    if ((int64_t)moe_plan_rows(cfg, T, capacity, align) > (int64_t)INT32_MAX) return MOE_ERR_INVALID_ARG;
    const StackLayout S = stack_layout(*cfg, T, capacity, align);
    if (!a->workspace || a->workspace_bytes < S.total) return MOE_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(a->workspace) & 255u) return MOE_ERR_ALIGNMENT;

    const moe_config& c = *cfg;
    cudaStream_t cs = (cudaStream_t)compute_s, ms = (cudaStream_t)comm_s;
    int s = split == 0 ? (T + 1) / 2 : split;
    const bool two = T >= (min_tokens > 2 ? min_tokens : 2) && s > 0 && s < T;
    if (!two) s = T;
    const int t0[2] = {0, s};
    const int tn[2] = {s, T - s};
    const int sms = device_info().num_sms;
    const bool budget = comm_sms > 0 && cs != ms;  // as in moe_layer_dbo_ex
    const int comm_cap = budget ? comm_sms * kCommCtasPerSm : sms * 8;
    const int comb_cap = budget ? comm_sms * combine_ctas_per_sm() : sms * 8;
    const int ffn_cap = budget ? (sms - comm_sms > 1 ? sms - comm_sms : 1) : sms * 8;
    char* ws = static_cast<char*>(a->workspace);
    int32_t* err = a->err_flag ? a->err_flag : reinterpret_cast<int32_t*>(ws);
    const UbLayout& U = S.ub;
    const size_t H = c.hidden, rowb = H * io_bytes(c.dtype);
    if (cudaMemsetAsync(err, 0, sizeof(int32_t), cs) != cudaSuccess) return MOE_ERR_CUDA;

    int layer[2] = {-1, -1};  // current layer of each ubatch (advanced by its stand-in)
    bool forked = false;      // the comm stream has been forked from the compute stream
    for (const Op& op : make_stack_schedule(L, two, event_before_yield != 0)) {
        cudaStream_t q = op.stream == 0 ? cs : ms;
        const int u = op.ub < 0 ? 0 : op.ub;
        if (op.op == MOE_OP_STANDIN) ++layer[u];
        const int l = layer[u] < 0 ? 0 : layer[u];
        char* b = ws + S.ub_base[u];
        int32_t* counts = reinterpret_cast<int32_t*>(b + U.counts);
        int32_t* offsets = reinterpret_cast<int32_t*>(b + U.offsets);
        int32_t* slot_of = reinterpret_cast<int32_t*>(b + U.slot_of);
        void* xe = b + U.xe;
        float* xe_scale = fp8 ? reinterpret_cast<float*>(b + U.xe_scale) : nullptr;
        void* ye = b + U.ye;
        int32_t* ids = reinterpret_cast<int32_t*>(ws + S.ids[u]);
        float* wts = reinterpret_cast<float*>(ws + S.w[u]);
        char* act = ws + S.a[u];  // the stand-in's output (rows of this ubatch from 0)
        // layer input / output rows of this ubatch
        const char* xin = l == 0 ? static_cast<const char*>(a->x) + t0[u] * rowb
                                 : ws + S.pp[(l - 1) % 2] + t0[u] * rowb;
        char* xout = l == L - 1 ? static_cast<char*>(a->out) + t0[u] * rowb : ws + S.pp[l % 2] + t0[u] * rowb;
        const int Tu = tn[u];
        // the SM budget applies where a comm step runs beside an FFN: ubatch 1's route,
        // plan and dispatch (beside F0) and ubatch 0's combine (beside F1).  Ubatch 0's
        // head and ubatch 1's combine run beside a stand-in block only and take the GPU.
        const bool beside_ffn = two && (op.op == MOE_OP_COMBINE ? u == 0 : u == 1);
        const int comm_grid = beside_ffn ? (op.op == MOE_OP_COMBINE ? comb_cap : comm_cap) : sms * 8;
        const int ffn_grid = two ? ffn_cap : sms * 8;
        cudaError_t ce = cudaSuccess;
        switch (op.op) {
            case MOE_OP_RECORD: ce = cudaEventRecord(h->ev[op.ev], q); break;
            case MOE_OP_WAIT: ce = cudaStreamWaitEvent(q, h->ev[op.ev], 0); break;
            case MOE_OP_STANDIN: ce = launch_standin(c, Tu, xin, a->wa[l], act, ffn_grid, q); break;
            case MOE_OP_ROUTE:
                ce = launch_route(c, Tu, a->logits[l] + (size_t)t0[u] * c.num_experts, a->bias, ids, wts, comm_grid, q);
                break;
            case MOE_OP_PLAN:
                if (plan_dispatch_fusable(c, Tu))
                    ce = launch_plan_dispatch(c, Tu, ids, capacity, align, counts, offsets, slot_of, err, act, xe,
                                              xe_scale, U.rows, comm_grid, q);
                else
                    ce = launch_plan(c, Tu, ids, capacity, align, counts, offsets, slot_of, nullptr, err,
                                     reinterpret_cast<int32_t*>(b + U.hist), comm_grid, q);
                break;
            case MOE_OP_DISPATCH:
                if (!plan_dispatch_fusable(c, Tu))
                    ce = launch_dispatch(c, Tu, act, slot_of, xe, xe_scale, U.rows, comm_grid, q);
                break;
            case MOE_OP_FFN: {
                FfnArgs fa{counts, offsets, U.rows, xe, xe_scale, a->w13[l], fp8 ? a->w13_scale[l] : nullptr, a->w2[l],
                           fp8 ? a->w2_scale[l] : nullptr, ye, b + U.ffn, err, two && u == 1 ? 1 : 0, U.rows,
                           (int64_t)Tu * (c.top_k + c.num_shared)};
                ce = launch_ffn(c, fa, ffn_grid, q);
                break;
            }
            case MOE_OP_COMBINE: ce = launch_combine(c, Tu, ye, wts, slot_of, xout, comm_grid, q, act, err); break;
        }
        if (ce != cudaSuccess) {
            if (forked) join_after_failure(h, cs, ms);
            return MOE_ERR_CUDA;
        }
        if (op.op == MOE_OP_WAIT && op.ev == kEvStart) forked = true;
    }
    return MOE_OK;
}

}  // extern "C"
