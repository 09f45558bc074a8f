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

enum { kEvStart = 0, kEvDisp0, kEvFfn0, kEvDisp1, kEvFfn1, kEvDone, kNumEvents };

struct Op {
    int stream;  // 0 compute, 1 comm
    int op;      // MOE_OP_*
    int ub;      // ubatch or -1
    int ev;      // event id for RECORD / WAIT, else -1
};

std::vector<Op> make_schedule(bool two) {
    std::vector<Op> s;
    auto add = [&](int st, int op, int ub, int ev) { s.push_back(Op{st, op, ub, ev}); };
    if (!two) {
        add(0, MOE_OP_ROUTE, 0, -1);
        add(0, MOE_OP_PLAN, 0, -1);
        add(0, MOE_OP_DISPATCH, 0, -1);
        add(0, MOE_OP_FFN, 0, -1);
        add(0, MOE_OP_COMBINE, 0, -1);
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

// Byte layout of one ubatch's slice of the layer workspace.
struct UbLayout {
    size_t counts, offsets, slot_of, token_of, hist, xe, xe_scale, ye, ffn, total;
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
    L.token_of = take((size_t)L.rows * 4);
    L.hist = take(moe_plan_workspace_size(&c, T));
    L.xe = take((size_t)L.rows * H * elt_bytes(c.dtype));
    L.xe_scale = take(c.dtype == MOE_FP8_E4M3 ? (size_t)L.rows * (H / 128) * 4 : 0);
    L.ye = take((size_t)L.rows * H * io_bytes(c.dtype));
    L.ffn = take(ffn_scratch_bytes(c, L.rows));
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
    std::vector<Op> s = make_schedule(two_ubatches != 0);
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
    if (!h || !cfg || !a) return MOE_ERR_INVALID_ARG;
    if (T < 0 || split < 0 || capacity < 0 || align < 1 || comm_sms < 0) return MOE_ERR_INVALID_ARG;
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
    const int comm_cap = comm_sms > 0 ? comm_sms : sms * 8;
    const int ffn_cap = comm_sms > 0 ? (sms - comm_sms > 1 ? sms - comm_sms : 1) : sms * 8;

    char* ws = static_cast<char*>(a->workspace);
    int32_t* err = a->err_flag ? a->err_flag : reinterpret_cast<int32_t*>(ws);
    const UbLayout L = ub_layout(c, T, capacity, align);
    char* ub_base[2] = {ws + 256, ws + 256 + L.total};

    const size_t H = c.hidden;
    const size_t k = c.top_k;
    moe_status st = MOE_OK;
    cudaError_t ce = cudaMemsetAsync(err, 0, sizeof(int32_t), cs);
    if (ce != cudaSuccess) return MOE_ERR_CUDA;

    for (const Op& op : make_schedule(two)) {
        cudaStream_t q = op.stream == 0 ? cs : ms;
        const int u = op.ub < 0 ? 0 : op.ub;
        char* b = ub_base[u];
        int32_t* counts = reinterpret_cast<int32_t*>(b + L.counts);
        int32_t* offsets = reinterpret_cast<int32_t*>(b + L.offsets);
        int32_t* slot_of = reinterpret_cast<int32_t*>(b + L.slot_of);
        int32_t* token_of = reinterpret_cast<int32_t*>(b + L.token_of);
        void* xe = b + L.xe;
        float* xe_scale = c.dtype == MOE_FP8_E4M3 ? reinterpret_cast<float*>(b + L.xe_scale) : nullptr;
        void* ye = b + L.ye;
        const int Tu = tn[u];
        const int comm_grid = two ? comm_cap : sms * 8;
        const int ffn_grid = two ? ffn_cap : sms * 8;
        const float* logits_u = a->logits + (size_t)t0[u] * c.num_experts;
        int32_t* ids_u = a->topk_ids + (size_t)t0[u] * k;
        float* w_u = a->topk_w + (size_t)t0[u] * k;
        switch (op.op) {
            case MOE_OP_RECORD: ce = cudaEventRecord(h->ev[op.ev], q); break;
            case MOE_OP_WAIT: ce = cudaStreamWaitEvent(q, h->ev[op.ev], 0); break;
            case MOE_OP_ROUTE: ce = launch_route(c, Tu, logits_u, a->bias, ids_u, w_u, comm_grid, q); break;
            case MOE_OP_PLAN:
                ce = launch_plan(c, Tu, ids_u, capacity, align, counts, offsets, slot_of, token_of, err,
                                 reinterpret_cast<int32_t*>(b + L.hist), comm_grid, q);
                break;
            case MOE_OP_DISPATCH: {
                const char* xu = static_cast<const char*>(a->x) + (size_t)t0[u] * H * io_bytes(c.dtype);
                ce = launch_dispatch(c, Tu, xu, slot_of, xe, xe_scale, comm_grid, q);
                break;
            }
            case MOE_OP_FFN: {
                FfnArgs fa{counts, offsets, L.rows, xe, xe_scale, a->w13, a->w13_scale, a->w2, a->w2_scale,
                           ye, b + L.ffn, err, two && u == 1 ? 1 : 0};
                ce = launch_ffn(c, fa, ffn_grid, q);
                break;
            }
            case MOE_OP_COMBINE: {
                char* yu = static_cast<char*>(a->y) + (size_t)t0[u] * H * io_bytes(c.dtype);
                ce = launch_combine(c, Tu, ye, w_u, slot_of, yu, comm_grid, q);
                break;
            }
        }
        if (ce != cudaSuccess) {
            st = MOE_ERR_CUDA;
            break;
        }
    }
    return st;
}

}  // extern "C"
