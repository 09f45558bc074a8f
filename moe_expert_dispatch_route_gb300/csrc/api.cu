// C ABI of libmoe_gb300: argument validation, workspace layout and the
// Dual-Batch Overlap schedule.  Every computing step runs in the kernels of this
// library; this file only checks arguments and enqueues.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "moe.h"

namespace moe {

const DeviceInfo& device_info() {
    static thread_local DeviceInfo cache[16];
    static thread_local bool ready[16] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 16) dev = 0;
    if (!ready[dev]) {
        DeviceInfo d{};
        d.device = dev;
        cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
        int optin = 0;
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        d.smem_optin = (size_t)optin;
        if (d.num_sms <= 0) d.num_sms = 1;
        cache[dev] = d;
        ready[dev] = true;
    }
    return cache[dev];
}

namespace {

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <typename F>
F driver_fn(const char* name) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<F>(f);
}

}  // namespace

unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) {
        int dev = 0;  // no context on this thread yet: make the device's primary context current
        if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess) return 0;
        if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    }
    unsigned long long id = 0;
    return get_id(ctx, &id) == CUDA_SUCCESS ? id : 0;
}

cudaError_t ensure_max_dynamic_smem(const void* func, int bytes) {
    struct Entry {
        const void* func;
        unsigned long long ctx;
        int bytes;
    };
    static std::mutex mu;
    static std::vector<Entry> done;
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lk(mu);
    if (ctx != 0)
        for (const Entry& e : done)
            if (e.func == func && e.ctx == ctx && e.bytes >= bytes) return cudaSuccess;
    cudaError_t err = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (err == cudaSuccess && ctx != 0) done.push_back(Entry{func, ctx, bytes});
    return err;
}

namespace {
std::atomic<long long> g_inject_wait_ns{0};

// Sticky error word of the staged dispatch / combine kernels called without a caller
// flag (moe_dispatch, moe_combine).
__device__ int32_t g_comm_error;

constexpr int kMaxDevices = 64;
std::mutex g_comm_mu;
struct CommWord {
    unsigned long long ctx;  // context the address was looked up in
    int32_t* ptr;
};
CommWord g_comm_word[kMaxDevices] = {};
}  // namespace

int64_t wait_injection_ns() { return g_inject_wait_ns.load(std::memory_order_relaxed); }

// The address of g_comm_error is looked up with the device current, once per context
// (a device reset followed by a new context gets a fresh lookup).
int32_t* comm_error_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lk(g_comm_mu);
    if (!g_comm_word[dev].ptr || ctx == 0 || g_comm_word[dev].ctx != ctx) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_comm_error) != cudaSuccess) return nullptr;
        g_comm_word[dev] = CommWord{ctx, static_cast<int32_t*>(p)};
    }
    return g_comm_word[dev].ptr;
}

namespace {

int grid_cap_of(int max_ctas) {
    const int sms = device_info().num_sms;
    return max_ctas > 0 ? max_ctas : sms * 8;
}

moe_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return MOE_OK;
    if (getenv("MOE_DEBUG")) fprintf(stderr, "libmoe_gb300: CUDA error %s\n", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
}

}  // namespace

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status check_config(const moe_config* c) {
    if (!c) return MOE_ERR_INVALID_ARG;
    const int E = c->num_experts, S = c->num_shared, k = c->top_k;
    if (c->hidden <= 0 || c->inter <= 0 || E <= 0 || S < 0 || k <= 0) return MOE_ERR_INVALID_ARG;
    if (k > E || k > 32 || k + S > kMaxSlotsPerToken || E + S > kMaxExperts) return MOE_ERR_INVALID_ARG;
    if (c->dtype != MOE_F32 && c->dtype != MOE_BF16 && c->dtype != MOE_FP8_E4M3) return MOE_ERR_INVALID_ARG;
    if (c->gate == MOE_GATE_SIGMOID_GROUPED || c->gate == MOE_GATE_SQRT_SOFTPLUS) {
        const int G = c->n_group, TG = c->topk_group;
        if (G <= 0 || G > 32 || E % G != 0 || E / G < 2 || TG <= 0 || TG > G || k > TG * (E / G))
            return MOE_ERR_INVALID_ARG;
    } else if (c->gate != MOE_GATE_SOFTMAX) {
        return MOE_ERR_INVALID_ARG;
    }
    // rows of x / xe / h / ye / y must be whole 16-byte vectors
    if ((size_t)c->hidden * io_bytes(c->dtype) % 16 || (size_t)c->hidden * elt_bytes(c->dtype) % 16 ||
        (size_t)c->inter * elt_bytes(c->dtype) % 16)
        return MOE_ERR_ALIGNMENT;
    if (c->dtype == MOE_FP8_E4M3 && (c->hidden % kQG || c->inter % kQG)) return MOE_ERR_ALIGNMENT;
    return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" {

moe_status moe_debug_inject_wait(int32_t enable, int64_t timeout_ns) {
    if (enable && timeout_ns <= 0) return MOE_ERR_INVALID_ARG;
    g_inject_wait_ns.store(enable ? (long long)timeout_ns : 0, std::memory_order_relaxed);
    return MOE_OK;
}

moe_status moe_comm_error(int32_t* code, int32_t clear) {
    if (!code) return MOE_ERR_INVALID_ARG;
    int32_t* word = comm_error_word();
    if (!word) return MOE_ERR_CUDA;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(code, word, sizeof(int32_t), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess && clear) e = cudaMemset(word, 0, sizeof(int32_t));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    return cuda_status(e);
}

const char* moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED: return "unsupported";
        case MOE_ERR_ALIGNMENT: return "misaligned buffer or row size";
        case MOE_ERR_WORKSPACE: return "workspace missing or too small";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_CAPACITY: return "expert capacity exceeded";
        case MOE_ERR_BAD_INDEX: return "expert index out of range";
        case MOE_ERR_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

moe_status moe_route(const moe_config* cfg, int32_t T, const float* logits, const float* bias,
                     int32_t* topk_ids, float* topk_w, int32_t max_ctas, moe_stream_t stream) {
    moe_status s = check_config(cfg);
    if (s != MOE_OK) return s;
    if (T < 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!logits || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_route(*cfg, T, logits, bias, topk_ids, topk_w, grid_cap_of(max_ctas),
                                    (cudaStream_t)stream));
}

moe_status moe_route_hash(const moe_config* cfg, int32_t T, const float* logits, const int32_t* token_ids,
                          const int32_t* table, int32_t vocab, int32_t* topk_ids, float* topk_w, int32_t max_ctas,
                          moe_stream_t stream) {
    moe_status s = check_config(cfg);
    if (s != MOE_OK) return s;
    if (cfg->gate != MOE_GATE_SQRT_SOFTPLUS) return MOE_ERR_UNSUPPORTED;
    if (T < 0 || vocab < 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!logits || !token_ids || !topk_ids || !topk_w || (vocab > 0 && !table)) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_route_hash(*cfg, T, logits, token_ids, table, vocab, topk_ids, topk_w,
                                         grid_cap_of(max_ctas), (cudaStream_t)stream));
}

size_t moe_plan_rows(const moe_config* cfg, int32_t T, int32_t capacity, int32_t align) {
    if (check_config(cfg) != MOE_OK || T < 0 || capacity < 0) return 0;
    const size_t NE = (size_t)cfg->num_experts + cfg->num_shared;
    if (capacity > 0) return NE * (size_t)capacity;
    if (align < 1) return 0;
    return (size_t)T * (cfg->top_k + cfg->num_shared) + NE * (size_t)(align - 1);
}

size_t moe_plan_workspace_size(const moe_config* cfg, int32_t T) {
    if (check_config(cfg) != MOE_OK || T < 0) return 0;
    const int nchunks = plan_num_chunks(*cfg, T);
    if (nchunks <= 1) return 0;
    return (size_t)nchunks * (cfg->num_experts + cfg->num_shared) * sizeof(int32_t);
}

moe_status moe_plan(const moe_config* cfg, int32_t T, const int32_t* topk_ids, int32_t capacity,
                    int32_t align, int32_t* counts, int32_t* offsets, int32_t* slot_of,
                    int32_t* token_of, int32_t* err_flag, void* ws, size_t ws_bytes,
                    int32_t max_ctas, moe_stream_t stream) {
    moe_status s = check_config(cfg);
    if (s != MOE_OK) return s;
    if (T < 0 || capacity < 0 || align < 1) return MOE_ERR_INVALID_ARG;
    if (!counts || !offsets || !err_flag || (T > 0 && (!topk_ids || !slot_of))) return MOE_ERR_INVALID_ARG;
    if ((int64_t)moe_plan_rows(cfg, T, capacity, align) > (int64_t)INT32_MAX) return MOE_ERR_INVALID_ARG;
    const size_t need = moe_plan_workspace_size(cfg, T);
    if (need > 0 && (!ws || ws_bytes < need)) return MOE_ERR_WORKSPACE;
    if (ws && (reinterpret_cast<uintptr_t>(ws) & 3u)) return MOE_ERR_ALIGNMENT;
    return cuda_status(launch_plan(*cfg, T, topk_ids, capacity, align, counts, offsets, slot_of, token_of,
                                   err_flag, static_cast<int32_t*>(ws), grid_cap_of(max_ctas),
                                   (cudaStream_t)stream));
}

moe_status moe_dispatch(const moe_config* cfg, int32_t T, const void* x, const int32_t* slot_of,
                        void* xe, float* xe_scale, int64_t xe_scale_ld, int32_t max_ctas,
                        moe_stream_t stream) {
    moe_status s = check_config(cfg);
    if (s != MOE_OK) return s;
    if (T < 0 || xe_scale_ld < 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!x || !slot_of || !xe || (cfg->dtype == MOE_FP8_E4M3 && !xe_scale)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(xe)) return MOE_ERR_ALIGNMENT;
    return cuda_status(launch_dispatch(*cfg, T, x, slot_of, xe, xe_scale, xe_scale_ld, grid_cap_of(max_ctas),
                                       (cudaStream_t)stream));
}

size_t moe_ffn_workspace_size(const moe_config* cfg, int64_t max_rows) {
    if (check_config(cfg) != MOE_OK || max_rows < 0) return 0;
    return ffn_scratch_bytes(*cfg, max_rows);
}

moe_status moe_expert_ffn(const moe_config* cfg, const int32_t* counts, const int32_t* offsets,
                          int64_t max_rows, const void* xe, const float* xe_scale, int64_t xe_scale_ld,
                          const void* w13, const float* w13_scale, const void* w2, const float* w2_scale,
                          void* ye, void* ws, size_t ws_bytes, int32_t* err_flag, int32_t max_ctas,
                          moe_stream_t stream) {
    moe_status s = check_config(cfg);
    if (s != MOE_OK) return s;
    if (max_rows < 0 || max_rows > INT32_MAX) return MOE_ERR_INVALID_ARG;
    if (max_rows == 0) return MOE_OK;
    if (!counts || !offsets || !xe || !w13 || !w2 || !ye) return MOE_ERR_INVALID_ARG;
    const bool fp8 = cfg->dtype == MOE_FP8_E4M3;
    if (fp8 && (!xe_scale || !w13_scale || !w2_scale)) return MOE_ERR_INVALID_ARG;
    if (xe_scale_ld < 0 || (xe_scale_ld > 0 && xe_scale_ld < max_rows)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(xe) || !aligned16(w13) || !aligned16(w2) || !aligned16(ye)) return MOE_ERR_ALIGNMENT;
    const size_t need = ffn_scratch_bytes(*cfg, max_rows);
    if (!ws || ws_bytes < need) return MOE_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(ws) & 255u) return MOE_ERR_ALIGNMENT;
    FfnArgs a{counts, offsets, max_rows, xe, xe_scale, w13, w13_scale, w2, w2_scale, ye, ws, err_flag, 0,
              xe_scale_ld};
    return cuda_status(launch_ffn(*cfg, a, grid_cap_of(max_ctas), (cudaStream_t)stream));
}

moe_status moe_combine(const moe_config* cfg, int32_t T, const void* ye, const float* topk_w,
                       const int32_t* slot_of, void* y, int32_t max_ctas, moe_stream_t stream) {
    moe_status s = check_config(cfg);
    if (s != MOE_OK) return s;
    if (T < 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!ye || !topk_w || !slot_of || !y) return MOE_ERR_INVALID_ARG;
    if (!aligned16(ye) || !aligned16(y)) return MOE_ERR_ALIGNMENT;
    return cuda_status(launch_combine(*cfg, T, ye, topk_w, slot_of, y, grid_cap_of(max_ctas),
                                      (cudaStream_t)stream));
}

}  // extern "C"
