// moe_plan_noalloc: moe_plan for callers that cannot allocate device memory.
//
// The plan's only scratch is the per-chunk expert histograms of large batches.
// Here that scratch is a fixed array in the library's own device memory, so the
// caller passes only inputs and outputs.  The array is a file-scope __device__
// variable: every GPU that loads the library holds it until the process exits.
#include <cuda_runtime.h>
#include <stdio.h>
#include <stdlib.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "moe.h"

namespace moe {
namespace {

constexpr int kNoAllocScratchInts = 65536;  // 256 KiB of chunk histograms
static __device__ __align__(256) int32_t g_plan_scratch[kNoAllocScratchInts];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct ScratchAddr {
    unsigned long long ctx;  // context the address was looked up in
    int32_t* ptr;
};
ScratchAddr g_scratch[kMaxDevices] = {};

// Device address of g_plan_scratch in the context current on this thread.  The
// host-side name of the array is only a stand-in, so the address is looked up with
// the device current, once per context: a device reset followed by a new context
// gets a fresh lookup instead of a stale address.
int32_t* scratch_for_current_device(cudaError_t* err) {
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= kMaxDevices) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch[dev].ptr || ctx == 0 || g_scratch[dev].ctx != ctx) {
        void* p = nullptr;
        *err = cudaGetSymbolAddress(&p, g_plan_scratch);
        if (*err != cudaSuccess) return nullptr;
        g_scratch[dev] = ScratchAddr{ctx, static_cast<int32_t*>(p)};
    }
    return g_scratch[dev].ptr;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status moe_plan_noalloc(const moe_config* cfg, int32_t T, const int32_t* topk_ids,
                                       int32_t capacity, int32_t align, int32_t* counts, int32_t* offsets,
                                       int32_t* slot_of, int32_t* token_of, int32_t* err_flag,
                                       int32_t max_ctas, moe_stream_t stream) {
    moe_status s = check_config(cfg);
    if (s != MOE_OK) return s;
    if (T < 0 || capacity < 0 || align < 1) return MOE_ERR_INVALID_ARG;
    if (!counts || !offsets || !err_flag || (T > 0 && (!topk_ids || !slot_of))) return MOE_ERR_INVALID_ARG;
    if ((int64_t)moe_plan_rows(cfg, T, capacity, align) > (int64_t)INT32_MAX) return MOE_ERR_INVALID_ARG;
    const size_t need = moe_plan_workspace_size(cfg, T);
    if (need > sizeof(int32_t) * (size_t)kNoAllocScratchInts) {
        if (getenv("MOE_DEBUG"))
            fprintf(stderr,
                    "libmoe_gb300: moe_plan_noalloc: T=%d needs %zu bytes of plan scratch, above the built-in "
                    "%zu bytes; use moe_plan with a workspace\n",
                    T, need, sizeof(int32_t) * (size_t)kNoAllocScratchInts);
        return MOE_ERR_WORKSPACE;
    }
    int32_t* scratch = nullptr;
    if (need > 0) {
        cudaError_t e;
        scratch = scratch_for_current_device(&e);
        if (!scratch) return MOE_ERR_CUDA;
    }
    // every histogram entry the second pass reads is written by the first pass of
    // the same call, so the array needs no clearing between calls
    cudaError_t e = launch_plan(*cfg, T, topk_ids, capacity, align, counts, offsets, slot_of, token_of, err_flag,
                                scratch, max_ctas > 0 ? max_ctas : device_info().num_sms * 8,
                                (cudaStream_t)stream);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
