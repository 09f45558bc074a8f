// Internal launch interface between the C-ABI layer (api.cu) and the kernels.
// Arguments are already validated by the caller; each launcher only enqueues.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

struct DeviceInfo {
    int device;
    int num_sms;
    int cc_major, cc_minor;
    size_t smem_optin;
};
const DeviceInfo& device_info();
moe_status check_config(const moe_config* c);  // shape limits and row alignment
bool aligned16(const void* p);

// Identity of the CUDA context current on the calling thread: unique for the life of
// the process (a device reset followed by a new context gives a new id); 0 when it
// cannot be read.  Host-side caches of per-context state -- device addresses of module
// variables, kernel attributes -- are keyed on it so that they never go stale.
unsigned long long current_context_id();
// Test hook (moe_debug_inject_wait): > 0 makes every expert-FFN kernel launched from
// now on first wait this long on a barrier nothing arrives on, then report
// MOE_ERR_TIMEOUT and skip its work; 0 = off (the default).
int64_t wait_injection_ns();
// Device address, in the context current on this thread, of the library's sticky error
// word: the staged combine kernel called on its own (no caller flag) stores
// MOE_ERR_TIMEOUT there when a bounded wait runs out.  NULL if it cannot be looked up.
int32_t* comm_error_word();
// Raises the dynamic shared memory limit of a kernel to `bytes`, once per context
// (thread-safe); later calls in the same context return at once.
cudaError_t ensure_max_dynamic_smem(const void* func, int bytes);
template <typename... A>
cudaError_t ensure_max_dynamic_smem(void (*kern)(A...), int bytes) {
    return ensure_max_dynamic_smem(reinterpret_cast<const void*>(kern), bytes);
}

// route.cu
cudaError_t launch_route(const moe_config& c, int T, const float* logits, const float* bias,
                         int32_t* ids, float* w, int grid_cap, cudaStream_t st);

cudaError_t launch_route_hash(const moe_config& c, int T, const float* logits, const int32_t* token_ids,
                              const int32_t* table, int vocab, int32_t* ids, float* w, int grid_cap, cudaStream_t st);

// plan.cu
int plan_tokens_per_chunk(const moe_config& c, int T);
int plan_num_chunks(const moe_config& c, int T);
cudaError_t launch_plan(const moe_config& c, int T, const int32_t* ids, int capacity, int align,
                        int32_t* counts, int32_t* offsets, int32_t* slot_of, int32_t* token_of,
                        int32_t* err, int32_t* hist_ws, int grid_cap, cudaStream_t st);

// head.cu: plan + dispatch in one launch when the plan is a single chunk; route + plan +
// dispatch in one launch (thread-block clusters) when, in addition, the batch is small
bool plan_dispatch_fusable(const moe_config& c, int T);
bool head_fusable(const moe_config& c, int T);
cudaError_t launch_route_plan_dispatch(const moe_config& c, int T, const float* logits, const float* bias,
                                       int32_t* ids, float* w, int capacity, int align, int32_t* counts,
                                       int32_t* offsets, int32_t* slot_of, int32_t* err, const void* x, void* xe,
                                       float* xe_scale, int64_t scale_cs, int grid_cap, cudaStream_t st);
cudaError_t launch_plan_dispatch(const moe_config& c, int T, const int32_t* ids, int capacity, int align,
                                 int32_t* counts, int32_t* offsets, int32_t* slot_of, int32_t* err, const void* x,
                                 void* xe, float* xe_scale, int64_t scale_cs, int grid_cap, cudaStream_t st);

// dispatch.cu / combine.cu.  fp8 row scales: scale (row r, group g) sits at
// xe_scale[r * (H/128) + g] when scale_cs == 0 (the ABI's row-major layout), else at
// xe_scale[g * scale_cs + r] (column-major, as the layer keeps them internally: the FFN
// then reads 32 consecutive rows' scales in one request).
cudaError_t launch_dispatch(const moe_config& c, int T, const void* x, const int32_t* slot_of,
                            void* xe, float* xe_scale, int64_t scale_cs, int grid_cap, cudaStream_t st);
// fused gather, fp8: x [T][H] bf16 -> x_q [T][H] e4m3 + scales column-major [H/128][scale_cs]
cudaError_t launch_quantize_rows(const moe_config& c, int T, const void* x, void* xq, float* xs, int64_t scale_cs,
                                 int grid_cap, cudaStream_t st);
// Resident CTAs per SM of the 256-thread comm-side kernels (route, plan, dispatch,
// quantize_rows: 2048 threads per SM, registers well under the limit) and of the staged
// combine: an SM budget for them is that many CTAs per SM.
constexpr int kCommCtasPerSm = 8;
int combine_ctas_per_sm();
// err: device int32 receiving MOE_ERR_TIMEOUT if a bounded wait of the staged kernels
// runs out (NULL: the library's own sticky word, read by moe_comm_error).
cudaError_t launch_combine(const moe_config& c, int T, const void* ye, const float* w,
                           const int32_t* slot_of, void* y, int grid_cap, cudaStream_t st,
                           const void* resid = nullptr, int32_t* err = nullptr);

// FFN: scratch = h [max_rows][I] (+ fp8 scales) followed by the kernels' own scratch.
size_t ffn_scratch_bytes(const moe_config& c, int64_t max_rows);
struct FfnArgs {
    const int32_t* counts;
    const int32_t* offsets;
    int64_t max_rows;
    const void* xe;
    const float* xe_scale;
    const void* w13;
    const float* w13_scale;
    const void* w2;
    const float* w2_scale;
    void* ye;
    void* ws;
    int32_t* err;
    int reverse;     // walk experts in descending order (L2 reuse across ubatches)
    int64_t xs_cs;   // layout of xe_scale: 0 = row-major, else column-major with this column stride
    int64_t rows_hint = 0;  // rows actually used (tokens x (k+S)) when known, else 0
    // Fused gather: A rows are taken by token (token_of) from gx -- x (bf16) or x_q (fp8,
    // scales gx_scale column-major [H/128][gT]) -- instead of xe.  Fused combine (with
    // y): the down kernel forms y [gT][H] from ye, slot_of and topk_w; cnt: gT * H/128
    // counters (cleared by the up kernel).  The one-CTA tensor-core kernels only.
    const int32_t* token_of = nullptr;
    const void* gx = nullptr;
    const float* gx_scale = nullptr;
    int gT = 0;
    const int32_t* slot_of = nullptr;
    const float* topk_w = nullptr;
    void* y = nullptr;
    int32_t* cnt = nullptr;
};
cudaError_t launch_ffn(const moe_config& c, const FfnArgs& a, int grid_cap, cudaStream_t st);
// the layer's FFN runs on the tensor-core kernels (not forced onto the CUDA cores)
bool ffn_tc_selected(const moe_config& c);

// ffn_pair.cu: the same FFN on CTA pairs (tcgen05.mma.cta_group::2, 256 x 256 tiles),
// chosen for bf16 batches averaging at least 128 rows per expert (MOE_FFN_TILE=pair /
// single forces either family for any layer)
bool ffn_pair_supported(const moe_config& c);
bool ffn_pair_preferred(const moe_config& c, int64_t rows_hint);
cudaError_t launch_ffn_pair(const moe_config& c, const FfnArgs& a, int grid_cap, cudaStream_t st);

// ffn_simt.cu: portable CUDA-core grouped GEMM (fp32 layers, and any layer on request)
cudaError_t launch_ffn_simt(const moe_config& c, const FfnArgs& a, int grid_cap, cudaStream_t st);

// ffn_tc.cu: tcgen05 / TMEM / TMA grouped GEMM, one CTA per tile (bf16 and fp8 layers)
bool ffn_tc_supported(const moe_config& c);
void* tma_encode_fn();  // cuTensorMapEncodeTiled from the driver, or null
// 2-D K-major [rows][inner] tensor map, 128-byte swizzle, box = one 128-byte row x box_rows
bool make_tma_map_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, bool fp8, int box_rows);
cudaError_t launch_ffn_tc(const moe_config& c, const FfnArgs& a, int grid_cap, cudaStream_t st);
// the stand-in for a layer's non-MoE compute in a stack: out = x + x . Wa^T (bf16)
bool standin_tc_supported(const moe_config& c);
cudaError_t launch_standin(const moe_config& c, int rows, const void* x, const void* wa, void* out, int grid_cap,
                           cudaStream_t st);

// Launches `kern` with programmatic stream serialisation: it may be scheduled while
// the previous kernel on the stream finishes; the kernel calls pdl_begin() before it
// touches that kernel's outputs.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), int grid, int block, size_t smem, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, ((KArgs)args)...);
}

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline int elt_bytes(int dtype) { return dtype == MOE_F32 ? 4 : dtype == MOE_BF16 ? 2 : 1; }
// bytes of one element of x / ye / y (fp8 layers keep bf16 there)
inline int io_bytes(int dtype) { return dtype == MOE_F32 ? 4 : 2; }

}  // namespace moe
