/*
 * moe.h -- C ABI of libmoe_gb300: one Mixture-of-Experts layer on one GB300
 * (sm_103a), as hand-written CUDA kernels.
 *
 *   moe_route      gate: top-k experts and weights per token
 *   moe_plan       per-expert counts, aligned exclusive prefix sums, token -> row slots
 *   moe_dispatch   gather token rows into expert-contiguous rows (fused fp8 quantisation)
 *   moe_expert_ffn grouped gate/up GEMM -> SwiGLU -> down GEMM on the tensor cores
 *   moe_combine    top-k weighted gather-reduce back to token order
 *   moe_layer_dbo  all of the above on two micro-batches ("ubatches") overlapped on a
 *                  compute stream and a comm stream (Dual-Batch Overlap)
 *
 * The operations follow the problem statement of the vLLM Dual-Batch Overlap pages:
 *   [A] "[Core/DBO][1/N] Add Dual-Batch Overlap mechanism to VLLM", Purpose
 *   [B] "[Core/DBO][2/N] Dual-Batch Overlap add DeepEP High Throughput support and
 *       Prefill support", Purpose
 *   [C] "[Perf] Fix DBO overlap: capture DeepEP event before yield", Purpose
 *   [D] "DeepEP HT: full decode CUDA graphs via worst-token dispatch (whole-step +
 *       graphed TBO)", description and commit messages
 * The pages give no gate or FFN formulas; the arithmetic each call performs is
 * stated beside it (the "readings").
 *
 * Conventions for every call
 *  - Ownership: the caller owns every buffer, stream and workspace.  Pointers named
 *    "device" must point to device memory of the current device.  No call allocates
 *    device memory; the only library object is the DBO handle (a few CUDA events).
 *  - Asynchrony: every call only enqueues work on the given stream(s) and returns;
 *    results are valid after the stream work completes.  No call synchronises with
 *    the host, so every call can be captured into a CUDA graph.
 *  - Errors: argument, shape and alignment problems are detected on the host before
 *    anything is enqueued and returned as a moe_status.  Data-dependent problems
 *    found by a kernel (an expert id out of range, a capacity overflow, a bounded wait
 *    that gave up) are stored in the caller's device int32 `err_flag` as a moe_status
 *    value (the first one wins; the library never clears the flag -- zero it before
 *    the call); the kernel then skips the offending entry, never traps.
 *    A failed launch returns MOE_ERR_CUDA.
 *  - Alignment: every device row buffer must start on a 16-byte boundary and rows
 *    are packed with no stride; MOE_ERR_ALIGNMENT otherwise (never copied).
 *  - max_ctas: upper bound on the CTAs a call's kernels may occupy (its SM budget);
 *    <= 0 means "the whole GPU".
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* moe_stream_t;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1, /* null pointer, bad size, unsupported shape combination */
    MOE_ERR_UNSUPPORTED = 2, /* valid request this build cannot serve (e.g. no sm_103a GPU) */
    MOE_ERR_ALIGNMENT = 3,   /* a buffer or row is not 16-byte aligned */
    MOE_ERR_WORKSPACE = 4,   /* workspace missing or smaller than the *_workspace_size query */
    MOE_ERR_CUDA = 5,        /* a CUDA call or launch failed */
    MOE_ERR_CAPACITY = 6,    /* device flag: an expert received more rows than `capacity` */
    MOE_ERR_BAD_INDEX = 7,   /* device flag: an expert id outside [0, num_experts) */
    MOE_ERR_TIMEOUT = 8      /* device flag: a bounded device-side wait gave up */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1, MOE_FP8_E4M3 = 2 } moe_dtype;
typedef enum { MOE_GATE_SOFTMAX = 0, MOE_GATE_SIGMOID_GROUPED = 1, MOE_GATE_SQRT_SOFTPLUS = 2 } moe_gate;

/* Shape of one layer.  E = num_experts routed experts, S = num_shared always-on
 * experts (stored after the routed ones: expert ids E .. E+S-1), k = top_k.
 * dtype selects the layer's storage types:
 *   MOE_F32       x, xe, h, ye, y fp32;  weights fp32
 *   MOE_BF16      x, xe, h, ye, y bf16;  weights bf16
 *   MOE_FP8_E4M3  x, ye, y bf16; xe and h e4m3 with one fp32 power-of-two scale per
 *                 1x128 group of a row; weights e4m3 with one fp32 scale per
 *                 128x128 block.  hidden and inter must be multiples of 128.
 * Limits: k >= 1, k + S <= 32, k <= E, E + S <= 512; grouped gates: E % n_group == 0,
 * 2 <= E / n_group, n_group <= 32, 1 <= topk_group <= n_group,
 * k <= topk_group * (E / n_group). */
typedef struct {
    int32_t hidden;       /* H */
    int32_t inter;        /* I, intermediate size of one expert */
    int32_t num_experts;  /* E */
    int32_t num_shared;   /* S */
    int32_t top_k;        /* k */
    int32_t gate;         /* moe_gate */
    int32_t renormalize;  /* 1: chosen weights sum to 1 (times routed_scale) */
    int32_t n_group;      /* grouped gates only */
    int32_t topk_group;   /* grouped gates only */
    float routed_scale;   /* grouped gates only: multiplies the routed weights */
    int32_t dtype;        /* moe_dtype */
} moe_config;

/* ---------------------------------------------------------------------------
 * moe_route -- the gate.  Logits are an input: the router projection x . W_g is an
 * ordinary dense GEMM upstream of the layer (reading; the pages name the gate kinds
 * only through the models they serve, [C] Test Plan, [D] description).
 *   softmax gate: the k largest logits, descending, equal logits -> lower id first;
 *     w = the softmax probability over all E logits, or (renormalize) the softmax
 *     over the k chosen logits.
 *   grouped sigmoid gate: s_e = sigma(l_e) by the library's specified binary32
 *     sigma (Cody-Waite reduced exp, degree-7 Taylor, see the design notes), choice
 *     score c_e = s_e + bias_e; experts form n_group groups of consecutive ids; a
 *     group scores the sum of its two best c; the topk_group best groups are kept
 *     (equal -> lower group id); the k best c inside them are chosen (equal -> lower
 *     id); w = sigmoid(l) of the chosen (no bias), / their sum if renormalize, times
 *     routed_scale.  Selection is bit-reproducible; weights are fp32.
 *   sqrt-softplus gate (DeepSeek-V4 shaped; the pages name a sqrt-softplus top-k op
 *     and give no formula -- reading): the grouped gate with the score
 *     s_e = sqrt(softplus(l_e)), softplus specified as max(x, 0) + log1p(e^-|x|) on
 *     [-80, 80] with the library's specified exp and a specified log1p (the 2 atanh
 *     series to z^15), then IEEE sqrt; n_group = 1 is plain top-k; w = sqrt(softplus(l))
 *     of the chosen, / their sum if renormalize, times routed_scale.
 * logits   device fp32 [T][E], row-major.  The gates are defined for finite logits;
 *          a NaN logit (or score) is ranked as -inf, so every id written is in [0, E)
 *          whatever the input holds (the weights of such a row are unspecified).
 * bias     device fp32 [E] or NULL (grouped gate only; NULL = 0).
 * topk_ids device int32 [T][k] (out), descending score order.
 * topk_w   device fp32 [T][k] (out).
 * T = 0 is a no-op. */
MOE_API moe_status moe_route(const moe_config* cfg, int32_t T, const float* logits, const float* bias,
                     int32_t* topk_ids, float* topk_w, int32_t max_ctas, moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * moe_route_hash -- hash routing of the DeepSeek-V4-shaped layers (the pages name
 * hash-routing metadata, int32 expert ids, passed to the sqrt-softplus top-k op;
 * reading): token t's k experts are row token_ids[t] of a fixed table, and the weights
 * are the sqrt-softplus gate's -- sqrt(softplus(l)) of those experts, / their sum if
 * renormalize, times routed_scale.  Requires cfg->gate == MOE_GATE_SQRT_SOFTPLUS
 * (else MOE_ERR_UNSUPPORTED).
 * logits    device fp32 [T][E];  token_ids device int32 [T];
 * table     device int32 [vocab][k];
 * topk_ids  device int32 [T][k] (out): the table's entries, passed on unchecked (an
 *           entry outside [0, E) gets weight 0, and moe_plan flags it); a token id
 *           outside [0, vocab) gives ids -1 and weights 0 for its row.
 * topk_w    device fp32 [T][k] (out). */
MOE_API moe_status moe_route_hash(const moe_config* cfg, int32_t T, const float* logits, const int32_t* token_ids,
                                  const int32_t* table, int32_t vocab, int32_t* topk_ids, float* topk_w,
                                  int32_t max_ctas, moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * moe_plan -- per-expert counts, aligned exclusive prefix sums and the row ("slot")
 * of every (token, choice) pair: a stable counting sort.  Per-expert counts stay in
 * device memory and a static worst-case capacity keeps shapes fixed for graph
 * capture ([D] description: worst-token dispatch, device-side counts; the
 * BatchedExperts vs Standard activation formats of its commit messages).
 * Entry (t, j) is expert topk_ids[t][j] for j < k and shared expert E + (j - k) for
 * k <= j < k + S.  Rows of one expert are in (t, j) order.
 *   capacity == 0 ("exact", contiguous): expert e owns rows [offsets[e],
 *     offsets[e] + counts[e]); offsets[e+1] = offsets[e] + counts[e] rounded up to a
 *     multiple of `align` (>= 1); offsets[E+S] = rows used.
 *   capacity  > 0 ("worst-token", per-expert padded): expert e owns rows
 *     [e*capacity, (e+1)*capacity); counts[e] = rows placed; an entry ranked
 *     >= capacity gets slot -1 and sets MOE_ERR_CAPACITY (never dropped silently).
 *     capacity = T is the single-GPU worst case (a token picks an expert once).
 * topk_ids device int32 [T][k].
 * counts   device int32 [E+S] (out); offsets device int32 [E+S+1] (out).
 * slot_of  device int32 [T][k+S] (out): row of each entry, -1 if not placed.
 * token_of device int32 [moe_plan_rows(...)] (out, may be NULL when not wanted): token of
 *          each row, -1 = padding.
 * err_flag device int32 (required): MOE_ERR_BAD_INDEX / MOE_ERR_CAPACITY.
 * ws       device scratch of moe_plan_workspace_size(cfg, T) bytes (may be NULL when
 *          that is 0). */
MOE_API size_t moe_plan_rows(const moe_config* cfg, int32_t T, int32_t capacity, int32_t align);
MOE_API size_t moe_plan_workspace_size(const moe_config* cfg, int32_t T);
MOE_API moe_status moe_plan(const moe_config* cfg, int32_t T, const int32_t* topk_ids, int32_t capacity,
                    int32_t align, int32_t* counts, int32_t* offsets, int32_t* slot_of,
                    int32_t* token_of, int32_t* err_flag, void* ws, size_t ws_bytes,
                    int32_t max_ctas, moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * moe_plan_noalloc -- moe_plan for callers that cannot allocate device memory:
 * code that runs where cudaMalloc is unavailable or forbidden (inside a CUDA-graph
 * capture with a locked memory pool, under an allocator that owns all device memory,
 * in a plugin that receives only tensor pointers), or that cannot size a workspace
 * ahead of time.  The pages have no counterpart to this call; it is a convenience of
 * this library.
 * Same arguments, results and errors as moe_plan, minus the workspace.  The plan's
 * scratch (per-chunk expert histograms) is a fixed 256 KiB array inside the
 * library's device memory, held by every GPU that loads the library until the
 * process exits.  Limit: moe_plan_workspace_size(cfg, T) <= 262144 bytes, i.e.
 * ceil(T / floor(1024 / (k+S))) * (E+S) <= 65536 (a batch of more than 4096
 * entries is cut into chunks of about 1024; a smaller one needs no scratch); a larger T returns
 * MOE_ERR_WORKSPACE before anything is enqueued (MOE_DEBUG=1 prints why).
 * The first call on a device that needs the scratch looks up the array's device
 * address with that device current (and so does the first such call in a new context
 * of the device, e.g. after cudaDeviceReset); make that first call before any stream
 * capture.
 * All calls share the one array, so calls whose kernels overlap on the GPU (on
 * different streams without ordering) race; calls ordered on one stream do not.
 * The array keeps the last call's contents; every entry a call reads is written
 * earlier in that same call, so nothing needs clearing.  No call allocates. */
MOE_API moe_status moe_plan_noalloc(const moe_config* cfg, int32_t T, const int32_t* topk_ids,
                                    int32_t capacity, int32_t align, int32_t* counts, int32_t* offsets,
                                    int32_t* slot_of, int32_t* token_of, int32_t* err_flag,
                                    int32_t max_ctas, moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * moe_dispatch -- on-device analogue of the all-to-all dispatch ([A] Purpose):
 * xe[slot_of[t][j]] = x[t] for every placed entry (slot >= 0).  FP8 layers quantise
 * each 1x128 group of the bf16 row with the power-of-two scale 2^s, s the smallest
 * integer with amax <= 448 * 2^s (amax = 0 -> s = 0), e4m3 round-to-nearest-even:
 * scale(row, g) = 2^s.  Rows no entry maps to are not written.
 * x        device [T][H]: fp32 (MOE_F32) or bf16.
 * xe       device [rows][H]: fp32 / bf16 / e4m3 (out).
 * xe_scale device fp32 (out, FP8 only; else NULL): with xe_scale_ld == 0 row-major
 *          [rows][H/128], scale(row, g) = xe_scale[row * H/128 + g]; with xe_scale_ld > 0
 *          column-major, scale(row, g) = xe_scale[g * xe_scale_ld + row] (xe_scale_ld >=
 *          rows; the layout moe_layer_dbo keeps internally, where the FFN reads 32
 *          consecutive rows' scales in one request).  xe_scale_ld < 0: MOE_ERR_INVALID_ARG. */
MOE_API moe_status moe_dispatch(const moe_config* cfg, int32_t T, const void* x, const int32_t* slot_of,
                        void* xe, float* xe_scale, int64_t xe_scale_ld, int32_t max_ctas,
                        moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * moe_expert_ffn -- every expert's SwiGLU FFN on its rows (the grouped expert GEMMs
 * and the fused activation the pages name: DeepGEMM / batched Triton MoE GEMM with
 * act_and_mul / silu_mul_fp8_quant, [A] discussion, [B] Purpose):
 *   g|u = xe[r] . W13[e]^T   (W13 rows 0..I-1 gate, I..2I-1 up),
 *   h   = silu(g) * u        stored as the activation type (fp8: 1x128 scales),
 *   ye[r] = h . W2[e]^T      stored as fp32 (MOE_F32) or bf16,
 * for r in [offsets[e], offsets[e] + counts[e]), e in [0, E+S); fp32 accumulation.
 * Tile work is derived from the device counts/offsets: no host synchronisation.
 * Rows outside the used ranges are neither read into results nor written.
 * counts, offsets device int32 [E+S], [E+S+1] (from moe_plan).
 * max_rows  rows of xe / ye (moe_plan_rows); a range beyond it sets MOE_ERR_BAD_INDEX.
 * w13      device [E+S][2I][H]; w2 device [E+S][H][I]; fp32 / bf16 / e4m3.
 * xe_scale, xe_scale_ld  the activation scales in either layout of moe_dispatch (FP8
 *          only); a column-major xe_scale_ld below max_rows is MOE_ERR_INVALID_ARG.
 * w13_scale device fp32 [E+S][2I/128][H/128]; w2_scale [E+S][H/128][I/128] (FP8 only).
 * ye       device [max_rows][H] (out).
 * ws       device scratch of moe_ffn_workspace_size(cfg, max_rows) bytes.
 * err_flag device int32 or NULL. */
MOE_API size_t moe_ffn_workspace_size(const moe_config* cfg, int64_t max_rows);
MOE_API moe_status moe_expert_ffn(const moe_config* cfg, const int32_t* counts, const int32_t* offsets,
                          int64_t max_rows, const void* xe, const float* xe_scale, int64_t xe_scale_ld,
                          const void* w13, const float* w13_scale, const void* w2, const float* w2_scale,
                          void* ye, void* ws, size_t ws_bytes, int32_t* err_flag, int32_t max_ctas,
                          moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * moe_combine -- on-device analogue of the all-to-all combine ([A] Purpose):
 * y[t] = sum_{j<k} topk_w[t][j] * ye[slot_of[t][j]] + sum_{s<S} ye[slot_of[t][k+s]],
 * accumulated in fp32 in (j, then s) order, rounded once to the output type; entries
 * with slot -1 contribute nothing.  Deterministic (no atomics).
 * ye device [rows][H] fp32/bf16; topk_w device fp32 [T][k]; y device [T][H] (out). */
MOE_API moe_status moe_combine(const moe_config* cfg, int32_t T, const void* ye, const float* topk_w,
                       const int32_t* slot_of, void* y, int32_t max_ctas, moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * Dual-Batch Overlap.  The batch is split into two ubatches, tokens [0, s) and
 * [s, T).  One ubatch's route / plan / dispatch and combine run on the comm stream
 * while the other's expert FFN runs on the compute stream ([A] Purpose); every
 * event a comm step waits on is recorded on the compute stream right after the
 * producing kernel, before the other ubatch's compute is enqueued, so it covers
 * only that ubatch's compute tail ([C] Purpose); the comm stream is joined back to
 * the compute stream before the call returns, so no comm work is left in flight
 * ([D] commit messages: dispatch and combine joined to the compute stream).  The
 * enqueue order is one fixed schedule: no host threads and no yields are needed
 * for a single layer.
 */
typedef struct moe_dbo_handle moe_dbo_handle;
MOE_API moe_status moe_dbo_create(moe_dbo_handle** out);
MOE_API void moe_dbo_destroy(moe_dbo_handle* h);

/* Everything moe_layer_dbo reads and writes.  Inputs: logits fp32 [T][E], bias
 * (nullable), x [T][H], the weights and scales as for moe_expert_ffn.  Outputs:
 * y [T][H], topk_ids int32 [T][k], topk_w fp32 [T][k], err_flag (nullable: then a
 * flag inside the workspace is used).  workspace: moe_layer_workspace_size bytes,
 * 256-byte aligned, holding both ubatches' plans, xe, h and ye. */
typedef struct {
    const float* logits;
    const float* bias;
    const void* x;
    const void* w13;
    const float* w13_scale;
    const void* w2;
    const float* w2_scale;
    void* y;
    int32_t* topk_ids;
    float* topk_w;
    int32_t* err_flag;
    void* workspace;
    size_t workspace_bytes;
} moe_layer_args;

/* Workspace for moe_layer_dbo with T tokens (either split or not). */
MOE_API size_t moe_layer_workspace_size(const moe_config* cfg, int32_t T, int32_t capacity, int32_t align);

/* The whole layer.
 * split     0 -> ceil(T/2); s in [1, T) -> ubatches [0, s), [s, T); s >= T -> no split.
 *           T < min_tokens also runs unsplit (never an empty ubatch, [B] commit list).
 * capacity  0 = exact layout; > 0 = worst-token layout with that many rows per expert
 *           per ubatch (must be >= the ubatch's token count for no overflow).
 * comm_sms  SMs given to route/plan/dispatch/combine while they overlap an expert FFN
 *           (each of their kernels is capped at as many CTAs as fit on that many SMs);
 *           the FFN gets one CTA on each remaining SM.  Steps that overlap nothing get
 *           the whole GPU.  0 = no split of the GPU.
 * compute, comm  the two streams; comm == compute runs the identical two-ubatch
 *           schedule serialised on one stream, every kernel on the whole GPU (the SM
 *           budget applies only when the streams differ).
 * The call resets *err_flag to 0 on the compute stream before its kernels run. */
MOE_API moe_status moe_layer_dbo(moe_dbo_handle* h, const moe_config* cfg, const moe_layer_args* args,
                         int32_t T, int32_t split, int32_t min_tokens, int32_t capacity,
                         int32_t align, int32_t comm_sms, moe_stream_t compute, moe_stream_t comm);

/* moe_layer_dbo_ex -- moe_layer_dbo with options: the exchange around the experts fused
 * into the grouped GEMM ("DeepEP HT: full decode CUDA graphs via worst-token dispatch",
 * description: dispatch and combine around the experts).  flags (either or both):
 *   MOE_LAYER_FUSED_GATHER  the plan also records the token of every row, and the
 *     gate/up kernel takes each A row straight from x by that token (TMA gather of 4 rows
 *     at a time) instead of from a dispatched copy; fp8 layers quantise each token's row
 *     once instead of once per chosen expert.
 *   MOE_LAYER_FUSED_COMBINE  the down kernel's epilogue stores ye and the last of a
 *     token's k+S rows to finish a slab of 128 columns (256 for bf16) forms that slab of
 *     y in the fixed (j, then s) order of moe_combine; there is no combine step.  With an
 *     entry dropped by a capacity overflow (MOE_ERR_CAPACITY) its token's y row is left
 *     unwritten in this mode.
 * No float atomics: the result is the same, bit for bit, as the unfused layer.  Served by
 * the tensor-core FFN (bf16 and fp8 layers); other layers (fp32, or the CUDA-core FFN
 * forced) run unfused.  Other bits: MOE_ERR_INVALID_ARG.  flags = 0 is moe_layer_dbo. */
enum { MOE_LAYER_FUSED_GATHER = 1, MOE_LAYER_FUSED_COMBINE = 2, MOE_LAYER_FUSED = 3 };
MOE_API moe_status moe_layer_dbo_ex(moe_dbo_handle* h, const moe_config* cfg, const moe_layer_args* args,
                                    int32_t T, int32_t split, int32_t min_tokens, int32_t capacity,
                                    int32_t align, int32_t comm_sms, int32_t flags, moe_stream_t compute,
                                    moe_stream_t comm);

/* The enqueue schedule moe_layer_dbo follows, for inspection (host only, no GPU
 * needed).  Writes up to max_ops records of 4 int32 each: {stream (0 compute,
 * 1 comm), op (see MOE_OP_*), ubatch (0/1, -1 = none), event id (record/wait) or -1}
 * and returns the number of records.  two_ubatches = 0 gives the unsplit schedule. */
enum {
    MOE_OP_ROUTE = 0,
    MOE_OP_PLAN = 1,
    MOE_OP_DISPATCH = 2,
    MOE_OP_FFN = 3,
    MOE_OP_COMBINE = 4,
    MOE_OP_RECORD = 5,
    MOE_OP_WAIT = 6,
    MOE_OP_STANDIN = 7
};
MOE_API int32_t moe_dbo_schedule(int32_t two_ubatches, int32_t* ops, int32_t max_ops);
/* The schedule of moe_layer_dbo_ex with these flags (MOE_LAYER_FUSED_COMBINE: no combine step). */
MOE_API int32_t moe_dbo_schedule_ex(int32_t two_ubatches, int32_t flags, int32_t* ops, int32_t max_ops);

/* ---------------------------------------------------------------------------
 * A stack of L layers with Dual-Batch Overlap across layer boundaries.  The pages'
 * overlap is across a whole model step: one ubatch's dispatch and combine run under
 * the other ubatch's non-MoE compute as well as its experts ([C] Purpose: combine of
 * one ubatch overlapped with the other ubatch's non-MoE compute).  Layer l here is
 *     a   = x_l + x_l . Wa_l^T            a stand-in for the non-MoE compute
 *     x_{l+1} = a + MoE_l(a)              routed by the given logits_l,
 * the stand-in a dense bf16 projection with a residual (one rounding), the MoE part
 * as moe_layer_dbo with the residual added inside combine (one rounding).
 * Compute stream: stand-in and experts; comm stream: route, plan, dispatch, combine.
 * event_before_yield = 1 records each event a comm step waits on right after the
 * compute kernel it stands for ([C] Purpose); 0 reproduces the placement before that
 * fix (recorded after the other ubatch's compute was enqueued), for measurement.  Both
 * give identical results.  Activations must be bf16 (MOE_BF16 / MOE_FP8_E4M3 layers)
 * and hidden a multiple of 256, else MOE_ERR_UNSUPPORTED. */
typedef struct {
    const void* x;                      /* device [T][H] bf16: input of layer 0 */
    void* out;                          /* device [T][H] bf16: output of layer L-1 */
    const float* const* logits;         /* host array of L device pointers, each fp32 [T][E] */
    const float* bias;                  /* device fp32 [E] or NULL, every layer */
    const void* const* wa;              /* host array of L device pointers, each bf16 [H][H] (K-major) */
    const void* const* w13;             /* host arrays of L device pointers, layouts as in */
    const float* const* w13_scale;      /* moe_expert_ffn (scales: FP8 only, else NULL) */
    const void* const* w2;
    const float* const* w2_scale;
    int32_t* err_flag;                  /* device int32 or NULL (workspace flag); reset by the call */
    void* workspace;                    /* moe_stack_workspace_size bytes, 256-byte aligned */
    size_t workspace_bytes;
} moe_stack_args;

MOE_API size_t moe_stack_workspace_size(const moe_config* cfg, int32_t T, int32_t capacity, int32_t align);
MOE_API moe_status moe_stack_dbo(moe_dbo_handle* h, const moe_config* cfg, const moe_stack_args* args,
                                 int32_t L, int32_t T, int32_t split, int32_t min_tokens, int32_t capacity,
                                 int32_t align, int32_t comm_sms, int32_t event_before_yield,
                                 moe_stream_t compute, moe_stream_t comm);
/* The stack's enqueue schedule (same record format as moe_dbo_schedule; layer by layer). */
MOE_API int32_t moe_stack_schedule(int32_t layers, int32_t two_ubatches, int32_t event_before_yield,
                                   int32_t* ops, int32_t max_ops);

MOE_API const char* moe_status_string(moe_status s);

/* ---------------------------------------------------------------------------
 * moe_debug_inject_wait -- test hook for the failure path of the bounded device
 * waits (the pages have no counterpart).  With enable != 0, every expert-FFN kernel
 * launched afterwards (by moe_expert_ffn, moe_layer_dbo or moe_stack_dbo) begins with a
 * wait, limited to timeout_ns, on a barrier that nothing ever completes, before it
 * issues any copy: the wait runs out, the kernel stores MOE_ERR_TIMEOUT in err_flag,
 * skips its work, frees its tensor memory and returns normally, so the context stays
 * usable.  The staged combine kernel takes the same path (its error goes to the
 * layer's err_flag, or, called on its own, to the word moe_comm_error reads).
 * enable = 0 (the default) turns it off.  Process-wide, host-side only;
 * enable != 0 with timeout_ns <= 0 is MOE_ERR_INVALID_ARG. */
MOE_API moe_status moe_debug_inject_wait(int32_t enable, int64_t timeout_ns);

/* ---------------------------------------------------------------------------
 * moe_comm_error -- the library's sticky error word for moe_combine, whose signature
 * carries no error flag: MOE_ERR_TIMEOUT once a bounded wait of its staged kernel ran
 * out on the current device (never on a healthy GPU; see moe_debug_inject_wait), else
 * 0.  (moe_dispatch has no waits.)  Synchronises the current device, writes the word to
 * *code (host), and resets it to 0 when clear != 0.  code NULL: MOE_ERR_INVALID_ARG. */
MOE_API moe_status moe_comm_error(int32_t* code, int32_t clear);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
