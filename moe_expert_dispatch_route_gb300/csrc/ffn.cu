// moe_expert_ffn: chooses the expert-FFN kernels for a layer and owns the layout of
// their scratch memory (h, the SwiGLU output, and its fp8 scales).
#include <stdlib.h>
#include <string.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {

size_t ffn_scratch_bytes(const moe_config& c, int64_t max_rows) {
    size_t b = align_up((size_t)max_rows * c.inter * elt_bytes(c.dtype), 256);
    if (c.dtype == MOE_FP8_E4M3) b += align_up((size_t)max_rows * (c.inter / kQG) * 4, 256);
    return b;
}

// MOE_FFN_IMPL=simt selects the CUDA-core kernels for every layer (a second,
// independent implementation to compare the tensor-core kernels with).
static bool force_simt() {
    static int v = -1;
    if (v < 0) {
        const char* e = getenv("MOE_FFN_IMPL");
        v = (e && strcmp(e, "simt") == 0) ? 1 : 0;
    }
    return v == 1;
}

// Rows the batch really uses: the caller's hint, else max_rows less the largest padding
// an exact layout with 128-row alignment adds.
static int64_t rows_estimate(const moe_config& c, const FfnArgs& a) {
    if (a.rows_hint > 0) return a.rows_hint;
    const int64_t pad = (int64_t)(c.num_experts + c.num_shared) * 127;
    return a.max_rows > pad ? a.max_rows - pad : 0;
}

bool ffn_tc_selected(const moe_config& c) { return !force_simt() && ffn_tc_supported(c); }

cudaError_t launch_ffn(const moe_config& c, const FfnArgs& a, int grid_cap, cudaStream_t st) {
    if (a.token_of) return launch_ffn_tc(c, a, grid_cap, st);  // fused gather / combine: one-CTA kernels
    if (!force_simt() && ffn_tc_supported(c)) {
        // prefill-sized batches: 256 x 256 tiles on CTA pairs; decode: one CTA per tile
        if (ffn_pair_preferred(c, rows_estimate(c, a))) return launch_ffn_pair(c, a, grid_cap, st);
        return launch_ffn_tc(c, a, grid_cap, st);
    }
    return launch_ffn_simt(c, a, grid_cap, st);
}

}  // namespace moe
