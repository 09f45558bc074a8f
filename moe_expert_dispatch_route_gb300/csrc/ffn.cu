// moe_expert_ffn: chooses the expert-FFN kernels for a layer and owns the layout of
// their scratch memory (h, the SwiGLU output, and its fp8 scales).
#include "common.cuh"
#include "kernels.h"

namespace moe {

size_t ffn_scratch_bytes(const moe_config& c, int64_t max_rows) {
    size_t b = align_up((size_t)max_rows * c.inter * elt_bytes(c.dtype), 256);
    if (c.dtype == MOE_FP8_E4M3) b += align_up((size_t)max_rows * (c.inter / kQG) * 4, 256);
    return b;
}

cudaError_t launch_ffn(const moe_config& c, const FfnArgs& a, int grid_cap, cudaStream_t st) {
    return launch_ffn_simt(c, a, grid_cap, st);
}

}  // namespace moe
