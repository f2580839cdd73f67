// dispatch.cu — chooses the kernel that runs each stage for a given shape.
#include <stdlib.h>
#include <string.h>

#include "common.cuh"

namespace m2 {

cudaError_t launch_state_pass(const Geom& g, bool bf16, const StatePassArgs& a, cudaStream_t st) {
    if (bf16 && state_pass_tc_fits(g)) return launch_state_pass_tc(g, a, st);
    return launch_state_pass_simt(g, bf16, a, st);
}

cudaError_t launch_chunk_out(const Geom& g, bool bf16, const ChunkOutArgs& a, cudaStream_t st) {
    if (bf16 && chunk_out_tc_fits(g)) return launch_chunk_out_tc(g, a, st);
    return launch_chunk_out_simt(g, bf16, a, st);
}

// The fused kernel keeps one CTA per pair of heads of a batch row on the chip
// for the whole sequence.  Measured on GB300 it is still slower than the
// separate stages (long-sequence workload: 0.42 ms against 0.31 ms per pass),
// so the separate stages stay the default.  MAMBA2_FWD_PATH=fused or =staged
// forces a path (fused only where it fits), for testing and for timing both on
// one shape.
bool use_fused_forward(const Geom& g, bool bf16) {
    if (!bf16 || !ssd_fused_fits(g)) return false;
    const char* env = getenv("MAMBA2_FWD_PATH");
    return env && strcmp(env, "fused") == 0;
}

// fp32 problems whose stages 2 and 3 the split-bf16 tensor-core kernels
// cover run them inside mamba2_ssd_fwd (the stage entry points keep the
// CUDA-core kernels: they take no workspace for the bf16 planes).
// MAMBA2_FP32_PATH=simt forces the CUDA-core kernel, for timing both.
bool use_f32_tensor_cores(const Geom& g, bool bf16) {
    if (bf16 || !chunk_out_f32tc_fits(g) || !state_pass_split_fits(g)) return false;
    const char* env = getenv("MAMBA2_FP32_PATH");
    return !(env && strcmp(env, "simt") == 0);
}

}  // namespace m2
