// dispatch.cu — chooses the kernel that runs each stage for a given shape.
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

}  // namespace m2
