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
    if (f32_chunk_out_tensor_cores(g, bf16)) {
        const F32ChunkOutArgs f{static_cast<const float*>(a.x), a.dt, static_cast<const float*>(a.B),
                                static_cast<const float*>(a.C), a.D, a.G, static_cast<const float*>(a.chunk_states),
                                static_cast<float*>(a.y)};
        return launch_chunk_out_f32tc(g, f, st);
    }
    return launch_chunk_out_simt(g, bf16, a, st);
}

// Heads of 64 columns run in pairs (two heads of one group per CTA, as one
// head of 128 columns, one CTA per SM) where the state has 128 rows or more
// and single heads would give 256 to 2048 CTAs: the pairs then still give
// 128 CTAs or more, and beyond that many waves of single heads at two CTAs
// per SM do better.  Measured on GB300 (whole forward pass, µs, single heads
// / pairs, CTAs of single heads): long_seq_carried_state (256) 261.5 /
// 256.3; state 128, L 16384 (256) 500.9 / 489.4; state 256, L 32768 (256)
// 789.4 / 774.0; state 128, L 4096 (1024) 511.5 / 505.5; state 256, L 4096
// (2048) 762.9 / 756.5; state 128, L 1024 (4096) 528.1 / 529.8; state 256,
// L 1024 (8192) 843.0 / 848.6; state 64, L 4096 (1024) 442.1 / 452.3;
// mamba2_1p3b_layer (128) 50.1 / 60.3.  Chunks of 256 (two 128-token
// sub-blocks per chunk) lose with pairs: long_seq_carried_state run at chunk
// 256 306.5 / 310.9, state 128, L 4096 596 / 606, state 256, L 4096 1066 /
// 1086; so the pairs run at chunk 128 only (the forward pass's usual chunk).
// Over sequence segments (few (batch, head) pairs) they are off: the blog's
// example problem 124.0 / 122.7, but b 1, L 32768, 4 heads 62.0 / 65.0 and
// chunk 256 57.1 / 66.7, state 256 with 8 heads 102.7 / 103.3.
// MAMBA2_STATE_PAIRS=0 or =1 turns the pairs off or on (where they apply),
// for timing both on one shape.
bool use_head_pairs(const Geom& g, const StatePassArgs& a) {
    if (a.split || g.headdim != 64) return false;
    if (g.nheads % 2 != 0 || g.heads_per_group % 2 != 0) return false;
    const char* env = getenv("MAMBA2_STATE_PAIRS");
    if (env && (env[0] == '0' || env[0] == '1') && env[1] == 0) return env[0] == '1';
    if (a.segments > 1) return false;
    const int64_t ctas = g.batch * g.nheads * ((g.dstate + 127) / 128);  // single heads
    return g.chunk == 128 && g.dstate >= 128 && ctas >= 2 * 128 && ctas <= 2048;
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

// fp32 problems run on the split-bf16 tensor-core kernels where they cover
// the shape: stage 3 in both the forward pass and its own entry point (it
// reads fp32 directly), stage 2 only inside mamba2_ssd_fwd (it reads B as
// bf16 hi/lo planes, made in the forward pass's workspace; the stage entry
// point takes no workspace and keeps the CUDA-core kernel).
// MAMBA2_FP32_PATH=simt forces the CUDA-core kernels, for timing both.
static bool fp32_path_simt() {
    const char* env = getenv("MAMBA2_FP32_PATH");
    return env && strcmp(env, "simt") == 0;
}

bool f32_chunk_out_tensor_cores(const Geom& g, bool bf16) {
    return !bf16 && chunk_out_f32tc_fits(g) && !fp32_path_simt();
}

bool use_f32_tensor_cores(const Geom& g, bool bf16) {
    return f32_chunk_out_tensor_cores(g, bf16) && state_pass_split_fits(g);
}

}  // namespace m2
