// common.cuh — small helpers shared by the CUDA translation units of the
// library (element conversion, problem geometry, internal launch interface).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mamba2_ssd.h"

namespace m2 {

// log2(e) rounded to fp32: stage 1 scales the natural-log cumsum by it so the
// later stages can use exp2 [blog §Kernel 1].
constexpr float kLog2e = 1.4426950408889634f;

// Problem geometry resolved once on the host and passed by value to kernels.
struct Geom {
    int64_t batch, seqlen, nheads, headdim, dstate, ngroups, chunk;
    int64_t nchunks;      // ceil(seqlen / chunk)
    int64_t heads_per_group;
};

inline Geom make_geom(const mamba2_shape& s) {
    Geom g;
    g.batch = s.batch;
    g.seqlen = s.seqlen;
    g.nheads = s.nheads;
    g.headdim = s.headdim;
    g.dstate = s.dstate;
    g.ngroups = s.ngroups;
    g.chunk = s.chunk_size;
    g.nchunks = (s.seqlen + s.chunk_size - 1) / s.chunk_size;
    g.heads_per_group = s.nheads / s.ngroups;
    return g;
}

__host__ __device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// Status word values written by kernels (mirrors mamba2_status codes).
constexpr unsigned int kStatusTimeout = MAMBA2_ERR_TIMEOUT;

// ---------------------------------------------------------------- launchers
// Each returns the cudaError_t of its launch(es).  Arguments were validated
// by the C-ABI layer; pointers are device pointers.
struct StatePassArgs {
    const void* x;
    const float* dt;
    const void* B;
    const float* G;
    const float* init;  // may be null
    void* chunk_states;
    float* final_state;  // may be null
    // Launch with programmatic stream serialization (the forward pass: the
    // kernel may start while stage 1 runs and waits for it before reading G).
    bool pdl = false;
    // Sequence segments (tensor-core kernel only, k_state_pass_tc.cu): with
    // segments > 1 the launch is the summary pass (summary) or the segment
    // pass over seg_states, [b, nh, segments - 1, S, H] fp32.
    int segments = 1;
    bool summary = false;
    float* seg_states = nullptr;
    // fp32 on the tensor cores (chunk 128, one pass): x is fp32, B comes as
    // bf16 hi/lo planes [b, L, 2 G, S], and the chunk states are written in
    // fp32; init and final are fp32 as always.
    bool split = false;
};

struct ChunkOutArgs {
    const void* x;
    const float* dt;
    const void* B;
    const void* C;
    const float* D;  // may be null
    const float* G;
    const void* chunk_states;
    void* y;
    // As StatePassArgs::pdl: may start while stage 2 runs.
    bool pdl = false;
};

struct SsdStepArgs {
    const void* x;  // [b, nh, H]
    const float* dt;
    const float* A;
    const void* B;  // [b, G, S]
    const void* C;
    const float* D;         // may be null
    const float* state_in;  // may be null (zeros); may equal state_out
    float* state_out;
    void* y;
};

// The fused state pass + chunk output (k_ssd_fused_tc.cu): y and the final
// state straight from x, dt, B, C, D, G and the initial state.
struct FusedArgs {
    const void* x;
    const float* dt;
    const void* B;
    const void* C;
    const float* D;     // may be null
    const float* G;
    const float* init;  // may be null
    void* y;
    float* final_state;  // may be null
    bool pdl = false;    // may start while stage 1 runs
};

cudaError_t launch_chunk_cumsum(const Geom& g, const float* dt, const float* A, float* G,
                                cudaStream_t st);
cudaError_t launch_state_pass_simt(const Geom& g, bool bf16, const StatePassArgs& a, cudaStream_t st);
cudaError_t launch_chunk_out_simt(const Geom& g, bool bf16, const ChunkOutArgs& a, cudaStream_t st);

cudaError_t launch_ssd_step(const Geom& g, bool bf16, const SsdStepArgs& a, cudaStream_t st);

// Tensor-core kernels (bf16) and the shapes they cover.
bool chunk_out_tc_fits(const Geom& g);
cudaError_t launch_chunk_out_tc(const Geom& g, const ChunkOutArgs& a, cudaStream_t st);
bool state_pass_tc_fits(const Geom& g);
bool state_pass_split_fits(const Geom& g);
cudaError_t launch_state_pass_tc(const Geom& g, const StatePassArgs& a, cudaStream_t st);
// Whether the tensor-core state pass runs heads of 64 columns in pairs
// (dispatch.cu).
bool use_head_pairs(const Geom& g, const StatePassArgs& a);
// Segments the forward pass splits each sequence into for stage 2 (1: one
// pass over the whole sequence), the bytes of their states, and the carry
// between the summary and segment passes.
int state_pass_segments(const Geom& g);
int64_t state_pass_segment_bytes(const Geom& g);
cudaError_t launch_state_carry(const Geom& g, const float* G, float* seg_states, int nseg, bool pdl,
                               cudaStream_t st);

// fp32 stage 3 on the tensor cores (k_chunk_out_f32tc.cu): fp32 x, B, C and
// chunk states, split on chip into bf16 hi/lo pairs.
struct F32ChunkOutArgs {
    const float* x;
    const float* dt;
    const float* B;
    const float* C;
    const float* D;  // may be null
    const float* G;
    const float* cs;
    float* y;
};
// rows of `width` fp32 values (width % 4 == 0) -> rows of 2 x width bf16 (hi, lo)
cudaError_t launch_split_bf16(const float* src, void* dst, int64_t rows, int width, cudaStream_t st);
bool chunk_out_f32tc_fits(const Geom& g);
cudaError_t launch_chunk_out_f32tc(const Geom& g, const F32ChunkOutArgs& a, cudaStream_t st);
// Whether an fp32 problem's stage 3 runs on the tensor cores, and whether
// mamba2_ssd_fwd runs its stages 2 and 3 there (dispatch.cu).
bool f32_chunk_out_tensor_cores(const Geom& g, bool bf16);
bool use_f32_tensor_cores(const Geom& g, bool bf16);

bool ssd_fused_fits(const Geom& g);
cudaError_t launch_ssd_fused(const Geom& g, const FusedArgs& a, cudaStream_t st);

// Dispatchers: pick the tensor-core kernel when the shape has one, else the
// CUDA-core kernel (dispatch.cu).
cudaError_t launch_state_pass(const Geom& g, bool bf16, const StatePassArgs& a, cudaStream_t st);
cudaError_t launch_chunk_out(const Geom& g, bool bf16, const ChunkOutArgs& a, cudaStream_t st);
// Whether mamba2_ssd_fwd runs the fused kernel after stage 1 for this shape
// (else stages 2 and 3 separately).
bool use_fused_forward(const Geom& g, bool bf16);

// Device address of the current device's status word (api.cu).
unsigned int* device_status_word();

// Streaming multiprocessors of the current device (queried once per device;
// 0 if the query fails) (api.cu).
int sm_count();

// Raises `func`'s dynamic shared-memory limit to at least `bytes` on the
// current device.  The driver call is made once per (device, kernel) and again
// only when a launch needs more than was set before, so launches do no
// attribute work on the host (api.cu).
cudaError_t ensure_max_dynamic_smem(const void* func, int bytes);

}  // namespace m2
