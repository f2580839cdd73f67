// api.cu — the extern "C" boundary: argument checks, workspace layout and
// launch sequencing.  No arithmetic of the method lives here; every step of
// the forward pass runs in the kernels of the other translation units.
#include <stdlib.h>
#include <string.h>

#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"

namespace m2 {
namespace {

constexpr int kVersion = 1 * 10000 + 2 * 100 + 0;

// Per-device status word: kernels with bounded waits record a timeout here.
__device__ unsigned int g_status_word = 0;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t elt_size(const mamba2_shape& s) { return s.dtype == MAMBA2_BF16 ? 2 : 4; }

// Shape checks shared by every entry point.
mamba2_status check_shape(const mamba2_shape* s) {
    if (!s) return MAMBA2_ERR_INVALID_ARG;
    if (s->dtype != MAMBA2_F32 && s->dtype != MAMBA2_BF16) return MAMBA2_ERR_INVALID_ARG;
    if (s->reserved != 0) return MAMBA2_ERR_INVALID_ARG;
    if (s->batch < 0 || s->seqlen < 0 || s->nheads < 1 || s->headdim < 1 || s->dstate < 1 ||
        s->ngroups < 1 || s->chunk_size < 1)
        return MAMBA2_ERR_INVALID_ARG;
    if (s->nheads % s->ngroups != 0) return MAMBA2_ERR_INVALID_ARG;
    if (s->headdim > 256 || s->dstate > 256 || s->chunk_size > 256) return MAMBA2_ERR_UNSUPPORTED;
    // grid-dimension and index-range limits of the kernels
    if (s->batch > 65535 || s->nheads > 65535) return MAMBA2_ERR_UNSUPPORTED;
    if (s->batch * s->nheads >= ((int64_t)1 << 31)) return MAMBA2_ERR_UNSUPPORTED;
    const int64_t lim = (int64_t)1 << 40;
    if (s->seqlen > lim / 1024 || s->batch * s->seqlen > lim / (s->nheads * s->headdim) ||
        s->batch * s->seqlen > lim / (s->ngroups * s->dstate))
        return MAMBA2_ERR_UNSUPPORTED;
    return MAMBA2_OK;
}

struct Range {
    uintptr_t lo, hi;
};
Range range_of(const void* p, int64_t bytes) {
    return {reinterpret_cast<uintptr_t>(p), reinterpret_cast<uintptr_t>(p) + (uintptr_t)bytes};
}
bool overlap(Range a, Range b) {
    return a.lo != a.hi && b.lo != b.hi && a.lo < b.hi && b.lo < a.hi;
}

// A tensor argument: pointer, byte size, whether it may be null.
struct Arg {
    const void* p;
    int64_t bytes;
    bool optional;
};

mamba2_status check_ptrs(const Arg* in, int nin, const Arg* out, int nout) {
    for (int i = 0; i < nin + nout; ++i) {
        const Arg& a = i < nin ? in[i] : out[i - nin];
        if (!a.p) {
            if (!a.optional && a.bytes > 0) return MAMBA2_ERR_INVALID_ARG;
            continue;
        }
        if (!aligned16(a.p)) return MAMBA2_ERR_INVALID_ARG;
    }
    for (int o = 0; o < nout; ++o) {
        if (!out[o].p) continue;
        const Range ro = range_of(out[o].p, out[o].bytes);
        for (int i = 0; i < nin; ++i)
            if (in[i].p && overlap(ro, range_of(in[i].p, in[i].bytes))) return MAMBA2_ERR_INVALID_ARG;
        for (int j = o + 1; j < nout; ++j)
            if (out[j].p && overlap(ro, range_of(out[j].p, out[j].bytes))) return MAMBA2_ERR_INVALID_ARG;
    }
    return MAMBA2_OK;
}

struct Sizes {
    int64_t x, dt, A, bc, D, G, cs, state;
};
Sizes sizes_of(const mamba2_shape& s) {
    const int64_t e = elt_size(s);
    const int64_t nc = (s.seqlen + s.chunk_size - 1) / s.chunk_size;
    Sizes z;
    z.x = s.batch * s.seqlen * s.nheads * s.headdim * e;
    z.dt = s.batch * s.seqlen * s.nheads * 4;
    z.A = s.nheads * 4;
    z.D = s.nheads * 4;
    z.bc = s.batch * s.seqlen * s.ngroups * s.dstate * e;
    z.G = s.batch * s.nheads * s.seqlen * 4;
    z.cs = s.batch * s.nheads * nc * s.dstate * s.headdim * e;
    z.state = s.batch * s.nheads * s.dstate * s.headdim * 4;
    return z;
}

mamba2_status from_cuda(cudaError_t e) { return e == cudaSuccess ? MAMBA2_OK : MAMBA2_ERR_CUDA; }

// final_state <- initial_state (or zeros) for an empty sequence.
mamba2_status empty_sequence_state(const mamba2_shape& s, const float* init, float* final_state,
                                   cudaStream_t st) {
    if (!final_state || s.batch == 0) return MAMBA2_OK;
    const size_t bytes = (size_t)sizes_of(s).state;
    cudaError_t e = init ? cudaMemcpyAsync(final_state, init, bytes, cudaMemcpyDeviceToDevice, st)
                         : cudaMemsetAsync(final_state, 0, bytes, st);
    return from_cuda(e);
}

int64_t round_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

}  // namespace

cudaError_t ensure_max_dynamic_smem(const void* func, int bytes) {
    static std::mutex mu;
    static std::map<std::pair<int, const void*>, int> done;  // (device, kernel) -> bytes set
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    auto it = done.find({dev, func});
    if (it != done.end() && it->second >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done[{dev, func}] = bytes;
    return e;
}

int sm_count() {
    static std::mutex mu;
    static std::map<int, int> known;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(mu);
    auto it = known.find(dev);
    if (it != known.end()) return it->second;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    known[dev] = n;
    return n;
}

unsigned int* device_status_word() {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    return static_cast<unsigned int*>(p);
}

// Stage drivers shared by the per-stage entry points and mamba2_ssd_fwd.
mamba2_status run_state_pass(const mamba2_shape& s, const StatePassArgs& a, cudaStream_t st) {
    if (s.seqlen == 0) return empty_sequence_state(s, a.init, a.final_state, st);
    if (s.batch == 0) return MAMBA2_OK;
    const Geom g = make_geom(s);
    return from_cuda(launch_state_pass(g, s.dtype == MAMBA2_BF16, a, st));
}

mamba2_status run_chunk_out(const mamba2_shape& s, const ChunkOutArgs& a, cudaStream_t st) {
    if (s.seqlen == 0 || s.batch == 0) return MAMBA2_OK;
    const Geom g = make_geom(s);
    return from_cuda(launch_chunk_out(g, s.dtype == MAMBA2_BF16, a, st));
}

// Whether the forward pass runs an fp32 problem's stage 3 on the tensor cores.
bool fwd_f32_tensor_cores(const mamba2_shape& s) {
    if (s.dtype != MAMBA2_F32 || s.batch == 0 || s.seqlen == 0) return false;
    return use_f32_tensor_cores(make_geom(s), false);
}

// The chunk the forward pass evaluates with.  The output and the final state
// do not depend on the chunk length (regrouping the sums of the chunked form
// changes rounding only), and mamba2_ssd_fwd exposes neither G nor the chunk
// states, so it runs the chunk measured fastest for the shape on GB300:
//  - fp32 shapes the split-bf16 tensor-core kernels cover at chunk 128: 128;
//  - bf16 tensor-core shapes: 128, except with fewer than 16 (batch, head)
//    pairs, where the state pass walks long sequence segments and the
//    caller's chunk is kept (64 becomes 128: chunks of 64 were never the
//    fastest);
//  - everything else (the CUDA-core kernels): the caller's chunk.
// MAMBA2_FWD_CHUNK=given keeps the caller's; =64, =128 or =256 forces one
// (for tests and for timing the candidates on one shape).
int64_t fwd_chunk(const mamba2_shape& s) {
    const char* env = getenv("MAMBA2_FWD_CHUNK");
    if (env && strcmp(env, "given") == 0) return s.chunk_size;
    if (env && (strcmp(env, "64") == 0 || strcmp(env, "128") == 0 || strcmp(env, "256") == 0))
        return atoi(env);
    if (s.batch == 0 || s.seqlen == 0) return s.chunk_size;
    mamba2_shape t = s;
    t.chunk_size = 128;
    if (s.dtype == MAMBA2_F32) return use_f32_tensor_cores(make_geom(t), false) ? 128 : s.chunk_size;
    const bool tc_h = s.headdim == 64 || s.headdim == 128;
    const bool tc_s = s.dstate == 64 || s.dstate == 128 || s.dstate == 256;
    if (!tc_h || !tc_s) return s.chunk_size;
    const int64_t want = (s.batch * s.nheads >= 16 || s.chunk_size == 64) ? 128 : s.chunk_size;
    t.chunk_size = want;
    const Geom g = make_geom(t);
    return (chunk_out_tc_fits(g) && state_pass_tc_fits(g)) ? want : s.chunk_size;
}

mamba2_shape fwd_shape(const mamba2_shape& s) {
    mamba2_shape r = s;
    r.chunk_size = fwd_chunk(s);
    return r;
}

// Segments of the forward pass's state pass (bf16 on tensor cores only).
int fwd_segments(const mamba2_shape& s) {
    if (s.dtype != MAMBA2_BF16 || s.batch == 0 || s.seqlen == 0) return 1;
    return state_pass_segments(make_geom(s));
}

}  // namespace m2

using namespace m2;

extern "C" {

mamba2_status mamba2_chunk_cumsum(const mamba2_shape* shape, const float* dt, const float* A,
                                  float* G, struct CUstream_st* stream) {
    mamba2_status rc = check_shape(shape);
    if (rc != MAMBA2_OK) return rc;
    const Sizes z = sizes_of(*shape);
    const Arg in[] = {{dt, z.dt, false}, {A, z.A, false}};
    const Arg out[] = {{G, z.G, false}};
    if ((rc = check_ptrs(in, 2, out, 1)) != MAMBA2_OK) return rc;
    return from_cuda(launch_chunk_cumsum(make_geom(*shape), dt, A, G, (cudaStream_t)stream));
}

mamba2_status mamba2_state_pass(const mamba2_shape* shape, const void* x, const float* dt,
                                const void* B, const float* G, const float* initial_state,
                                void* chunk_states, float* final_state, struct CUstream_st* stream) {
    mamba2_status rc = check_shape(shape);
    if (rc != MAMBA2_OK) return rc;
    const Sizes z = sizes_of(*shape);
    const Arg in[] = {{x, z.x, false}, {dt, z.dt, false}, {B, z.bc, false}, {G, z.G, false},
                      {initial_state, z.state, true}};
    const Arg out[] = {{chunk_states, z.cs, false}, {final_state, z.state, true}};
    if ((rc = check_ptrs(in, 5, out, 2)) != MAMBA2_OK) return rc;
    const StatePassArgs a{x, dt, B, G, initial_state, chunk_states, final_state};
    return run_state_pass(*shape, a, (cudaStream_t)stream);
}

mamba2_status mamba2_chunk_out(const mamba2_shape* shape, const void* x, const float* dt,
                               const void* B, const void* C, const float* D, const float* G,
                               const void* chunk_states, void* y, struct CUstream_st* stream) {
    mamba2_status rc = check_shape(shape);
    if (rc != MAMBA2_OK) return rc;
    const Sizes z = sizes_of(*shape);
    const Arg in[] = {{x, z.x, false}, {dt, z.dt, false}, {B, z.bc, false}, {C, z.bc, false},
                      {D, z.D, true}, {G, z.G, false}, {chunk_states, z.cs, false}};
    const Arg out[] = {{y, z.x, false}};
    if ((rc = check_ptrs(in, 7, out, 1)) != MAMBA2_OK) return rc;
    const ChunkOutArgs a{x, dt, B, C, D, G, chunk_states, y};
    return run_chunk_out(*shape, a, (cudaStream_t)stream);
}

int64_t mamba2_ssd_fwd_chunk_size(const mamba2_shape* shape) {
    if (check_shape(shape) != MAMBA2_OK) return 0;
    return fwd_chunk(*shape);
}

size_t mamba2_ssd_fwd_workspace_size(const mamba2_shape* user_shape) {
    if (check_shape(user_shape) != MAMBA2_OK) return 0;
    const mamba2_shape si = fwd_shape(*user_shape);  // the chunk the pass runs with
    const mamba2_shape* shape = &si;
    const Sizes z = sizes_of(*shape);
    // fp32 on the tensor cores: G, the fp32 chunk states, then B as bf16
    // hi/lo planes (the bytes of fp32 B)
    if (fwd_f32_tensor_cores(*shape))
        return (size_t)(round_up(z.G, 256) + round_up(z.cs, 256) + round_up(z.bc, 256));
    const int64_t seg = fwd_segments(*shape) > 1 ? state_pass_segment_bytes(make_geom(*shape)) : 0;
    return (size_t)(round_up(z.G, 256) + round_up(z.cs, 256) + round_up(seg, 256));
}

mamba2_status mamba2_ssd_fwd(const mamba2_shape* user_shape, const void* x, const float* dt,
                             const float* A, const void* B, const void* C, const float* D,
                             const float* initial_state, void* y, float* final_state,
                             void* workspace, size_t workspace_bytes, struct CUstream_st* stream) {
    mamba2_status rc = check_shape(user_shape);
    if (rc != MAMBA2_OK) return rc;
    const mamba2_shape si = fwd_shape(*user_shape);  // the chunk the pass runs with
    const mamba2_shape* shape = &si;
    const Sizes z = sizes_of(*shape);
    const size_t need = mamba2_ssd_fwd_workspace_size(user_shape);
    if (workspace_bytes < need) return MAMBA2_ERR_INVALID_ARG;
    if (need > 0 && (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u)))
        return MAMBA2_ERR_INVALID_ARG;
    const Arg in[] = {{x, z.x, false}, {dt, z.dt, false}, {A, z.A, false}, {B, z.bc, false},
                      {C, z.bc, false}, {D, z.D, true}, {initial_state, z.state, true}};
    const Arg out[] = {{y, z.x, false}, {final_state, z.state, true},
                       {workspace, (int64_t)need, true}};
    if ((rc = check_ptrs(in, 7, out, 3)) != MAMBA2_OK) return rc;
    cudaStream_t st = (cudaStream_t)stream;
    if (shape->seqlen == 0) return empty_sequence_state(*shape, initial_state, final_state, st);
    if (shape->batch == 0) return MAMBA2_OK;

    char* ws = static_cast<char*>(workspace);
    float* G = reinterpret_cast<float*>(ws);
    void* cs = ws + round_up(z.G, 256);
    const Geom g = make_geom(*shape);
    if ((rc = from_cuda(launch_chunk_cumsum(g, dt, A, G, st))) != MAMBA2_OK) return rc;
    if (use_fused_forward(g, shape->dtype == MAMBA2_BF16)) {
        // stages 2 and 3 in one kernel: the carried states stay on the chip
        FusedArgs fa{x, dt, B, C, D, G, initial_state, y, final_state};
        fa.pdl = true;
        return from_cuda(launch_ssd_fused(g, fa, st));
    }
    if (fwd_f32_tensor_cores(*shape)) {
        // fp32: stages 2 and 3 on the tensor cores with three products per
        // product, each operand split on the chip into a bf16 hi/lo pair; only
        // B, which every head of a group shares in stage 2, is split once
        // here into hi/lo planes
        void* cs = ws + round_up(z.G, 256);
        void* B2 = static_cast<char*>(cs) + round_up(z.cs, 256);
        if ((rc = from_cuda(launch_split_bf16(static_cast<const float*>(B), B2,
                                              shape->batch * shape->seqlen * shape->ngroups, shape->dstate,
                                              st))) != MAMBA2_OK)
            return rc;
        StatePassArgs sp{x, dt, B2, G, initial_state, cs, final_state};
        sp.split = true;
        if ((rc = from_cuda(launch_state_pass_tc(g, sp, st))) != MAMBA2_OK) return rc;
        const F32ChunkOutArgs co{static_cast<const float*>(x), dt, static_cast<const float*>(B),
                                 static_cast<const float*>(C), D, G, static_cast<const float*>(cs),
                                 static_cast<float*>(y)};
        return from_cuda(launch_chunk_out_f32tc(g, co, st));
    }
    // stages 2 and 3 may start while the stage before them runs (programmatic
    // dependent launch); they wait for it before reading its output
    StatePassArgs sp{x, dt, B, G, initial_state, cs, final_state};
    sp.pdl = true;
    const int nseg = fwd_segments(*shape);
    if (nseg > 1) {
        // few (batch, head) pairs: stage 2 over sequence segments (summary,
        // carry, segment pass), so that every SM walks a part of a sequence
        float* seg = reinterpret_cast<float*>(ws + round_up(z.G, 256) + round_up(z.cs, 256));
        sp.segments = nseg;
        sp.seg_states = seg;
        sp.summary = true;
        if ((rc = from_cuda(launch_state_pass_tc(g, sp, st))) != MAMBA2_OK) return rc;
        if ((rc = from_cuda(launch_state_carry(g, G, seg, nseg, true, st))) != MAMBA2_OK) return rc;
        sp.summary = false;
        if ((rc = from_cuda(launch_state_pass_tc(g, sp, st))) != MAMBA2_OK) return rc;
    } else if ((rc = run_state_pass(*shape, sp, st)) != MAMBA2_OK) {
        return rc;
    }
    ChunkOutArgs co{x, dt, B, C, D, G, cs, y};
    co.pdl = true;
    return run_chunk_out(*shape, co, st);
}

mamba2_status mamba2_ssd_step(const mamba2_shape* shape, const void* x, const float* dt, const float* A,
                              const void* B, const void* C, const float* D, const float* state_in,
                              float* state_out, void* y, struct CUstream_st* stream) {
    mamba2_status rc = check_shape(shape);
    if (rc != MAMBA2_OK) return rc;
    if (shape->seqlen != 1) return MAMBA2_ERR_INVALID_ARG;
    const Sizes z = sizes_of(*shape);
    // In place (state_in == state_out) is allowed: each state element is read
    // and then written by the same thread.  Any other overlap is rejected.
    const bool in_place = state_in != nullptr && state_in == state_out;
    const Arg in[] = {{x, z.x, false},  {dt, z.dt, false}, {A, z.A, false},
                      {B, z.bc, false}, {C, z.bc, false},  {D, z.D, true},
                      {in_place ? nullptr : state_in, z.state, true}};
    const Arg out[] = {{y, z.x, false}, {state_out, z.state, false}};
    if ((rc = check_ptrs(in, 7, out, 2)) != MAMBA2_OK) return rc;
    if (shape->batch == 0) return MAMBA2_OK;
    const SsdStepArgs a{x, dt, A, B, C, D, state_in, state_out, y};
    return from_cuda(launch_ssd_step(make_geom(*shape), shape->dtype == MAMBA2_BF16, a, (cudaStream_t)stream));
}

mamba2_status mamba2_check_device_status(struct CUstream_st* stream) {
    cudaStream_t st = (cudaStream_t)stream;
    unsigned int word = 0;
    if (cudaMemcpyFromSymbolAsync(&word, g_status_word, sizeof(word), 0, cudaMemcpyDeviceToHost, st) !=
        cudaSuccess)
        return MAMBA2_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MAMBA2_ERR_CUDA;
    if (word != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpyToSymbolAsync(g_status_word, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, st) !=
                cudaSuccess ||
            cudaStreamSynchronize(st) != cudaSuccess)
            return MAMBA2_ERR_CUDA;
        return word == MAMBA2_ERR_TIMEOUT ? MAMBA2_ERR_TIMEOUT : MAMBA2_ERR_CUDA;
    }
    return MAMBA2_OK;
}

const char* mamba2_status_string(mamba2_status status) {
    switch (status) {
        case MAMBA2_OK: return "MAMBA2_OK";
        case MAMBA2_ERR_INVALID_ARG: return "MAMBA2_ERR_INVALID_ARG: invalid argument";
        case MAMBA2_ERR_UNSUPPORTED: return "MAMBA2_ERR_UNSUPPORTED: unsupported problem size";
        case MAMBA2_ERR_CUDA: return "MAMBA2_ERR_CUDA: CUDA runtime or launch error";
        case MAMBA2_ERR_TIMEOUT: return "MAMBA2_ERR_TIMEOUT: a bounded device wait ran out";
    }
    return "MAMBA2: unknown status";
}

int mamba2_version(void) { return kVersion; }

}  // extern "C"
