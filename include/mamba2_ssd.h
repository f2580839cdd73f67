/*
 * mamba2_ssd.h — C ABI of the GB300 (sm_103a) Mamba-2 chunked SSD forward pass.
 *
 * Source of the method: "Accelerating Mamba-2 with High-Performance Forward
 * Pass Kernels in NVIDIA CUDA Tile" (NVIDIA technical blog), cited below as
 * [blog §section].  The layer computes, per batch row b and head h
 * [blog §Mamba-2 architecture, the core recurrence and its renamed form]:
 *
 *     a_t = A[h] * dt_t,   h_t = exp(a_t) h_{t-1} + dt_t B_t x_t^T   (h: S x H)
 *     y_t = C_t^T h_t + D[h] x_t
 *
 * chunkwise, in three stages ([blog §Kernel 1], [§Kernel 2], [§Kernel 3]).
 * The output at token t uses the state INCLUDING token t (the diagonal of the
 * causal mask is kept).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All tensor pointers are DEVICE pointers owned by the caller, contiguous
 *    row-major in the layouts given below, 16-byte aligned.  The library
 *    allocates no memory (except where an entry point says otherwise), never
 *    synchronises the stream, and fully overwrites every output.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *    enqueued on it in order; inputs must stay valid until it completes.
 *  - Outputs must not alias inputs.
 *  - Arguments are checked on the host before anything is launched: a bad
 *    pointer, shape or alignment returns MAMBA2_ERR_INVALID_ARG and an
 *    unsupported combination MAMBA2_ERR_UNSUPPORTED, both with nothing
 *    enqueued.  A failed launch returns MAMBA2_ERR_CUDA.
 *  - Device-side waits are bounded.  A kernel whose wait runs out records
 *    MAMBA2_ERR_TIMEOUT in a per-device status word and returns early (its
 *    outputs are then undefined); mamba2_check_device_status reads it.
 *
 * Shapes: b = batch, L = seqlen, nh = nheads, H = headdim, S = dstate,
 * G = ngroups (nh % G == 0; head h uses group h / (nh / G)), T = chunk_size,
 * nc = ceil(L / T).  L need not be a multiple of T: the last chunk may be
 * partial.
 *
 * Tensors:
 *   x            [b, L, nh, H]      dtype          input (values of the layer)
 *   dt           [b, L, nh]         fp32           per-token step, already activated
 *   A            [nh]               fp32           per-head decay rate (normally < 0)
 *   B, C         [b, L, G, S]       dtype          input / output projections
 *   D            [nh]               fp32           skip coefficient; NULL means 0
 *   G (cumsum)   [b, nh, L]         fp32           stage-1 output, log2 units
 *   chunk_states [b, nh, nc, S, H]  dtype          state entering each chunk
 *   initial_state, final_state [b, nh, S, H]  fp32
 *   y            [b, L, nh, H]      dtype          output
 * where dtype is MAMBA2_F32 or MAMBA2_BF16 (x, B, C, y and chunk_states share it).
 */
#ifndef MAMBA2_SSD_H
#define MAMBA2_SSD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t is `struct CUstream_st *` */

#if defined(__GNUC__)
#define MAMBA2_API __attribute__((visibility("default")))
#else
#define MAMBA2_API
#endif

typedef enum {
    MAMBA2_OK = 0,
    MAMBA2_ERR_INVALID_ARG = 1, /* null / misaligned pointer, bad shape, aliasing */
    MAMBA2_ERR_UNSUPPORTED = 2, /* valid but not implemented (sizes beyond the limits below) */
    MAMBA2_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
    MAMBA2_ERR_TIMEOUT = 4      /* a bounded device-side wait ran out */
} mamba2_status;

typedef enum { MAMBA2_F32 = 0, MAMBA2_BF16 = 1 } mamba2_dtype;

/* Problem description.  Limits: every size >= 1 except batch and seqlen
 * (>= 0; an empty problem enqueues only what is needed to write final_state);
 * headdim <= 256; dstate <= 256; chunk_size in [1, 256]; nheads % ngroups == 0. */
typedef struct {
    int64_t batch;
    int64_t seqlen;
    int64_t nheads;
    int64_t headdim;
    int64_t dstate;
    int64_t ngroups;
    int64_t chunk_size;
    int32_t dtype; /* mamba2_dtype */
    int32_t reserved; /* must be 0 */
} mamba2_shape;

/* Stage 1 [blog §Kernel 1]: G[b,h,t] = log2(e) * sum of A[h] * dt[b,k,h] over
 * the tokens k of t's chunk up to and including t (fp32; the sum restarts at
 * every chunk start).  Writes G in the [b, nh, L] layout, so the later stages
 * read each head's decays contiguously. */
MAMBA2_API mamba2_status mamba2_chunk_cumsum(const mamba2_shape* shape, const float* dt, const float* A,
                                  float* G, struct CUstream_st* stream);

/* Stage 2 [blog §Kernel 2]: the state carried across chunks.  For
 * c = 0 .. nc-1: chunk_states[b,h,c] = h (rounded to dtype), then
 *     h <- exp2(G_last) h + sum_{t in chunk c} exp2(G_last - G_t) dt_t B_t x_t^T,
 * G_last being G at the chunk's last token.  h starts at initial_state (NULL
 * means zeros); after the last chunk it is written to final_state (NULL means
 * not written).  Accumulation is fp32; with bf16 the products use bf16
 * operands. */
MAMBA2_API mamba2_status mamba2_state_pass(const mamba2_shape* shape, const void* x, const float* dt,
                                const void* B, const float* G, const float* initial_state,
                                void* chunk_states, float* final_state,
                                struct CUstream_st* stream);

/* Stage 3 [blog §Kernel 3]: the outputs of every chunk from its entering state.
 * For token i of chunk c (h_c = chunk_states[b,h,c]):
 *     y_i = exp2(G_i) C_i^T h_c
 *         + sum_{j in chunk c, j <= i} (C_i . B_j) exp2(G_i - G_j) dt_j x_j + D[h] x_i.
 * The T x T interaction matrix is formed on chip only.  fp32 accumulation;
 * with bf16 the products use bf16 operands. */
MAMBA2_API mamba2_status mamba2_chunk_out(const mamba2_shape* shape, const void* x, const float* dt,
                               const void* B, const void* C, const float* D, const float* G,
                               const void* chunk_states, void* y, struct CUstream_st* stream);

/* Bytes of device workspace mamba2_ssd_fwd needs for `shape` (0 for an
 * invalid shape): G, the chunk states (at the chunk the pass runs with, see
 * mamba2_ssd_fwd), for bf16 problems with too few (batch, head) pairs to fill
 * the GPU the fp32 states at the boundaries of the sequence segments its
 * state pass runs over, and for fp32 problems on the tensor cores B as bf16
 * hi/lo planes.  A pure function of the shape (and of the environment
 * variables MAMBA2_STATE_SEGMENTS, "1" = no segments, MAMBA2_FWD_CHUNK and
 * MAMBA2_FP32_PATH, which force a variant).  The workspace holds
 * intermediates only; its contents on entry do not matter. */
MAMBA2_API size_t mamba2_ssd_fwd_workspace_size(const mamba2_shape* shape);

/* The chunk mamba2_ssd_fwd runs `shape` with (see there): one of 64, 128 or
 * 256 chosen per shape, or shape->chunk_size; 0 for an invalid shape.  A pure
 * function of the shape and of the environment variables named under
 * mamba2_ssd_fwd_workspace_size. */
MAMBA2_API int64_t mamba2_ssd_fwd_chunk_size(const mamba2_shape* shape);

/* The whole forward pass [blog §Mamba-2 architecture, "three kernels"]:
 * y and final_state of the recurrence above, from x, dt, A, B, C, D and an
 * optional initial_state (NULL means zeros; final_state NULL means not
 * written).  `workspace` must be a 256-byte aligned device buffer of at least
 * mamba2_ssd_fwd_workspace_size(shape) bytes, not overlapping any tensor.
 * Enqueues the stages on `stream`.  y and final_state do not depend on the
 * chunk length (it regroups the sums; only rounding changes), and neither G
 * nor the chunk states leave this call, so the pass runs with the chunk
 * measured fastest for the shape (64, 128 or 256), which need not be
 * shape->chunk_size; MAMBA2_FWD_CHUNK=given makes it use shape->chunk_size. */
MAMBA2_API mamba2_status mamba2_ssd_fwd(const mamba2_shape* shape, const void* x, const float* dt,
                             const float* A, const void* B, const void* C, const float* D,
                             const float* initial_state, void* y, float* final_state,
                             void* workspace, size_t workspace_bytes, struct CUstream_st* stream);

/* The whole forward pass for callers that cannot allocate device memory
 * (code running under a custom pool or an allocator-free runtime, or a host
 * that must not grow device memory mid-flight).  The blog has no counterpart;
 * this is a convenience of the library.  Same inputs, outputs and semantics as
 * mamba2_ssd_fwd, but the intermediates live in a fixed 32 MiB device array
 * inside the library (held on every GPU that loads the library until the
 * process exits), so no workspace is passed and nothing is allocated.
 *  - Problems with mamba2_ssd_fwd_workspace_size(shape) > 32 MiB return
 *    MAMBA2_ERR_UNSUPPORTED with nothing enqueued.
 *  - Every call looks up the array's device address on the current device (a
 *    runtime query, no allocation), so the address is never stale after a
 *    device reset.  The first call on a device may also load the library's
 *    device code there; make that first call before any stream capture on
 *    that device.
 *  - All calls share the one array: calls that overlap on the GPU race on it
 *    and must be ordered by the caller (one stream, or explicit events).  The
 *    array's previous contents never affect a result. */
MAMBA2_API mamba2_status mamba2_ssd_fwd_noalloc(const mamba2_shape* shape, const void* x, const float* dt,
                                                const float* A, const void* B, const void* C, const float* D,
                                                const float* initial_state, void* y, float* final_state,
                                                struct CUstream_st* stream);

/* One recurrent step: the single-token decode step that continues each
 * (batch, head) sequence from a carried state [blog §Mamba-2 architecture:
 * the recurrent form is the one suited to sequential inference; §Kernel 2:
 * the final state of a pass is fed back as the next call's initial state].
 *
 *   h  <- exp(A[h] dt[b,h]) h + dt[b,h] B[b,g] x[b,h]^T    (g = h / (nh/G))
 *   y[b,h] = C[b,g]^T h + D[h] x[b,h]                      (updated h)
 *
 * This is mamba2_ssd_fwd on a one-token sequence: `shape->seqlen` must be 1
 * (else MAMBA2_ERR_INVALID_ARG) and chunk_size is not used (any valid value).
 * Layouts are mamba2_ssd_fwd's with L = 1:
 *   x, y        [b, nh, H]  dtype of shape->dtype
 *   dt          [b, nh]     fp32 (already activated, >= 0)
 *   A, D        [nh]        fp32 (D may be NULL: no skip term)
 *   B, C        [b, G, S]   dtype of shape->dtype
 *   state_in    [b, nh, S, H] fp32, NULL means zeros
 *   state_out   [b, nh, S, H] fp32, required
 * state_out may be the same pointer as state_in (update in place); any other
 * overlap between tensors is MAMBA2_ERR_INVALID_ARG.  The decay is computed
 * as exp2(log2(e) * A * dt) in fp32, like stage 1 of the forward pass.  All
 * pointers are caller-owned device memory, 16-byte aligned; nothing is
 * allocated; the step is enqueued on `stream` and never synchronises. */
MAMBA2_API mamba2_status mamba2_ssd_step(const mamba2_shape* shape, const void* x, const float* dt,
                                         const float* A, const void* B, const void* C, const float* D,
                                         const float* state_in, float* state_out, void* y,
                                         struct CUstream_st* stream);

/* Self-test of the bounded device waits (a diagnostic of this library's own
 * failure handling; the blog has no counterpart).  Enqueues one small kernel
 * that holds tensor memory and waits on a barrier that nothing ever completes,
 * with a wall-clock limit of `limit_ns` (1e3 .. 1e8 ns, else
 * MAMBA2_ERR_INVALID_ARG): the wait runs out, the kernel records
 * MAMBA2_ERR_TIMEOUT in the current device's status word, a second waiter in
 * the same kernel leaves through the kernel's abort flag, the tensor memory is
 * freed and the kernel returns.  The next mamba2_check_device_status therefore
 * returns MAMBA2_ERR_TIMEOUT (and clears the word); the context stays usable.
 * Allocates nothing; does not synchronise. */
MAMBA2_API mamba2_status mamba2_selftest_wait_timeout(int64_t limit_ns, struct CUstream_st* stream);

/* Reads (and clears) the current device's status word.  SYNCHRONISES `stream`.
 * Returns MAMBA2_ERR_TIMEOUT if a kernel's bounded wait ran out since the
 * last check, MAMBA2_ERR_CUDA if the stream reports an error, else MAMBA2_OK. */
MAMBA2_API mamba2_status mamba2_check_device_status(struct CUstream_st* stream);

/* Static, human-readable name of a status code. */
MAMBA2_API const char* mamba2_status_string(mamba2_status status);

/* Library version as major * 10000 + minor * 100 + patch. */
MAMBA2_API int mamba2_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MAMBA2_SSD_H */
