// noalloc.cu — the forward pass for callers that cannot allocate device memory.
//
// Some callers are not allowed to call cudaMalloc (or any allocator) at the
// point where they run the layer: code inside a custom memory pool or an
// allocator-free runtime, callers that must not grow device memory while other
// work is in flight, or plain-C hosts without a device allocator of their own.
// mamba2_ssd_fwd_noalloc serves them: its intermediates (the cumsum G and the
// chunk states) live in one file-scope device array of fixed size, so the
// caller passes only its inputs and outputs.
//
// The array (kScratchBytes) is part of the library's device image: every GPU
// on which the library is loaded holds it until the process exits.  Problems
// whose workspace would exceed it are rejected with MAMBA2_ERR_UNSUPPORTED.
// All calls share the one array, so calls that overlap on the GPU (different
// streams, or different host threads without ordering) race on it.  Nothing in
// the array needs to start at zero: every byte the pass reads it wrote first.
#include "common.cuh"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;  // 32 MiB

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// The name g_noalloc_scratch is only a host-side stand-in; the array's device
// address is looked up on every call, with the caller's device current (a
// runtime query, no allocation), so it is never stale after a cudaDeviceReset
// or a switch of the current device or context.
mamba2_status scratch_address(void** out) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MAMBA2_ERR_CUDA;
    *out = p;
    return MAMBA2_OK;
}

}  // namespace

extern "C" MAMBA2_API mamba2_status mamba2_ssd_fwd_noalloc(const mamba2_shape* shape, const void* x,
                                                           const float* dt, const float* A, const void* B,
                                                           const void* C, const float* D,
                                                           const float* initial_state, void* y,
                                                           float* final_state, struct CUstream_st* stream) {
    const size_t need = mamba2_ssd_fwd_workspace_size(shape);  // 0 for an invalid shape
    if (need > kScratchBytes) return MAMBA2_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    const mamba2_status rc = scratch_address(&scratch);
    if (rc != MAMBA2_OK) return rc;
    return mamba2_ssd_fwd(shape, x, dt, A, B, C, D, initial_state, y, final_state, scratch, kScratchBytes,
                          stream);
}
