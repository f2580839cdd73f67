// selftest.cu — a self-test of the library's failure handling on the device.
//
// Every wait in the tensor-core kernels is an mbarrier wait bounded by a wall
// clock limit; a wait that runs out sets the CTA's abort flag, records
// MAMBA2_ERR_TIMEOUT in the per-device status word, and the CTA unwinds:
// the other waiters see the flag and stop, tensor memory is freed, the kernel
// returns.  k_wait_selftest runs exactly that sequence on purpose, with a short
// limit, on a barrier that nothing ever arrives on:
//   warp 0   allocates tensor memory (as the real kernels' allocator warp
//            does), then waits on a second never-completed barrier with the
//            full default limit; it must leave through the abort flag long
//            before that limit;
//   warp 1   waits on the first barrier with the caller's limit, gives up,
//            sets the abort flag and the status word.
// Both then meet at the final barrier and warp 0 frees the tensor memory.  No
// address is ever out of range and every wait is bounded, so the kernel
// always returns and the context stays usable.
#include "common.cuh"
#include "tc_ptx.cuh"

namespace m2 {
namespace {

__global__ void __launch_bounds__(64, 1) k_wait_selftest(uint64_t limit_ns, unsigned int* status) {
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bars[0], 1);
        tc::mbar_init(&bars[1], 1);
        abort_flag = 0;
        tc::fence_barrier_init();
    }
    if (warp == 0) {
        tc::tmem_alloc(&tmem_base, 32);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    volatile int* abort_p = &abort_flag;
    if (warp == 1 && lane == 0) {
        // nothing arrives on bars[0]: this wait runs out after limit_ns
        if (!tc::mbar_wait(&bars[0], 0, abort_p, limit_ns)) {
            *abort_p = 1;
            atomicExch(status, kStatusTimeout);
        }
    } else if (warp == 0 && lane == 0) {
        // nothing arrives on bars[1] either; the abort flag ends this wait
        (void)tc::mbar_wait(&bars[1], 0, abort_p);
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem_base, 32);
    }
}

}  // namespace
}  // namespace m2

using namespace m2;

extern "C" MAMBA2_API mamba2_status mamba2_selftest_wait_timeout(int64_t limit_ns, struct CUstream_st* stream) {
    if (limit_ns < 1000 || limit_ns > 100000000) return MAMBA2_ERR_INVALID_ARG;
    unsigned int* status = device_status_word();
    if (!status) return MAMBA2_ERR_CUDA;
    k_wait_selftest<<<1, 64, 0, (cudaStream_t)stream>>>((uint64_t)limit_ns, status);
    return cudaGetLastError() == cudaSuccess ? MAMBA2_OK : MAMBA2_ERR_CUDA;
}
