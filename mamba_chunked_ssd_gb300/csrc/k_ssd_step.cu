// k_ssd_step.cu — one recurrent step per (batch, head): the single-token
// decode step that continues a sequence from the final state of a forward
// pass ("Accelerating Mamba-2 with High-Performance Forward Pass Kernels in
// NVIDIA CUDA Tile", §Mamba-2 architecture: the recurrent form is the one for
// sequential inference; §Kernel 2: the final state is the next call's initial
// state).
//
//   h <- exp(A[h] dt) h + dt B x^T        (h is S x H, fp32)
//   y  = C^T h + D[h] x                    (the updated state, as in the
//                                           forward pass's chunk output)
//
// The decay is formed as exp2(log2e * A * dt), the same fp32 arithmetic the
// forward pass's stage 1 uses, so a step and a one-token forward pass agree.
//
// The work is a stream over the state: S*H*4 bytes read and written per
// (batch, head), a few hundred bytes of x, B, C besides.  One CTA owns one
// (batch, head); its threads tile the state as (row-slab, 4-column group), read
// whole 16-byte vectors of a row, and keep a partial y for their columns in
// registers.  The partial sums meet in shared memory at the end.
#include <type_traits>

#include "common.cuh"

namespace m2 {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 8;  // independent state loads in flight per thread

template <typename T, int VEC>
__global__ void __launch_bounds__(kThreads) k_ssd_step(Geom g, const T* __restrict__ x,
                                                        const float* __restrict__ dt,
                                                        const float* __restrict__ A, const T* __restrict__ B,
                                                        const T* __restrict__ C, const float* __restrict__ D,
                                                        const float* state_in, float* state_out, T* __restrict__ y) {
    // Shared: the weighted B row (dt * B), the C row, x, and the partial sums.
    __shared__ float s_b[256], s_c[256], s_x[256];
    __shared__ float s_part[kThreads * VEC];

    const int S = (int)g.dstate, H = (int)g.headdim;
    const int64_t h = blockIdx.x, b = blockIdx.y;
    const int64_t grp = h / g.heads_per_group;
    const int tid = threadIdx.x;
    const int cols = H / VEC;              // column groups per row
    const int rows_per_pass = kThreads / cols;
    const int c = tid % cols, r0 = tid / cols;
    const bool active = r0 < rows_per_pass;  // threads beyond rows_per_pass * cols idle
    const int64_t base = (b * g.nheads + h) * (int64_t)S * H;

    // The state stream depends on nothing else: its first pass of loads is in
    // flight before the small loads of dt, B, C and x below (each thread
    // reads and later writes only its own elements, so an in-place update is
    // safe).
    using V = typename std::conditional<VEC == 4, float4, float>::type;
    V hv[kUnroll];
    auto load_pass = [&](int r) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int rr = r + u * rows_per_pass;
            if (rr < S) {
                if (state_in)
                    hv[u] = *reinterpret_cast<const V*>(state_in + base + (int64_t)rr * H + c * VEC);
                else
                    hv[u] = V{};
            }
        }
    };
    if (active) load_pass(r0);

    const float dtv = dt[b * g.nheads + h];
    const float decay = exp2f(kLog2e * (A[h] * dtv));
    const T* xr = x + (b * g.nheads + h) * H;
    const T* br = B + (b * g.ngroups + grp) * S;
    const T* cr = C + (b * g.ngroups + grp) * S;
    for (int i = tid; i < S; i += kThreads) {
        s_b[i] = dtv * to_f32(br[i]);
        s_c[i] = to_f32(cr[i]);
    }
    for (int i = tid; i < H; i += kThreads) s_x[i] = to_f32(xr[i]);
    __syncthreads();

    float acc[VEC];
#pragma unroll
    for (int k = 0; k < VEC; ++k) acc[k] = 0.f;
    float xv[VEC];
#pragma unroll
    for (int k = 0; k < VEC; ++k) xv[k] = s_x[c * VEC + k];

    if (active) {
        for (int r = r0; r < S; r += rows_per_pass * kUnroll) {
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int rr = r + u * rows_per_pass;
                if (rr < S) {
                    float* hp = reinterpret_cast<float*>(&hv[u]);
                    const float bw = s_b[rr], cw = s_c[rr];
#pragma unroll
                    for (int k = 0; k < VEC; ++k) {
                        hp[k] = fmaf(decay, hp[k], bw * xv[k]);
                        acc[k] = fmaf(cw, hp[k], acc[k]);
                    }
                    *reinterpret_cast<V*>(state_out + base + (int64_t)rr * H + c * VEC) = hv[u];
                }
            }
            if (r + rows_per_pass * kUnroll < S) load_pass(r + rows_per_pass * kUnroll);
        }
    }
    // Partial sums, laid out [row-slab][column], then one thread per column adds
    // the slabs in a fixed order.
#pragma unroll
    for (int k = 0; k < VEC; ++k) s_part[r0 * H + c * VEC + k] = active ? acc[k] : 0.f;
    __syncthreads();
    const float dv = D ? D[h] : 0.f;
    for (int j = tid; j < H; j += kThreads) {
        float s = 0.f;
        for (int q = 0; q < rows_per_pass; ++q) s += s_part[q * H + j];
        y[(b * g.nheads + h) * H + j] = from_f32<T>(fmaf(dv, s_x[j], s));
    }
}

template <typename T>
cudaError_t launch_t(const Geom& g, const SsdStepArgs& a, cudaStream_t st) {
    const dim3 grid((unsigned)g.nheads, (unsigned)g.batch);
    const T* x = static_cast<const T*>(a.x);
    const T* B = static_cast<const T*>(a.B);
    const T* C = static_cast<const T*>(a.C);
    T* y = static_cast<T*>(a.y);
    if (g.headdim % 4 == 0)
        k_ssd_step<T, 4><<<grid, kThreads, 0, st>>>(g, x, a.dt, a.A, B, C, a.D, a.state_in, a.state_out, y);
    else
        k_ssd_step<T, 1><<<grid, kThreads, 0, st>>>(g, x, a.dt, a.A, B, C, a.D, a.state_in, a.state_out, y);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ssd_step(const Geom& g, bool bf16, const SsdStepArgs& a, cudaStream_t st) {
    return bf16 ? launch_t<__nv_bfloat16>(g, a, st) : launch_t<float>(g, a, st);
}

}  // namespace m2
