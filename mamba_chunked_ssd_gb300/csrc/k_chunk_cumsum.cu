// k_chunk_cumsum.cu — stage 1, the intra-chunk log2-space cumsum of a_t.
//
// [blog §Kernel 1] "Computing cumulative sums": per (batch, chunk) the
// effective decay a[h] * dt[t, h] is summed along the chunk's tokens for every
// head and scaled by log2(e).  [blog §Mamba-2 performance optimization, GMEM
// layout]: the result is stored head-major, G[b, h, t], so that the later
// stages read one head's decays as one contiguous run.
//
// GB300 mapping: one CTA per (chunk, block of 32 heads, batch).  dt rows of 32
// heads (128 B) are read coalesced into shared memory (16-byte loads of four
// heads when the head count allows), each warp scans a
// 32-token segment of all 32 heads (one head per lane), segment offsets are
// added in order, and the tile is written back transposed, coalesced along t.
// Pure streaming: every thread issues all of its loads before it stores any of
// them.
#include "common.cuh"

namespace m2 {
namespace {

constexpr int kHeadsPerCta = 32;
constexpr int kThreads = 256;
constexpr int kMaxChunk = 256;

// VEC: nheads % 4 == 0, so every dt row segment of 4 heads starts on a 16-byte
// boundary and is read with one 16-byte load.
template <bool VEC>
__global__ void __launch_bounds__(kThreads)
k_chunk_cumsum(const float* __restrict__ dt, const float* __restrict__ A, float* __restrict__ G,
               Geom g) {
    // The state pass, launched after this kernel with programmatic stream
    // serialization, may start now; it waits for this grid before reading G.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ float tile[kMaxChunk][kHeadsPerCta + 1];
    __shared__ float seg_total[kThreads / 32][kHeadsPerCta];
    const int64_t c = blockIdx.x;
    const int64_t h0 = (int64_t)blockIdx.y * kHeadsPerCta;
    const int64_t b = blockIdx.z;
    const int64_t t0 = c * g.chunk;
    const int tc = (int)imin64(g.chunk, g.seqlen - t0);  // valid tokens (ragged tail)
    const int nh_here = (int)imin64(kHeadsPerCta, g.nheads - h0);
    const float* row0 = dt + (b * g.seqlen + t0) * g.nheads + h0;

    // a_t = A[h] * dt[b, t, h], read coalesced over heads; every thread issues
    // all of its loads before the first store, so their latencies overlap.
    // Rows past the chunk's valid tokens are zero.
    if (VEC) {
        // thread (r, q) owns heads 4q .. 4q+3 and rows r, r + 32, ...: a warp
        // reads four whole 128-byte rows per load
        constexpr int kQuads = kHeadsPerCta / 4;                 // 8
        constexpr int kRowsPerPass = kThreads / kQuads;          // 32
        constexpr int kPasses = kMaxChunk / kRowsPerPass;        // 8
        const int q = threadIdx.x % kQuads, r = threadIdx.x / kQuads;
        const bool hv = 4 * q < nh_here;
        const float4 a4 = hv ? *reinterpret_cast<const float4*>(A + h0 + 4 * q) : make_float4(0.f, 0.f, 0.f, 0.f);
        float4 v[kPasses];
#pragma unroll
        for (int k = 0; k < kPasses; ++k) {
            const int t = r + kRowsPerPass * k;
            v[k] = (hv && t < tc) ? *reinterpret_cast<const float4*>(row0 + (int64_t)t * g.nheads + 4 * q)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int k = 0; k < kPasses; ++k) {
            float* dst = &tile[r + kRowsPerPass * k][4 * q];  // banks r + 4q + i: conflict-free
            dst[0] = a4.x * v[k].x;
            dst[1] = a4.y * v[k].y;
            dst[2] = a4.z * v[k].z;
            dst[3] = a4.w * v[k].w;
        }
    } else {
        // thread (r, hh) owns head column hh and rows r, r + 8, ...
        constexpr int kRowsPerPass = kThreads / kHeadsPerCta;   // 8
        constexpr int kPasses = kMaxChunk / kRowsPerPass;       // 32
        const int hh = threadIdx.x % kHeadsPerCta, r = threadIdx.x / kHeadsPerCta;
        const bool hv = hh < nh_here;
        const float a = hv ? A[h0 + hh] : 0.f;
        float v[kPasses];
#pragma unroll
        for (int k = 0; k < kPasses; ++k) {
            const int t = r + kRowsPerPass * k;
            v[k] = (hv && t < tc) ? row0[(int64_t)t * g.nheads + hh] : 0.f;
        }
#pragma unroll
        for (int k = 0; k < kPasses; ++k) tile[r + kRowsPerPass * k][hh] = a * v[k];
    }
    __syncthreads();

    // Inclusive scan along t.  Warp w scans rows [32 w, 32 w + 32) with one
    // head per lane (conflict-free: a row's 32 heads sit in 32 banks); the
    // segment offsets are then summed from lower segments only, in a fixed
    // order, so G_t never depends on tokens after t.
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int seg0 = 32 * warp;
    float run = 0.f;
#pragma unroll 8
    for (int t = seg0; t < seg0 + 32; ++t) {
        run += tile[t][lane];
        tile[t][lane] = run;
    }
    seg_total[warp][lane] = run;
    __syncthreads();
    float off = 0.f;
    for (int w = 0; w < warp; ++w) off += seg_total[w][lane];
#pragma unroll 8
    for (int t = seg0; t < seg0 + 32; ++t) tile[t][lane] = (tile[t][lane] + off) * kLog2e;
    __syncthreads();

    // G[b, h, t0 + t], coalesced along t.
    for (int hw = warp; hw < nh_here; hw += kThreads / 32) {
        float* out = G + ((b * g.nheads) + h0 + hw) * g.seqlen + t0;
        for (int t = lane; t < tc; t += 32) out[t] = tile[t][hw];
    }
}

}  // namespace

cudaError_t launch_chunk_cumsum(const Geom& g, const float* dt, const float* A, float* G,
                                cudaStream_t st) {
    if (g.batch == 0 || g.seqlen == 0) return cudaSuccess;
    dim3 grid((unsigned)g.nchunks, (unsigned)((g.nheads + kHeadsPerCta - 1) / kHeadsPerCta),
              (unsigned)g.batch);
    if (g.nheads % 4 == 0)
        k_chunk_cumsum<true><<<grid, kThreads, 0, st>>>(dt, A, G, g);
    else
        k_chunk_cumsum<false><<<grid, kThreads, 0, st>>>(dt, A, G, g);
    return cudaGetLastError();
}

}  // namespace m2
