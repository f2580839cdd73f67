// k_chunk_cumsum.cu — stage 1, the intra-chunk log2-space cumsum of a_t.
//
// [blog §Kernel 1] "Computing cumulative sums": per (batch, chunk) the
// effective decay a[h] * dt[t, h] is summed along the chunk's tokens for every
// head and scaled by log2(e).  [blog §Mamba-2 performance optimization, GMEM
// layout]: the result is stored head-major, G[b, h, t], so that the later
// stages read one head's decays as one contiguous run.
//
// GB300 mapping: one CTA per (chunk, block of 32 heads, batch).  dt rows of 32
// heads (128 B) are read coalesced into shared memory, each warp scans a
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

    // a_t = A[h] * dt[b, t, h], coalesced over heads.  Thread (r, hh) owns
    // head column hh and rows r, r + 8, ...: all of its loads are issued
    // before the first store, so their latencies overlap.  Rows past the
    // chunk's valid tokens are zero.
    constexpr int kRowsPerPass = kThreads / kHeadsPerCta;       // 8
    constexpr int kPasses = kMaxChunk / kRowsPerPass;           // 32
    const int hh = threadIdx.x % kHeadsPerCta, r = threadIdx.x / kHeadsPerCta;
    const bool hv = hh < nh_here;
    const float a = hv ? A[h0 + hh] : 0.f;
    const float* dcol = dt + (b * g.seqlen + t0) * g.nheads + h0 + hh;
    float v[kPasses];
#pragma unroll
    for (int k = 0; k < kPasses; ++k) {
        const int t = r + kRowsPerPass * k;
        v[k] = (hv && t < tc) ? dcol[(int64_t)t * g.nheads] : 0.f;
    }
#pragma unroll
    for (int k = 0; k < kPasses; ++k) tile[r + kRowsPerPass * k][hh] = a * v[k];
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
    k_chunk_cumsum<<<grid, kThreads, 0, st>>>(dt, A, G, g);
    return cudaGetLastError();
}

}  // namespace m2
