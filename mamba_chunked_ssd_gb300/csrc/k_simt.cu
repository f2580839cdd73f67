// k_simt.cu — stages 2 and 3 on the CUDA cores (fp32 FFMA).
//
// These kernels serve the fp32 path (whose 1e-4 tolerance plain tf32 tensor
// cores cannot meet, since tf32 keeps 10 mantissa bits) and every shape the
// tensor-core kernels do not cover (small chunks, head dims other than 64/128,
// state sizes other than 64/128/256).  They compute in fp32 from fp32 or bf16
// inputs, following [blog §Kernel 2] and [blog §Kernel 3] term by term.
#include "common.cuh"

namespace m2 {
namespace {

constexpr int kThreads = 256;

// ----------------------------------------------------------------------------
// Stage 2: [blog §Kernel 2] the sequential chunk loop.  One CTA owns a
// 32 (state) x 64 (head dim) tile of one (batch, head) state and walks the
// chunks in order: store h, then h <- exp2(G_last) h + sum_t w_t B_t x_t^T with
// w_t = dt_t exp2(G_last - G_t).  Thread layout: 8 threads per state row, 8
// consecutive head-dim columns each.
constexpr int kSpS = 32;    // state rows per CTA
constexpr int kSpH = 64;    // head-dim columns per CTA
constexpr int kSpTok = 32;  // tokens staged per step

template <typename E>
__global__ void __launch_bounds__(kThreads)
k_state_pass_simt(const E* __restrict__ x, const float* __restrict__ dt, const E* __restrict__ Bm,
                  const float* __restrict__ G, const float* __restrict__ init,
                  E* __restrict__ chunk_states, float* __restrict__ final_state, Geom g) {
    __shared__ float w_s[256];
    __shared__ float b_s[kSpTok][kSpS + 1];
    __shared__ __align__(16) float x_s[kSpTok][kSpH];

    const int64_t bh = blockIdx.x;
    const int64_t b = bh / g.nheads, h = bh % g.nheads;
    const int64_t grp = h / g.heads_per_group;
    const int s0 = blockIdx.y * kSpS, k0 = blockIdx.z * kSpH;
    const int sl = threadIdx.x / 8, kl = (threadIdx.x % 8) * 8;
    const int s = s0 + sl;
    const bool row_ok = s < g.dstate;
    const int S = (int)g.dstate, H = (int)g.headdim;

    float st[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const int k = k0 + kl + q;
        st[q] = (init && row_ok && k < H) ? init[(bh * S + s) * H + k] : 0.f;
    }
    const float* Gbh = G + bh * g.seqlen;

    for (int64_t c = 0; c < g.nchunks; ++c) {
        // chunk_states[b, h, c] <- h
        if (row_ok) {
            E* dst = chunk_states + ((bh * g.nchunks + c) * S + s) * (int64_t)H;
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (k0 + kl + q < H) dst[k0 + kl + q] = from_f32<E>(st[q]);
        }
        const int64_t t0 = c * g.chunk;
        const int tc = (int)imin64(g.chunk, g.seqlen - t0);
        const float g_last = Gbh[t0 + tc - 1];
        __syncthreads();  // previous chunk's readers of w_s are done
        for (int t = threadIdx.x; t < tc; t += kThreads)
            w_s[t] = dt[(b * g.seqlen + t0 + t) * g.nheads + h] * exp2f(g_last - Gbh[t0 + t]);
        const float carry = exp2f(g_last);
#pragma unroll
        for (int q = 0; q < 8; ++q) st[q] *= carry;

        for (int tb = 0; tb < tc; tb += kSpTok) {
            const int nt = min(kSpTok, tc - tb);
            __syncthreads();
            for (int i = threadIdx.x; i < kSpTok * kSpS; i += kThreads) {
                const int tt = i / kSpS, ss = i % kSpS;
                float v = 0.f;
                if (tt < nt && s0 + ss < S)
                    v = to_f32(Bm[((b * g.seqlen + t0 + tb + tt) * g.ngroups + grp) * S + s0 + ss]);
                b_s[tt][ss] = v;
            }
            for (int i = threadIdx.x; i < kSpTok * kSpH; i += kThreads) {
                const int tt = i / kSpH, kk = i % kSpH;
                float v = 0.f;
                if (tt < nt && k0 + kk < H)
                    v = to_f32(x[((b * g.seqlen + t0 + tb + tt) * g.nheads + h) * H + k0 + kk]);
                x_s[tt][kk] = v;
            }
            __syncthreads();
            for (int tt = 0; tt < nt; ++tt) {
                const float coef = w_s[tb + tt] * b_s[tt][sl];
                const float4 xa = *reinterpret_cast<const float4*>(&x_s[tt][kl]);
                const float4 xb = *reinterpret_cast<const float4*>(&x_s[tt][kl + 4]);
                st[0] = fmaf(coef, xa.x, st[0]);
                st[1] = fmaf(coef, xa.y, st[1]);
                st[2] = fmaf(coef, xa.z, st[2]);
                st[3] = fmaf(coef, xa.w, st[3]);
                st[4] = fmaf(coef, xb.x, st[4]);
                st[5] = fmaf(coef, xb.y, st[5]);
                st[6] = fmaf(coef, xb.z, st[6]);
                st[7] = fmaf(coef, xb.w, st[7]);
            }
        }
    }
    if (final_state && row_ok) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
            if (k0 + kl + q < H) final_state[(bh * S + s) * H + k0 + kl + q] = st[q];
    }
}

// ----------------------------------------------------------------------------
// Stage 3: [blog §Kernel 3].  One CTA owns 32 output rows (tokens) of one
// chunk for one (batch, head).  Phase 1 builds P_ij = (C_i . B_j) for the
// rows' causal window j <= i in registers, then applies the pairwise decay
// exp2(G_i - G_j), dt_j and the mask and parks P in shared memory.  Phase 2
// forms y_i = exp2(G_i) C_i^T h_c + sum_j P_ij x_j + D x_i over 64-column
// slices of the head dim.
constexpr int kCoRows = 32;
constexpr int kCoK = 32;     // state columns staged per step
constexpr int kCoH = 64;     // head-dim columns per slice
constexpr int kMaxChunk = 256;

struct CoSmem {
    float G[kMaxChunk];
    float dt[kMaxChunk];
    float P[kCoRows][kMaxChunk + 1];
    union {
        struct {
            float c[kCoRows][kCoK + 1];
            float b[kMaxChunk][kCoK + 1];
        } p1;
        struct {
            float c[kCoRows][kCoK + 1];
            __align__(16) float v[kCoK][kCoH];  // h rows or x rows
        } p2;
    } u;
};

template <typename E>
__global__ void __launch_bounds__(kThreads)
k_chunk_out_simt(const E* __restrict__ x, const float* __restrict__ dt, const E* __restrict__ Bm,
                 const E* __restrict__ Cm, const float* __restrict__ Dv, const float* __restrict__ G,
                 const E* __restrict__ chunk_states, E* __restrict__ y, Geom g) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    CoSmem& sm = *reinterpret_cast<CoSmem*>(smem_raw);
    const int row_tiles = (int)((g.chunk + kCoRows - 1) / kCoRows);
    const int64_t c = blockIdx.x / row_tiles;
    const int r0 = (blockIdx.x % row_tiles) * kCoRows;  // first row inside the chunk
    const int64_t h = blockIdx.y, b = blockIdx.z;
    const int64_t bh = b * g.nheads + h;
    const int64_t grp = h / g.heads_per_group;
    const int64_t t0 = c * g.chunk;
    const int tc = (int)imin64(g.chunk, g.seqlen - t0);
    if (r0 >= tc) return;
    const int nrows = min(kCoRows, tc - r0);
    const int jmax = r0 + nrows;  // columns j < jmax can be unmasked
    const int S = (int)g.dstate, H = (int)g.headdim;
    const int tid = threadIdx.x;

    for (int t = tid; t < tc; t += kThreads) {
        sm.G[t] = G[bh * g.seqlen + t0 + t];
        sm.dt[t] = dt[(b * g.seqlen + t0 + t) * g.nheads + h];
    }

    // ---- phase 1: P = C B^T restricted to the causal window
    const int il = tid % kCoRows;   // row handled by this thread
    const int jl = tid / kCoRows;   // first column (stride 8)
    float acc[kMaxChunk / 8];
#pragma unroll
    for (int m = 0; m < kMaxChunk / 8; ++m) acc[m] = 0.f;
    for (int sb = 0; sb < S; sb += kCoK) {
        __syncthreads();
        for (int i = tid; i < kCoRows * kCoK; i += kThreads) {
            const int rr = i / kCoK, ss = i % kCoK;
            float v = 0.f;
            if (rr < nrows && sb + ss < S)
                v = to_f32(Cm[((b * g.seqlen + t0 + r0 + rr) * g.ngroups + grp) * S + sb + ss]);
            sm.u.p1.c[rr][ss] = v;
        }
        for (int i = tid; i < jmax * kCoK; i += kThreads) {
            const int jj = i / kCoK, ss = i % kCoK;
            float v = 0.f;
            if (sb + ss < S) v = to_f32(Bm[((b * g.seqlen + t0 + jj) * g.ngroups + grp) * S + sb + ss]);
            sm.u.p1.b[jj][ss] = v;
        }
        __syncthreads();
        const int kk_end = min(kCoK, S - sb);
#pragma unroll
        for (int m = 0; m < kMaxChunk / 8; ++m) {
            const int j = jl + 8 * m;
            if (j < jmax) {
                float a = acc[m];
                for (int kk = 0; kk < kk_end; ++kk) a = fmaf(sm.u.p1.c[il][kk], sm.u.p1.b[j][kk], a);
                acc[m] = a;
            }
        }
    }
    // decay, dt and the causal mask; masked entries are never exponentiated
    {
        const int i = r0 + il;
        const float gi = (il < nrows) ? sm.G[i] : 0.f;
#pragma unroll
        for (int m = 0; m < kMaxChunk / 8; ++m) {
            const int j = jl + 8 * m;
            if (j < jmax) {
                float p = 0.f;
                if (il < nrows && j <= i) p = acc[m] * exp2f(gi - sm.G[j]) * sm.dt[j];
                sm.P[il][j] = p;
            }
        }
    }

    // ---- phase 2: y rows over 64-column slices of H
    const int rl = tid / 8, kl = (tid % 8) * 8;
    const float dcoef = Dv ? Dv[h] : 0.f;
    for (int kb = 0; kb < H; kb += kCoH) {
        float ch[8], px[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) ch[q] = px[q] = 0.f;
        // carried-state term C_i^T h_c
        const E* hc = chunk_states + (bh * g.nchunks + c) * (int64_t)S * H;
        for (int sb = 0; sb < S; sb += kCoK) {
            __syncthreads();
            for (int i = tid; i < kCoRows * kCoK; i += kThreads) {
                const int rr = i / kCoK, ss = i % kCoK;
                float v = 0.f;
                if (rr < nrows && sb + ss < S)
                    v = to_f32(Cm[((b * g.seqlen + t0 + r0 + rr) * g.ngroups + grp) * S + sb + ss]);
                sm.u.p2.c[rr][ss] = v;
            }
            for (int i = tid; i < kCoK * kCoH; i += kThreads) {
                const int ss = i / kCoH, kk = i % kCoH;
                float v = 0.f;
                if (sb + ss < S && kb + kk < H) v = to_f32(hc[(int64_t)(sb + ss) * H + kb + kk]);
                sm.u.p2.v[ss][kk] = v;
            }
            __syncthreads();
            const int kk_end = min(kCoK, S - sb);
            for (int ss = 0; ss < kk_end; ++ss) {
                const float cv = sm.u.p2.c[rl][ss];
#pragma unroll
                for (int q = 0; q < 8; ++q) ch[q] = fmaf(cv, sm.u.p2.v[ss][kl + q], ch[q]);
            }
        }
        // interaction term sum_j P_ij x_j
        for (int jb = 0; jb < jmax; jb += kCoK) {
            const int nj = min(kCoK, jmax - jb);
            __syncthreads();
            for (int i = tid; i < kCoK * kCoH; i += kThreads) {
                const int jj = i / kCoH, kk = i % kCoH;
                float v = 0.f;
                if (jj < nj && kb + kk < H)
                    v = to_f32(x[((b * g.seqlen + t0 + jb + jj) * g.nheads + h) * H + kb + kk]);
                sm.u.p2.v[jj][kk] = v;
            }
            __syncthreads();
            for (int jj = 0; jj < nj; ++jj) {
                const float p = sm.P[rl][jb + jj];
#pragma unroll
                for (int q = 0; q < 8; ++q) px[q] = fmaf(p, sm.u.p2.v[jj][kl + q], px[q]);
            }
        }
        if (rl < nrows) {
            const int64_t tok = t0 + r0 + rl;
            const float carry = exp2f(sm.G[r0 + rl]);
            const E* xr = x + ((b * g.seqlen + tok) * g.nheads + h) * H;
            E* yr = y + ((b * g.seqlen + tok) * g.nheads + h) * H;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int k = kb + kl + q;
                if (k < H) yr[k] = from_f32<E>(carry * ch[q] + px[q] + dcoef * to_f32(xr[k]));
            }
        }
    }
}

}  // namespace

cudaError_t launch_state_pass_simt(const Geom& g, bool bf16, const StatePassArgs& a, cudaStream_t st) {
    dim3 grid((unsigned)(g.batch * g.nheads), (unsigned)((g.dstate + kSpS - 1) / kSpS),
              (unsigned)((g.headdim + kSpH - 1) / kSpH));
    if (bf16)
        k_state_pass_simt<__nv_bfloat16><<<grid, kThreads, 0, st>>>(
            (const __nv_bfloat16*)a.x, a.dt, (const __nv_bfloat16*)a.B, a.G, a.init,
            (__nv_bfloat16*)a.chunk_states, a.final_state, g);
    else
        k_state_pass_simt<float><<<grid, kThreads, 0, st>>>(
            (const float*)a.x, a.dt, (const float*)a.B, a.G, a.init, (float*)a.chunk_states,
            a.final_state, g);
    return cudaGetLastError();
}

cudaError_t launch_chunk_out_simt(const Geom& g, bool bf16, const ChunkOutArgs& a, cudaStream_t st) {
    const int row_tiles = (int)((g.chunk + kCoRows - 1) / kCoRows);
    dim3 grid((unsigned)(g.nchunks * row_tiles), (unsigned)g.nheads, (unsigned)g.batch);
    const size_t smem = sizeof(CoSmem);
    cudaError_t e;
    if (bf16) {
        e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(k_chunk_out_simt<__nv_bfloat16>), (int)smem);
        if (e != cudaSuccess) return e;
        k_chunk_out_simt<__nv_bfloat16><<<grid, kThreads, smem, st>>>(
            (const __nv_bfloat16*)a.x, a.dt, (const __nv_bfloat16*)a.B, (const __nv_bfloat16*)a.C,
            a.D, a.G, (const __nv_bfloat16*)a.chunk_states, (__nv_bfloat16*)a.y, g);
    } else {
        e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(k_chunk_out_simt<float>), (int)smem);
        if (e != cudaSuccess) return e;
        k_chunk_out_simt<float><<<grid, kThreads, smem, st>>>(
            (const float*)a.x, a.dt, (const float*)a.B, (const float*)a.C, a.D, a.G,
            (const float*)a.chunk_states, (float*)a.y, g);
    }
    return cudaGetLastError();
}

}  // namespace m2
