// k_chunk_out_tc.cu — stage 3 on the 5th-generation tensor cores (bf16).
//
// [blog §Kernel 3] computes, per chunk and head,
//     Y = exp2(G) (C h_c) + ((C B^T) . exp2(G_i - G_j) . dt_j . causal M) X + D X.
// GB300 design.  One CTA owns (batch, chunk, 128-row block I of the chunk,
// a block of heads sharing one B/C group):
//   warp 0      TMA producer: C rows of the block and B rows 0..Tj-1 once
//               (Tj = 128 (I + 1)), then per head X rows 0..Tj-1 and h_c;
//   warp 1      TMEM allocator and single-thread tcgen05.mma issuer:
//               CB = C B^T once into TMEM (per group, reused by every head),
//               per head Y = C h_c, then Y += P X;
//   warps 2..9  epilogue (two warps per TMEM lane quadrant, each taking half
//               of the columns): P = CB . decay . dt . mask from TMEM into
//               shared memory as bf16, Y <- exp2(G_i) Y in TMEM, and finally
//               y = Y + D x to global memory.
// The T x T interaction matrix lives only in TMEM, registers and shared
// memory.  Decays: for 32-column groups strictly below the diagonal the
// pairwise factor is evaluated as exp2(G_i - G_r) * exp2(G_r - G_j) with r the
// group's last column (both factors <= 1 because a_t <= 0 makes G
// non-increasing inside a chunk), which needs one exp2 per row and column
// instead of one per element; the diagonal 32 x 32 groups use exp2(G_i - G_j)
// directly and masked entries are selected to zero, never multiplied.
// Every wait is bounded; a timeout sets the status word and the CTA unwinds.
#include "common.cuh"
#include "tc_ptx.cuh"
#include "tmap_host.cuh"

namespace m2 {
namespace {

constexpr int kThreads = 320;
constexpr int kEpiWarps = 8;
constexpr int kSmemLimit = 232448;

struct CoTcParams {
    Geom g;
    int T;           // chunk size (128 or 256)
    int nhb;         // heads per CTA (all in one group)
    int nst;         // X/h pipeline stages
    int head_blocks; // nheads / nhb
    uint32_t off_C, off_P, off_stage, stage_bytes, off_h_in_stage, off_small, off_bar, smem_bytes;
    const float* dt;
    const float* G;
    const float* D;
    __nv_bfloat16* y;
    unsigned int* status;
};

// Barrier slots (uint64 each) inside the barrier area.
enum : int {
    kBarCbFull = 0,
    kBarCbDone = 1,
    kBarPReady = 2,
    kBarEpiSync = 3,
    kBarChDone = 4,     // [2]
    kBarYDone = 6,      // [2]
    kBarYFree = 8,      // [2]
    kBarFull = 10,      // [kMaxStages]
    kBarSlotFree = 12,  // [kMaxStages]
    kNumBars = 14
};
constexpr int kMaxStages = 2;

struct SharedCtl {
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ void set_abort(SharedCtl* ctl, unsigned int* status) {
    ctl->abort = 1;
    if (status) atomicExch(status, kStatusTimeout);
}

__global__ void __launch_bounds__(kThreads, 1)
k_chunk_out_tc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
               const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_h,
               const CoTcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const Geom& g = p.g;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    // ---- which tile
    const int nrb = p.T / 128;
    const int hb = blockIdx.x % p.head_blocks;
    const int I = blockIdx.x / p.head_blocks;  // row block inside the chunk
    const int64_t c = blockIdx.y;
    const int64_t b = blockIdx.z;
    const int h0 = hb * p.nhb;
    const int grp = (int)(h0 / g.heads_per_group);
    const int64_t t0 = c * g.chunk;
    const int tc = (int)imin64(g.chunk, g.seqlen - t0);  // valid tokens of the chunk
    const int Tj = 128 * (I + 1);                         // columns j that rows of block I can see
    const int S = (int)g.dstate, H = (int)g.headdim;
    (void)nrb;

    uint8_t* sC = smem + p.off_C;
    uint8_t* sP = smem + p.off_P;
    uint8_t* sB = sP;  // B lives in [P .. stages) until CB has been computed
    uint8_t* sStage = smem + p.off_stage;
    float* sSmall = reinterpret_cast<float*>(smem + p.off_small);  // [2][3][T]: G, dt, v
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
    SharedCtl* ctl = reinterpret_cast<SharedCtl*>(smem + p.off_bar + kNumBars * 8);

    if (threadIdx.x == 0) {
        tc::mbar_init(&bars[kBarCbFull], 1);
        tc::mbar_init(&bars[kBarCbDone], 1);
        tc::mbar_init(&bars[kBarPReady], kEpiWarps);
        tc::mbar_init(&bars[kBarEpiSync], kEpiWarps);
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&bars[kBarChDone + i], 1);
            tc::mbar_init(&bars[kBarYDone + i], 1);
            tc::mbar_init(&bars[kBarYFree + i], kEpiWarps);
        }
        for (int i = 0; i < kMaxStages; ++i) {
            tc::mbar_init(&bars[kBarFull + i], 1);
            tc::mbar_init(&bars[kBarSlotFree + i], 1 + kEpiWarps);
        }
        ctl->abort = 0;
        tc::fence_barrier_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(&ctl->tmem_base, 512);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    const uint32_t tm_cb = tmem;                          // columns [0, Tj)
    const uint32_t tm_y0 = tmem + 256;                    // Y buffers: 256 .. 256 + 2H
    volatile int* abort_flag = &ctl->abort;

    const uint32_t x_bytes = (uint32_t)Tj * H * 2;
    const uint32_t h_bytes = (uint32_t)S * H * 2;

    if (warp == 0) {
        // =========================== TMA producer ===========================
        if (lane == 0) {
            tc::tma_prefetch_desc(&tm_x);
            tc::tma_prefetch_desc(&tm_b);
            tc::tma_prefetch_desc(&tm_c);
            tc::tma_prefetch_desc(&tm_h);
            tc::mbar_arrive_expect_tx(&bars[kBarCbFull], (uint32_t)(128 * S * 2 + Tj * S * 2));
            for (int kb = 0; kb < S / 64; ++kb) {
                tc::tma_load_4d(sC + kb * 16384, &tm_c, &bars[kBarCbFull], kb * 64, grp, (int)(t0 + 128 * I), (int)b);
                for (int rb = 0; rb < Tj / 128; ++rb)
                    tc::tma_load_4d(sB + kb * (Tj * 128) + rb * 16384, &tm_b, &bars[kBarCbFull], kb * 64, grp,
                                    (int)(t0 + 128 * rb), (int)b);
            }
            bool ok = tc::mbar_wait(&bars[kBarCbDone], 0, abort_flag);  // B region is reused
            for (int k = 0; ok && k < p.nhb; ++k) {
                const int st = k % p.nst;
                if (k >= p.nst && !tc::mbar_wait(&bars[kBarSlotFree + st], ((k / p.nst) - 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                uint8_t* sX = sStage + st * p.stage_bytes;
                uint8_t* sH = sX + p.off_h_in_stage;
                tc::mbar_arrive_expect_tx(&bars[kBarFull + st], x_bytes + h_bytes);
                const int h = h0 + k;
                for (int cb = 0; cb < H / 64; ++cb) {
                    for (int rb = 0; rb < Tj / 128; ++rb)
                        tc::tma_load_4d(sX + cb * (Tj * 128) + rb * 16384, &tm_x, &bars[kBarFull + st], cb * 64, h,
                                        (int)(t0 + 128 * rb), (int)b);
                    tc::tma_load_2d(sH + cb * (S * 128), &tm_h, &bars[kBarFull + st], cb * 64,
                                    (int)(((b * g.nheads + h) * g.nchunks + c) * S));
                }
            }
            if (!ok) set_abort(ctl, p.status);
        }
    } else if (warp == 1) {
        // ============================ MMA issuer ============================
        if (lane == 0) {
            bool ok = tc::mbar_wait(&bars[kBarCbFull], 0, abort_flag);
            if (ok) {
                tc::tc_fence_after();
                const uint32_t id_cb = tc::idesc_bf16(128, Tj, false, false);
                const uint32_t aC = tc::smem_u32(sC), aB = tc::smem_u32(sB);
                for (int k16 = 0; k16 < S / 16; ++k16) {
                    const uint64_t da = tc::sdesc_sw128(aC + (k16 >> 2) * 16384 + (k16 & 3) * 32, 16, 1024);
                    const uint64_t db = tc::sdesc_sw128(aB + (k16 >> 2) * (Tj * 128) + (k16 & 3) * 32, 16, 1024);
                    tc::mma_bf16_ss(tm_cb, da, db, id_cb, k16 > 0);
                }
                tc::mma_commit(&bars[kBarCbDone]);
            }
            const uint32_t id_y = tc::idesc_bf16(128, H, false, true);
            const uint32_t aC = tc::smem_u32(sC), aP = tc::smem_u32(sP);
            for (int k = 0; ok && k < p.nhb; ++k) {
                const int st = k % p.nst, yb = k & 1;
                const uint32_t tm_y = tm_y0 + yb * H;
                uint8_t* sX = sStage + st * p.stage_bytes;
                const uint32_t aX = tc::smem_u32(sX), aH = tc::smem_u32(sX + p.off_h_in_stage);
                if (!tc::mbar_wait(&bars[kBarFull + st], (k / p.nst) & 1, abort_flag)) { ok = false; break; }
                if (k >= 2 && !tc::mbar_wait(&bars[kBarYFree + yb], ((k >> 1) - 1) & 1, abort_flag)) { ok = false; break; }
                tc::tc_fence_after();
                // Y = C h_c   (A: C, K-major over S; B: h_c, MN-major: rows s, columns H)
                for (int k16 = 0; k16 < S / 16; ++k16) {
                    const uint64_t da = tc::sdesc_sw128(aC + (k16 >> 2) * 16384 + (k16 & 3) * 32, 16, 1024);
                    const uint64_t db = tc::sdesc_sw128(aH + k16 * 2048, S * 128, 1024);
                    tc::mma_bf16_ss(tm_y, da, db, id_y, k16 > 0);
                }
                tc::mma_commit(&bars[kBarChDone + yb]);
                if (!tc::mbar_wait(&bars[kBarPReady], k & 1, abort_flag)) { ok = false; break; }
                tc::tc_fence_after();
                // Y += P X   (A: P, K-major over j; B: X, MN-major: rows j, columns H)
                for (int k16 = 0; k16 < Tj / 16; ++k16) {
                    const uint64_t da = tc::sdesc_sw128(aP + (k16 >> 2) * 16384 + (k16 & 3) * 32, 16, 1024);
                    const uint64_t db = tc::sdesc_sw128(aX + k16 * 2048, Tj * 128, 1024);
                    tc::mma_bf16_ss(tm_y, da, db, id_y, 1);
                }
                tc::mma_commit(&bars[kBarYDone + yb]);
                tc::mma_commit(&bars[kBarSlotFree + st]);
            }
            if (!ok) set_abort(ctl, p.status);
        }
    } else {
        // ============================== epilogue ==============================
        const int ew = warp - 2;          // 0..7
        const int q = warp & 3;           // TMEM lane quadrant this warp may access
        const int hf = ew >> 2;           // column half of P and Y handled by this warp
        const int et = ew * 32 + lane;    // 0..255: this thread's column j for per-head vectors
        const int il = q * 32 + lane;     // row inside the block = TMEM lane
        const int i = 128 * I + il;       // row inside the chunk (< Tj)
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        const int T = p.T;
        const int ilo = 128 * I + 32 * q;  // first row of this warp
        bool ok = true;
        int epi_phase = 0;

        // Per-head vectors G_j, dt_j (j = et), fetched one head ahead.
        float g_next = 0.f, dt_next = 0.f;
        auto fetch = [&](int k) {
            const int64_t bh = b * g.nheads + h0 + k;
            const int j = et < tc ? et : tc - 1;  // padding columns repeat the last G, dt = 0
            g_next = (et < Tj) ? p.G[bh * g.seqlen + t0 + j] : 0.f;
            dt_next = (et < Tj && et < tc) ? p.dt[(b * g.seqlen + t0 + et) * g.nheads + h0 + k] : 0.f;
        };
        fetch(0);
        ok = tc::mbar_wait(&bars[kBarCbDone], 0, abort_flag);
        tc::tc_fence_after();
        for (int k = 0; ok && k < p.nhb; ++k) {
            const int h = h0 + k, st = k % p.nst, yb = k & 1;
            float* sG = sSmall + (k & 1) * 3 * T;
            float* sDt = sG + T;
            float* sV = sDt + T;
            {
                // v_j = exp2(G_r - G_j) dt_j, r = last column of j's 32-group (lane 31)
                const float g_r = __shfl_sync(0xffffffffu, g_next, 31);
                if (et < Tj) {
                    sG[et] = g_next;
                    sDt[et] = dt_next;
                    sV[et] = exp2f(g_r - g_next) * dt_next;
                }
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[kBarEpiSync]);
            if (!tc::mbar_wait(&bars[kBarEpiSync], epi_phase & 1, abort_flag)) { ok = false; break; }
            ++epi_phase;
            if (k + 1 < p.nhb) fetch(k + 1);
            const float gi = sG[i];

            // ---- P = CB . decay . dt . mask -> shared memory (bf16, K-major, 128B swizzle)
            for (int gi32 = hf; gi32 < Tj / 32; gi32 += 2) {
                const int j0 = gi32 * 32;
                uint32_t pk[16];
                if (j0 > ilo + 31) {
#pragma unroll
                    for (int e = 0; e < 16; ++e) pk[e] = 0u;
                } else {
                    uint32_t r[32];
                    tc::tmem_ld32(tm_cb + lane_base + j0, r);
                    if (j0 + 31 <= ilo) {
                        const float u = exp2f(gi - sG[j0 + 31]);
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const float a = __uint_as_float(r[2 * e]) * u * sV[j0 + 2 * e];
                            const float bb = __uint_as_float(r[2 * e + 1]) * u * sV[j0 + 2 * e + 1];
                            pk[e] = tc::pack_bf16x2(a, bb);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int ja = j0 + 2 * e, jb = ja + 1;
                            const float a = (ja <= i) ? __uint_as_float(r[2 * e]) * exp2f(gi - sG[ja]) * sDt[ja] : 0.f;
                            const float bb = (jb <= i) ? __uint_as_float(r[2 * e + 1]) * exp2f(gi - sG[jb]) * sDt[jb] : 0.f;
                            pk[e] = tc::pack_bf16x2(a, bb);
                        }
                    }
                }
                uint8_t* pbase = sP + (j0 >> 6) * 16384 + il * 128;
                const int c0 = (j0 & 63) >> 3;
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4) {
                    uint4* dst = reinterpret_cast<uint4*>(pbase + (((c0 + s4) ^ (il & 7)) << 4));
                    *dst = make_uint4(pk[4 * s4], pk[4 * s4 + 1], pk[4 * s4 + 2], pk[4 * s4 + 3]);
                }
            }
            tc::fence_proxy_async_smem();

            // ---- Y <- exp2(G_i) Y (carried-state term) once C h_c is in TMEM
            if (!tc::mbar_wait(&bars[kBarChDone + yb], (k >> 1) & 1, abort_flag)) { ok = false; break; }
            tc::tc_fence_after();
            const float ei = exp2f(gi);
            const uint32_t ycol = tm_y0 + yb * H + hf * (H / 2);
            for (int m = 0; m < H / 64; ++m) {
                uint32_t r[32];
                tc::tmem_ld32(ycol + lane_base + 32 * m, r);
#pragma unroll
                for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * ei);
                tc::tmem_st32(ycol + lane_base + 32 * m, r);
            }
            tc::tmem_wait_st();
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[kBarPReady]);

            // ---- y = Y + D x once P X has been accumulated
            if (!tc::mbar_wait(&bars[kBarYDone + yb], (k >> 1) & 1, abort_flag)) { ok = false; break; }
            tc::tc_fence_after();
            const float dh = p.D ? p.D[h] : 0.f;
            const uint8_t* sX = sStage + st * p.stage_bytes;
            __nv_bfloat16* yrow = p.y + ((b * g.seqlen + t0 + i) * g.nheads + h) * H;
            for (int m = 0; m < H / 64; ++m) {
                const int k0 = hf * (H / 2) + 32 * m;
                uint32_t r[32];
                tc::tmem_ld32(ycol + lane_base + 32 * m, r);
                const uint8_t* xrow = sX + (k0 >> 6) * (Tj * 128) + i * 128;
                const int c0 = (k0 & 63) >> 3;
                uint32_t out[16];
#pragma unroll
                for (int s4 = 0; s4 < 4; ++s4) {
                    const uint4 xv = *reinterpret_cast<const uint4*>(xrow + (((c0 + s4) ^ (i & 7)) << 4));
                    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int cidx = s4 * 8 + 2 * e;
                        const float lo = __uint_as_float(r[cidx]) + dh * tc::bf16_lo(xw[e]);
                        const float hi = __uint_as_float(r[cidx + 1]) + dh * tc::bf16_hi(xw[e]);
                        out[s4 * 4 + e] = tc::pack_bf16x2(lo, hi);
                    }
                }
                if (i < tc) {
                    uint4* dst = reinterpret_cast<uint4*>(yrow + k0);
#pragma unroll
                    for (int s4 = 0; s4 < 4; ++s4)
                        dst[s4] = make_uint4(out[4 * s4], out[4 * s4 + 1], out[4 * s4 + 2], out[4 * s4 + 3]);
                }
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                tc::mbar_arrive(&bars[kBarSlotFree + st]);
                tc::mbar_arrive(&bars[kBarYFree + yb]);
            }
        }
        if (!ok) set_abort(ctl, p.status);
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

}  // namespace

// Shapes the tensor-core stage-3 kernel covers; others use the CUDA-core kernel.
bool chunk_out_tc_supported(const Geom& g) {
    if (g.chunk != 128 && g.chunk != 256) return false;
    if (g.headdim != 64 && g.headdim != 128) return false;
    if (g.dstate != 64 && g.dstate != 128 && g.dstate != 256) return false;
    if (g.batch * g.nheads * g.nchunks * g.dstate >= (int64_t(1) << 31)) return false;
    if (g.batch * g.seqlen >= (int64_t(1) << 31)) return false;
    return true;
}

namespace {
int pick_heads_per_cta(const Geom& g) {
    const int r = (int)g.heads_per_group;
    for (int n = 8; n >= 1; --n)
        if (r % n == 0) return n;
    return 1;
}

bool plan_smem(const Geom& g, CoTcParams& p) {
    const int T = (int)g.chunk, S = (int)g.dstate, H = (int)g.headdim;
    p.off_C = 0;
    p.off_P = p.off_C + 128 * S * 2;
    p.off_stage = p.off_P + 128 * T * 2;
    p.off_h_in_stage = T * H * 2;
    p.stage_bytes = T * H * 2 + S * H * 2;
    for (int nst = kMaxStages; nst >= 1; --nst) {
        const uint32_t stages_end = p.off_stage + nst * p.stage_bytes;
        if (stages_end - p.off_P < (uint32_t)(T * S * 2)) continue;  // B must fit over P + stages
        const uint32_t off_small = stages_end;
        const uint32_t off_bar = off_small + 2 * 3 * T * 4;
        const uint32_t total = off_bar + kNumBars * 8 + 64 + 1024;  // + ctl + alignment slack
        if (total <= (uint32_t)kSmemLimit) {
            p.nst = nst;
            p.off_small = off_small;
            p.off_bar = off_bar;
            p.smem_bytes = total;
            return true;
        }
    }
    return false;
}
}  // namespace

bool chunk_out_tc_fits(const Geom& g) {
    CoTcParams p;
    return chunk_out_tc_supported(g) && plan_smem(g, p);
}

cudaError_t launch_chunk_out_tc(const Geom& g, const ChunkOutArgs& a, cudaStream_t st) {
    CoTcParams p{};
    p.g = g;
    p.T = (int)g.chunk;
    if (!plan_smem(g, p)) return cudaErrorInvalidConfiguration;
    p.nhb = pick_heads_per_cta(g);
    p.head_blocks = (int)(g.nheads / p.nhb);
    p.dt = a.dt;
    p.G = a.G;
    p.D = a.D;
    p.y = static_cast<__nv_bfloat16*>(a.y);
    p.status = device_status_word();
    const uint64_t H = g.headdim, S = g.dstate, nh = g.nheads, L = g.seqlen, G = g.ngroups;
    CUtensorMap tm_x, tm_b, tm_c, tm_h;
    {
        const uint64_t dims[4] = {H, nh, L, (uint64_t)g.batch};
        const uint64_t strides[3] = {H * 2, nh * H * 2, L * nh * H * 2};
        const uint32_t box[4] = {64, 1, 128, 1};
        if (!make_tmap_bf16(&tm_x, a.x, 4, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[4] = {S, G, L, (uint64_t)g.batch};
        const uint64_t strides[3] = {S * 2, G * S * 2, L * G * S * 2};
        const uint32_t box[4] = {64, 1, 128, 1};
        if (!make_tmap_bf16(&tm_b, a.B, 4, dims, strides, box)) return cudaErrorInvalidValue;
        if (!make_tmap_bf16(&tm_c, a.C, 4, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t rows = (uint64_t)g.batch * nh * g.nchunks * S;
        const uint64_t dims[2] = {H, rows};
        const uint64_t strides[1] = {H * 2};
        const uint32_t box[2] = {64, (uint32_t)S};
        if (!make_tmap_bf16(&tm_h, a.chunk_states, 2, dims, strides, box)) return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaFuncSetAttribute(k_chunk_out_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)p.smem_bytes);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(p.head_blocks * (p.T / 128)), (unsigned)g.nchunks, (unsigned)g.batch);
    k_chunk_out_tc<<<grid, kThreads, p.smem_bytes, st>>>(tm_x, tm_b, tm_c, tm_h, p);
    return cudaGetLastError();
}

}  // namespace m2
