// k_chunk_out_f32tc.cu — stage 3 for fp32 problems on the 5th-generation
// tensor cores.
//
// "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in NVIDIA
// CUDA Tile", §Kernel 3, computes per chunk and head
//     Y = exp2(G) (C h_c) + ((C B^T) . exp2(G_i - G_j) . dt_j . causal M) X + D X.
// The fp32 path must stay within 1e-4 of the exact result, which one tf32 or
// bf16 product cannot.  Here every fp32 operand v is split on chip into
// v_hi = bf16(v) and v_lo = bf16(v - v_hi), and every product is taken as
// u_hi v_hi + u_hi v_lo + u_lo v_hi on the bf16 tensor cores with fp32
// accumulation: the terms left out are below 2^-16 |u v|.  x, B, C and the
// chunk states are read as fp32 (TMA boxes of 32 columns) and split in place
// in shared memory into bf16 tiles of the bf16 kernel's layouts.
//
// GB300 design, the bf16 stage-3 kernel's (k_chunk_out_tc.cu) reduced to
// chunks of 128 tokens and one head stream.  One CTA owns (batch, chunk, up to
// 16 virtual 64-wide heads of one B/C group):
//   warp 0       producer: TMA of C and B once, then per head X and h_c into
//                a ring of stages, its lanes gathering G, dt and D with
//                cp.async; stores y (fp32, TMA) before refilling a stage;
//   warp 1       TMEM allocator; one thread issues every tcgen05.mma;
//   warps 2..17  the hi/lo splits, P formation and the epilogue.
// Once per CTA:  C, B split; CB = C B^T (three products) -> TMEM fp32, masked.
// Per head:
//   X, h_c split in place
//   Z  = C h_c                          three products, B operand from smem
//   P  = CB . w_j  -> P_hi, P_lo         written to TMEM as the A operand
//   Y2 = P X                            three products, A from TMEM
//   y_i = exp2(G_i) Z + u_i Y2 + D x_i   fp32, written over X_hi | X_lo
// with the decay split at the quadrant reference as in the bf16 kernel
// (u_i w_j = exp2(G_i - G_j) dt_j; rows whose u_i would fall below 2^-96 take
// the direct weight).  Every wait is bounded; a timeout sets the status word.
#include "common.cuh"
#include "tc_ptx.cuh"
#include "tmap_host.cuh"

namespace m2 {
namespace {

constexpr int kEpiWarps = 16;
constexpr int kThreads = (2 + kEpiWarps) * 32;
constexpr int kSmemLimit = 232448;
constexpr int kMaxStages = 4;
constexpr int kFillArrivals = 1 + 32;  // the producer's expect-tx, then one per gathering lane
constexpr int H = 64;                  // virtual head width (one MMA's N)
constexpr int T = 128;                 // chunk (one 128-row block)

// TMEM columns (512 allocated): CB fp32 [0, 128); P_hi [128, 192) and P_lo
// [192, 256) (bf16 pairs, the A operand); Z [256, 320); Y2 [320, 384); when
// heads are split ahead, fp32 X of heads k even / odd for D x, [384, 448) /
// [448, 512).
constexpr uint32_t kColCB = 0, kColPhi = 128, kColPlo = 192, kColZ = 256, kColY2 = 320, kColX = 384;

// Shared memory: C_hi | C_lo (128 x S bf16 each), then the stage ring; B_hi |
// B_lo overlay the first stage slots until C B^T is done.  A stage holds
// X_hi [128 x 64] | X_lo | h_hi [S x 64] | h_lo | G[128] dt[128] D; y (fp32,
// two 32-column boxes of 16 KB) is written over X_hi | X_lo.
struct F32Params {
    Geom g;            // chunk 128
    int nhb;           // real heads per CTA
    int vs;            // virtual heads per real head (H_real / 64)
    int head_blocks;   // nheads / nhb
    int nst, rot;      // ring stages; stage slots under B (ring stage i in slot (i + rot) % nst)
    uint32_t off_C1, off_stage, stage_bytes, off_h, off_vec, off_small, off_bar, smem_bytes;
    const float* dt;
    const float* G;
    const float* D;
    unsigned int* status;
};

enum : int {
    kBarCbFull = 0,
    kBarCbSplit,  // C and B split into hi/lo tiles
    kBarSplit,    // [2] head k's X and h_c split (barrier k % 2)
    kBarSplit1,
    kBarCbDone,
    kBarPReady,
    kBarYDone,
    kBarYFree,
    kBarFull,                          // [kMaxStages]
    kBarYReady = kBarFull + kMaxStages,  // [kMaxStages]
    kNumBars = kBarYReady + kMaxStages
};

struct SharedCtl {
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ void set_abort(SharedCtl* ctl, unsigned int* status) {
    ctl->abort = 1;
    if (status) atomicExch(status, kStatusTimeout);
}

constexpr float kMildSpan = 96.f;
constexpr float kWMax = 0x1p120f;

__device__ __forceinline__ float exact_weight(float gi, float gj, float dtj) {
    const float w = exp2f(fminf(gi - gj, kMildSpan)) * dtj;
    return w > kWMax ? kWMax : w;
}

// The pair (hi, lo) of bf16x2 words of two fp32 values: hi = bf16(v),
// lo = bf16(v - hi).
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
    hi = tc::pack_bf16x2(a, b);
    lo = tc::pack_bf16x2(a - tc::bf16_lo(hi), b - tc::bf16_hi(hi));
}

// Splits, in place, a rows x cols fp32 tile loaded by TMA as boxes of 32
// columns (rows x 128 bytes each, 128-byte swizzle) into the bf16 tiles hi
// (at base) and lo (at base + rows cols 2), each in boxes of 64 columns
// (rows x 128 bytes, 128-byte swizzle): the same bytes, laid out as the
// tensor cores read bf16 operands.  A row keeps its lines (row r of every box
// in both layouts), so rows are independent: the 512 threads of the epilogue
// warps (index t) take 512 pieces of 8 columns per round, whole rows, and
// read their round's pieces before the named barrier `bar_id` and write them
// after it.  Every epilogue thread calls it (do_work = false skips the work
// only).
__device__ __forceinline__ void split_tile(uint8_t* base, int rows, int cols, int t, bool do_work, int bar_id) {
    constexpr int kN = kEpiWarps * 32;
    const int per_row = cols / 8;
    const int pieces = rows * per_row;
    const uint32_t lo_off = (uint32_t)rows * cols * 2;
    for (int u0 = 0; u0 < pieces; u0 += kN) {
        const int u = u0 + t;
        const bool mine = do_work && u < pieces;
        const int r = u / per_row, c0 = (u % per_row) * 8;
        float4 f[2];
        if (mine) {
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int c = c0 + 4 * q;
                f[q] = *reinterpret_cast<const float4*>(base + (c >> 5) * (rows * 128) + r * 128 +
                                                        ((((c & 31) >> 2) ^ (r & 7)) << 4));
            }
        }
        asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "r"(kN) : "memory");
        if (mine) {
            uint8_t* dst = base + (c0 >> 6) * (rows * 128) + r * 128 + ((((c0 & 63) >> 3) ^ (r & 7)) << 4);
            uint32_t hi[4], lo[4];
            split2(f[0].x, f[0].y, hi[0], lo[0]);
            split2(f[0].z, f[0].w, hi[1], lo[1]);
            split2(f[1].x, f[1].y, hi[2], lo[2]);
            split2(f[1].z, f[1].w, hi[3], lo[3]);
            *reinterpret_cast<uint4*>(dst) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *reinterpret_cast<uint4*>(dst + lo_off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
    }
    tc::fence_proxy_async_smem();  // the tiles are read by the tensor cores
}

// VS: virtual 64-wide heads per real head (1 or 2).  Every map is fp32 with
// boxes of 32 columns: tm_x, tm_y [b, L, nh, H_real]; tm_b, tm_c
// [b, L, G, S]; tm_h the chunk states, rows [b, nh, nc, S] x H_real.
// AHEAD: split head k + 1 while head k's products run (three or more stages).
template <int VS, bool AHEAD>
__global__ void __launch_bounds__(kThreads, 1)
k_chunk_out_f32tc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
                  const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_h,
                  const __grid_constant__ CUtensorMap tm_y, const F32Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const Geom& g = p.g;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    // blockIdx.x = hb + head_blocks c
    const int hb = (int)(blockIdx.x % (unsigned)p.head_blocks);
    const int64_t c = blockIdx.x / (unsigned)p.head_blocks;
    const int64_t b = blockIdx.y;
    const int64_t t0 = c * T;
    const int tc = (int)imin64(T, g.seqlen - t0);  // valid tokens of the chunk
    const int h0 = hb * p.nhb;
    const int nvh = p.nhb * VS;  // virtual heads of this CTA
    const int grp = (int)(h0 / g.heads_per_group);
    const int S = (int)g.dstate;

    uint8_t* sC = smem;                   // C_hi; C_lo at off_C1
    uint8_t* sC1 = smem + p.off_C1;
    uint8_t* sStage = smem + p.off_stage;
    uint8_t* sB = sStage;                 // B_hi | B_lo, until C B^T is done
    auto slot_of = [&](int i) { return i + p.rot >= p.nst ? i + p.rot - p.nst : i + p.rot; };
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
    SharedCtl* ctl = reinterpret_cast<SharedCtl*>(smem + p.off_bar + kNumBars * 8);

    if (threadIdx.x == 0) {
        tc::mbar_init(&bars[kBarCbFull], 1);
        tc::mbar_init(&bars[kBarCbSplit], kEpiWarps);
        tc::mbar_init(&bars[kBarSplit], kEpiWarps);
        tc::mbar_init(&bars[kBarSplit1], kEpiWarps);
        tc::mbar_init(&bars[kBarCbDone], 1);
        tc::mbar_init(&bars[kBarPReady], kEpiWarps);
        tc::mbar_init(&bars[kBarYDone], 1);
        tc::mbar_init(&bars[kBarYFree], kEpiWarps);
        for (int i = 0; i < kMaxStages; ++i) {
            tc::mbar_init(&bars[kBarFull + i], kFillArrivals);
            tc::mbar_init(&bars[kBarYReady + i], kEpiWarps);
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
    volatile int* abort_flag = &ctl->abort;
    const uint32_t x_tile = T * H * 2;            // X_hi (or X_lo) of a virtual head, bf16 (16 KB)
    const uint32_t h_tile = (uint32_t)S * H * 2;  // h_hi (or h_lo), bf16

    if (warp == 0) {
        // ================= TMA producer, G / dt / D gather, y stores =================
        if (lane == 0) {
            tc::tma_prefetch_desc(&tm_x);
            tc::tma_prefetch_desc(&tm_b);
            tc::tma_prefetch_desc(&tm_c);
            tc::tma_prefetch_desc(&tm_h);
            // C and B as fp32, boxes of 32 columns (split in place afterwards)
            tc::mbar_arrive_expect_tx(&bars[kBarCbFull], (uint32_t)(2 * T * S * 4));
            for (int kb = 0; kb < S / 32; ++kb) {
                tc::tma_load_4d(sC + kb * 16384, &tm_c, &bars[kBarCbFull], kb * 32, grp, (int)t0, (int)b);
                tc::tma_load_4d(sB + kb * 16384, &tm_b, &bars[kBarCbFull], kb * 32, grp, (int)t0, (int)b);
            }
        }
        tc::griddep_wait();  // the chunk states and G come from the previous kernels
        bool ok = true;
        bool b_free = false;  // the slots under B may be filled (C B^T done)
        int st = 0;
        uint32_t slot_phase = 1;  // phase of the stage's previous use
        // y of virtual head kp (fp32, two boxes of 32 columns over X_hi | X_lo)
        auto store_y = [&](int kp, int st_kp, uint32_t ph) -> bool {
            if (!tc::mbar_wait(&bars[kBarYReady + st_kp], ph, abort_flag)) return false;
            const uint8_t* sY = sStage + slot_of(st_kp) * p.stage_bytes;
            for (int cb = 0; cb < 2; ++cb)
                tc::tma_store_4d(&tm_y, sY + cb * 16384, (kp % VS) * H + cb * 32, h0 + kp / VS, (int)t0, (int)b);
            tc::bulk_commit();
            return true;
        };
        for (int k = 0; ok && k < nvh; ++k) {
            if (k >= p.nst) {
                bool w_ok = true;
                if (lane == 0) {
                    w_ok = store_y(k - p.nst, st, slot_phase);
                    tc::bulk_wait_read_all();  // the stage may be overwritten
                }
                if (!__shfl_sync(0xffffffffu, (int)w_ok, 0)) {
                    ok = false;
                    break;
                }
            }
            if (!b_free && (p.rot == 0 || slot_of(st) < p.rot)) {
                if (lane == 0) ok = tc::mbar_wait(&bars[kBarCbDone], 0, abort_flag);
                if (!__shfl_sync(0xffffffffu, (int)ok, 0)) {
                    ok = false;
                    break;
                }
                b_free = true;
            }
            uint8_t* sX = sStage + slot_of(st) * p.stage_bytes;
            float* vG = reinterpret_cast<float*>(sX + p.off_vec);  // G[128], dt[128], D
            float* vDt = vG + T;
            uint64_t* full = &bars[kBarFull + st];
            const int h = h0 + k / VS;
            const int col0 = (k % VS) * H;
            if (lane == 0) {
                // X and h_c as fp32 (the bytes of their hi and lo tiles)
                tc::mbar_arrive_expect_tx(full, 2 * x_tile + 2 * h_tile);
                const int64_t hrow = ((b * g.nheads + h) * g.nchunks + c) * S;
                for (int xb = 0; xb < 2; ++xb) {
                    tc::tma_load_4d(sX + xb * 16384, &tm_x, full, col0 + 32 * xb, h, (int)t0, (int)b);
                    tc::tma_load_2d(sX + p.off_h + xb * (S * 128), &tm_h, full, col0 + 32 * xb, (int)hrow);
                }
            }
            const float* Gh = p.G + (b * g.nheads + h) * g.seqlen + t0;
            const float* dth = p.dt + (b * g.seqlen + t0) * g.nheads + h;
            for (int j = lane; j < T; j += 32) {
                const int jv = j < tc ? j : tc - 1;
                tc::cp_async4(vG + j, Gh + jv, 4);
                tc::cp_async4(vDt + j, dth + (int64_t)jv * g.nheads, j < tc ? 4u : 0u);
            }
            if (lane == 0) tc::cp_async4(vDt + T, p.D ? p.D + h : p.dt, p.D ? 4u : 0u);
            tc::cp_async_mbar_arrive_noinc(full);
            if (++st == p.nst) {
                st = 0;
                slot_phase ^= 1u;
            }
        }
        if (lane == 0) {
            for (int kp = nvh > p.nst ? nvh - p.nst : 0; ok && kp < nvh; ++kp)
                ok = store_y(kp, kp % p.nst, (uint32_t)(kp / p.nst) & 1u);
            tc::bulk_wait_all();
        }
        if (!ok && lane == 0) set_abort(ctl, p.status);
    } else if (warp == 1) {
        // ========================= MMA issuer (one thread) =========================
        if (lane == 0) {
            bool ok = tc::mbar_wait(&bars[kBarCbSplit], 0, abort_flag);
            const uint32_t aC = tc::smem_u32(sC), aC1 = tc::smem_u32(sC1), aB = tc::smem_u32(sB);
            const uint32_t aB1 = aB + T * S * 2;
            if (ok) {
                tc::tc_fence_after();
                // CB = C_hi B_hi^T + C_hi B_lo^T + C_lo B_hi^T  (both K-major over s)
                const uint32_t id_cb = tc::idesc_bf16(128, 128, false, false);
                const uint32_t pa[3] = {aC, aC, aC1}, pb[3] = {aB, aB1, aB};
                for (int ps = 0; ps < 3; ++ps)
                    for (int k16 = 0; k16 < S / 16; ++k16) {
                        const uint32_t off = (k16 >> 2) * 16384 + (k16 & 3) * 32;
                        tc::mma_bf16_ss(tmem + kColCB, tc::sdesc_sw128(pa[ps] + off, 16, 1024),
                                        tc::sdesc_sw128(pb[ps] + off, 16, 1024), id_cb, (ps > 0 || k16 > 0) ? 1u : 0u);
                    }
                tc::mma_commit(&bars[kBarCbDone]);
            }
            const uint32_t id_y = tc::idesc_bf16(128, H, false, true);
            const uint64_t dC0 = tc::sdesc_sw128(aC, 16, 1024), dC1 = tc::sdesc_sw128(aC1, 16, 1024);
            const uint64_t dX0 = tc::sdesc_sw128(tc::smem_u32(sStage), T * 128, 1024);
            const uint64_t dH0 = tc::sdesc_sw128(tc::smem_u32(sStage + p.off_h), S * 128, 1024);
            const uint64_t stage_step = p.stage_bytes >> 4, xlo = x_tile >> 4, hlo = h_tile >> 4;
            int st = 0, pst = slot_of(0);
            uint64_t dstage = pst * stage_step;  // slot offset, in descriptor units
            for (int k = 0; ok && k < nvh; ++k) {
                // the head's X and h_c are split (after their fill)
                if (!tc::mbar_wait(&bars[kBarSplit + (k & 1)], (k >> 1) & 1, abort_flag)) { ok = false; break; }
                if (k >= 1 && !tc::mbar_wait(&bars[kBarYFree], (k - 1) & 1, abort_flag)) { ok = false; break; }
                tc::tc_fence_after();
                const uint64_t dH = dH0 + dstage, dX = dX0 + dstage;
                // Z = C_hi h_hi + C_hi h_lo + C_lo h_hi  (h: rows s = K, columns = N, MN-major)
                const uint64_t za[3] = {dC0, dC0, dC1}, zb[3] = {dH, dH + hlo, dH};
                for (int ps = 0; ps < 3; ++ps)
                    for (int k16 = 0; k16 < S / 16; ++k16)
                        tc::mma_bf16_ss(tmem + kColZ, za[ps] + (k16 >> 2) * 1024 + (k16 & 3) * 2, zb[ps] + 128 * k16,
                                        id_y, (ps > 0 || k16 > 0) ? 1u : 0u);
                if (!tc::mbar_wait(&bars[kBarPReady], k & 1, abort_flag)) { ok = false; break; }
                tc::tc_fence_after();
                // Y2 = P_hi X_hi + P_hi X_lo + P_lo X_hi  (A from TMEM; X: rows j = K, MN-major)
                const uint32_t ya[3] = {kColPhi, kColPhi, kColPlo};
                const uint64_t yb[3] = {dX, dX + xlo, dX};
                for (int ps = 0; ps < 3; ++ps)
#pragma unroll
                    for (int k16 = 0; k16 < 8; ++k16)
                        tc::mma_bf16_ts(tmem + kColY2, tmem + ya[ps] + k16 * 8, yb[ps] + 128 * k16, id_y,
                                        (ps > 0 || k16 > 0) ? 1u : 0u);
                tc::mma_commit(&bars[kBarYDone]);
                if (++st == p.nst) st = 0;
                if (++pst == p.nst) {
                    pst = 0;
                    dstage = 0;
                } else {
                    dstage += stage_step;
                }
            }
            if (!ok) set_abort(ctl, p.status);
        }
    } else {
        // ================== P formation and epilogue (warps 2..17) ==================
        const int e = warp - 2;                 // 0..15
        const int q = warp & 3;                 // TMEM lane quadrant this warp may access
        const int part = e >> 2;                // 32-column group of P; output columns 16 part ..
        const int il = q * 32 + lane;           // row of the chunk = TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        float* wv = reinterpret_cast<float*>(smem + p.off_small) + e * 32;
        const int rq = 32 * q - 1;              // the column before this quadrant (-1: before the chunk)
        const bool visible = part <= q;         // causal: group `part` is seen by this quadrant's rows

        const int t = e * 32 + lane;  // 0..511
        // C and B, loaded as fp32, become their hi/lo tiles
        bool ok = tc::mbar_wait(&bars[kBarCbFull], 0, abort_flag);
        split_tile(sC, T, S, t, ok, 3);
        split_tile(sB, T, S, t, ok, 3);
        __syncwarp();
        if (ok && lane == 0) tc::mbar_arrive(&bars[kBarCbSplit]);
        if (ok) ok = tc::mbar_wait(&bars[kBarCbDone], 0, abort_flag);
        tc::tc_fence_after();
        if (ok && e < 4) {
            // causal mask, once: zero CB above the diagonal inside this
            // quadrant's diagonal 32 x 32 group (the groups right of it are
            // never read)
            uint32_t ra[16], rb[16];
            tc::tmem_ld16_nowait(tmem + kColCB + lane_base + 32 * q, ra);
            tc::tmem_ld16_nowait(tmem + kColCB + lane_base + 32 * q + 16, rb);
            tc::tmem_wait_ld16(ra);
            tc::tmem_wait_ld16(rb);
#pragma unroll
            for (int x = 0; x < 16; ++x) {
                if (x > lane) ra[x] = 0u;
                if (16 + x > lane) rb[x] = 0u;
            }
            tc::tmem_st16(tmem + kColCB + lane_base + 32 * q, ra);
            tc::tmem_st16(tmem + kColCB + lane_base + 32 * q + 16, rb);
            tc::tmem_wait_st();
        }
        tc::tc_fence_before();
        asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
        tc::tc_fence_after();

        // Head j's X and h_c, loaded as fp32, become their hi/lo tiles.  The
        // thread's piece of X (row il, columns [16 part, 16 part + 16)) is
        // the one its output needs: its fp32 values stay in xr for D x, and
        // when heads are split ahead also go to tensor memory (xr is then
        // reused for the next head).  With three or more stages head k + 1 is split while head k's
        // products run, so the issuer finds it ready when it starts on head
        // k + 1 (measured faster); with two, head k + 1's stage is refilled
        // only after head k - 1's y has been stored, too late for that, and
        // each head is split at the start of its own turn.  Every epilogue
        // thread calls this, whatever its waits return; after a failed wait
        // it only skips the work.
        auto split_head = [&](int j, uint32_t (&xr)[16]) {
            const int sj = j % p.nst;
            if (ok) ok = tc::mbar_wait(&bars[kBarFull + sj], (uint32_t)((j / p.nst) & 1), abort_flag);
            uint8_t* sXj = sStage + slot_of(sj) * p.stage_bytes;
            if (ok) {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    const uint4 f = *reinterpret_cast<const uint4*>(
                        sXj + (part >> 1) * (T * 128) + il * 128 + (((4 * (part & 1) + q4) ^ (il & 7)) << 4));
                    xr[4 * q4] = f.x;
                    xr[4 * q4 + 1] = f.y;
                    xr[4 * q4 + 2] = f.z;
                    xr[4 * q4 + 3] = f.w;
                }
            }
            asm volatile("bar.sync 3, %0;" ::"r"(kEpiWarps * 32) : "memory");
            if (ok) {
#pragma unroll
                for (int h8 = 0; h8 < 2; ++h8) {
                    const uint32_t off = il * 128 + (((2 * part + h8) ^ (il & 7)) << 4);
                    uint32_t hi[4], lo[4];
#pragma unroll
                    for (int x = 0; x < 4; ++x)
                        split2(__uint_as_float(xr[8 * h8 + 2 * x]), __uint_as_float(xr[8 * h8 + 2 * x + 1]), hi[x],
                               lo[x]);
                    *reinterpret_cast<uint4*>(sXj + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                    *reinterpret_cast<uint4*>(sXj + x_tile + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                }
                if (AHEAD) {
                    tc::tmem_st16(tmem + kColX + 64 * (j & 1) + lane_base + 16 * part, xr);
                    tc::tmem_wait_st();
                }
            }
            split_tile(sXj + p.off_h, S, H, t, ok, 3);
            __syncwarp();
            if (ok && lane == 0) tc::mbar_arrive(&bars[kBarSplit + (j & 1)]);
        };

        uint32_t xr[16];  // this thread's fp32 piece of X
        if (AHEAD) split_head(0, xr);
        for (int k = 0; k < nvh; ++k) {
            if (!AHEAD) split_head(k, xr);
            const int st = k % p.nst;
            uint8_t* sX = sStage + slot_of(st) * p.stage_bytes;
            float si = 0.f, ui = 0.f, dh = 0.f;
            if (ok) {
                const float* vG = reinterpret_cast<const float*>(sX + p.off_vec);
                const float* vDt = vG + T;
                const float grow = vG[il];
                const float gref = rq < 0 ? 0.f : vG[rq];
                const bool mild = gref - grow <= kMildSpan;  // false for NaN
                const bool all_mild = __all_sync(0xffffffffu, mild);
                if (visible) {
                    const int j = 32 * part + lane;
                    const float wj = exp2f(fminf(gref - vG[j], kMildSpan)) * vDt[j];
                    wv[lane] = wj > kWMax ? kWMax : wj;
                }
                __syncwarp();
                if (!visible) {
                    uint32_t z[8];
#pragma unroll
                    for (int x = 0; x < 8; ++x) z[x] = 0u;
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        tc::tmem_st8(tmem + kColPhi + lane_base + 16 * part + 8 * hh, z);
                        tc::tmem_st8(tmem + kColPlo + lane_base + 16 * part + 8 * hh, z);
                    }
                } else {
                    uint32_t r[2][16];
                    tc::tmem_ld16_nowait(tmem + kColCB + lane_base + 32 * part, r[0]);
                    tc::tmem_ld16_nowait(tmem + kColCB + lane_base + 32 * part + 16, r[1]);
                    tc::tmem_wait_ld16(r[0]);
                    tc::tmem_tie16(r[1]);
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int col = 32 * part + 16 * hh;  // first column of this piece
                        uint32_t phi[8], plo[8];
#pragma unroll
                        for (int e4 = 0; e4 < 4; ++e4) {
                            const float4 w4 = *reinterpret_cast<const float4*>(wv + 16 * hh + 4 * e4);
                            float f0 = w4.x, f1 = w4.y, f2 = w4.z, f3 = w4.w;
                            if (!all_mild && !mild) {
                                const float4 g4 = *reinterpret_cast<const float4*>(vG + col + 4 * e4);
                                const float4 d4 = *reinterpret_cast<const float4*>(vDt + col + 4 * e4);
                                f0 = exact_weight(grow, g4.x, d4.x);
                                f1 = exact_weight(grow, g4.y, d4.y);
                                f2 = exact_weight(grow, g4.z, d4.z);
                                f3 = exact_weight(grow, g4.w, d4.w);
                            }
                            const uint32_t* rr = r[hh] + 4 * e4;
                            split2(__uint_as_float(rr[0]) * f0, __uint_as_float(rr[1]) * f1, phi[2 * e4], plo[2 * e4]);
                            split2(__uint_as_float(rr[2]) * f2, __uint_as_float(rr[3]) * f3, phi[2 * e4 + 1],
                                   plo[2 * e4 + 1]);
                        }
                        tc::tmem_st8(tmem + kColPhi + lane_base + col / 2, phi);
                        tc::tmem_st8(tmem + kColPlo + lane_base + col / 2, plo);
                    }
                }
                tc::tmem_wait_st();
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&bars[kBarPReady]);
                si = exp2f(grow);
                ui = mild ? exp2f(grow - gref) : 1.f;
                dh = vDt[T];
            }
            if (AHEAD && k + 1 < nvh) split_head(k + 1, xr);
            if (ok) ok = tc::mbar_wait(&bars[kBarYDone], k & 1, abort_flag);
            tc::tc_fence_after();
            // ---- y = exp2(G_i) Z + u_i Y2 + D x_i, fp32, 16 columns [16 part, 16 part + 16)
            float yv[16];
            if (ok) {
                uint32_t za[2][8], yb[2][8];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    tc::tmem_ld8_nowait(tmem + kColZ + lane_base + 16 * part + 8 * u, za[u]);
                    tc::tmem_ld8_nowait(tmem + kColY2 + lane_base + 16 * part + 8 * u, yb[u]);
                }
                if (AHEAD) tc::tmem_ld16_nowait(tmem + kColX + 64 * (k & 1) + lane_base + 16 * part, xr);
                tc::tmem_wait_ld8(za[0]);
                tc::tmem_tie8(yb[0]);
                tc::tmem_tie8(za[1]);
                tc::tmem_tie8(yb[1]);
                tc::tmem_tie16(xr);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
#pragma unroll
                    for (int x = 0; x < 4; ++x) {
                        const float x0 = __uint_as_float(xr[8 * u + 2 * x]), x1 = __uint_as_float(xr[8 * u + 2 * x + 1]);
                        yv[8 * u + 2 * x] = fmaf(si, __uint_as_float(za[u][2 * x]),
                                                 fmaf(ui, __uint_as_float(yb[u][2 * x]), dh * x0));
                        yv[8 * u + 2 * x + 1] = fmaf(si, __uint_as_float(za[u][2 * x + 1]),
                                                     fmaf(ui, __uint_as_float(yb[u][2 * x + 1]), dh * x1));
                    }
                }
            }
            // every warp has read its Z, Y2 and X before any y is written over
            // the stage's X tiles
            asm volatile("bar.sync 2, %0;" ::"r"(kEpiWarps * 32) : "memory");
            if (ok) {
                // fp32 y tile: box part / 2 (32 columns, 128 rows x 128 bytes),
                // 16-byte chunks 4 (part % 2) .. + 3 of row il, 128-byte swizzle
                uint8_t* yrow = sX + (part >> 1) * 16384 + il * 128;
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int j2 = 4 * (part & 1) + t;
                    *reinterpret_cast<float4*>(yrow + ((j2 ^ (il & 7)) << 4)) =
                        make_float4(yv[4 * t], yv[4 * t + 1], yv[4 * t + 2], yv[4 * t + 3]);
                }
            }
            // Z and Y2 have been read; y is in the stage for the producer's store
            tc::tc_fence_before();
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (ok && lane == 0) {
                tc::mbar_arrive(&bars[kBarYFree]);
                tc::mbar_arrive(&bars[kBarYReady + st]);
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

// Shared-memory plan: C_hi | C_lo, then the ring; B_hi | B_lo overlay the
// first stage slots.
bool plan_f32(const Geom& g, F32Params& p) {
    const uint32_t S = (uint32_t)g.dstate;
    const uint32_t x_tile = T * H * 2, h_tile = S * H * 2;
    p.off_C1 = T * S * 2;
    p.off_stage = 2 * T * S * 2;
    p.off_h = 2 * x_tile;
    p.off_vec = p.off_h + 2 * h_tile;
    p.stage_bytes = (p.off_vec + (2 * T + 4) * 4 + 1023) / 1024 * 1024;
    const uint32_t b_end = p.off_stage + 2 * T * S * 2;
    for (int nst = kMaxStages; nst >= 1; --nst) {
        const uint32_t stages_end = p.off_stage + nst * p.stage_bytes;
        p.off_small = stages_end > b_end ? stages_end : b_end;
        p.off_bar = p.off_small + kEpiWarps * 32 * 4;
        const uint32_t total = p.off_bar + kNumBars * 8 + 64 + 1024;  // + ctl + alignment slack
        if (total <= (uint32_t)kSmemLimit) {
            p.nst = nst;
            p.smem_bytes = total;
            const uint32_t over = b_end - p.off_stage;
            p.rot = (int)((over + p.stage_bytes - 1) / p.stage_bytes);
            if (p.rot >= nst) p.rot = 0;  // B covers every slot: the first fill waits for C B^T
            return true;
        }
    }
    return false;
}

int heads_per_cta_f32(const Geom& g, int vs) {
    const int r = (int)g.heads_per_group;
    for (int n = 16 / vs; n >= 1; --n)
        if (r % n == 0) return n;
    return 1;
}

}  // namespace

// fp32 shapes this kernel covers; other fp32 shapes run on the CUDA cores.
bool chunk_out_f32tc_fits(const Geom& g) {
    if (g.chunk != 128) return false;
    if (g.headdim != 64 && g.headdim != 128) return false;
    if (g.dstate != 64 && g.dstate != 128) return false;
    if (g.batch * g.seqlen >= (int64_t(1) << 31)) return false;
    if (g.batch * g.nheads * g.nchunks * g.dstate >= (int64_t(1) << 31)) return false;  // state rows
    if (g.nheads * g.nchunks >= (int64_t(1) << 31)) return false;                          // grid.x
    F32Params p;
    return plan_f32(g, p);
}

cudaError_t launch_chunk_out_f32tc(const Geom& g, const F32ChunkOutArgs& a, cudaStream_t st) {
    F32Params p{};
    p.g = g;
    if (!plan_f32(g, p)) return cudaErrorInvalidConfiguration;
    p.vs = (int)(g.headdim / H);
    p.nhb = heads_per_cta_f32(g, p.vs);
    p.head_blocks = (int)(g.nheads / p.nhb);
    p.dt = a.dt;
    p.G = a.G;
    p.D = a.D;
    p.status = device_status_word();
    const uint64_t Hr = g.headdim, S = g.dstate, nh = g.nheads, L = g.seqlen, G = g.ngroups;
    CUtensorMap tm_x, tm_b, tm_c, tm_h, tm_y;
    {
        const uint64_t dims[4] = {Hr, nh, L, (uint64_t)g.batch};
        const uint64_t strides[3] = {Hr * 4, nh * Hr * 4, L * nh * Hr * 4};
        const uint32_t box[4] = {32, 1, 128, 1};
        if (!make_tmap_f32(&tm_x, a.x, 4, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[4] = {S, G, L, (uint64_t)g.batch};
        const uint64_t strides[3] = {S * 4, G * S * 4, L * G * S * 4};
        const uint32_t box[4] = {32, 1, 128, 1};
        if (!make_tmap_f32(&tm_b, a.B, 4, dims, strides, box)) return cudaErrorInvalidValue;
        if (!make_tmap_f32(&tm_c, a.C, 4, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t rows = (uint64_t)g.batch * nh * g.nchunks * S;
        const uint64_t dims[2] = {Hr, rows};
        const uint64_t strides[1] = {Hr * 4};
        const uint32_t box[2] = {32, (uint32_t)S};
        if (!make_tmap_f32(&tm_h, a.cs, 2, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[4] = {Hr, nh, L, (uint64_t)g.batch};
        const uint64_t strides[3] = {Hr * 4, nh * Hr * 4, L * nh * Hr * 4};
        const uint32_t box[4] = {32, 1, 128, 1};
        if (!make_tmap_f32(&tm_y, a.y, 4, dims, strides, box)) return cudaErrorInvalidValue;
    }
    auto kern = (p.vs == 2) ? (p.nst >= 3 ? k_chunk_out_f32tc<2, true> : k_chunk_out_f32tc<2, false>)
                            : (p.nst >= 3 ? k_chunk_out_f32tc<1, true> : k_chunk_out_f32tc<1, false>);
    cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(kern), (int)p.smem_bytes);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((int64_t)p.head_blocks * g.nchunks), (unsigned)g.batch);
    kern<<<grid, kThreads, p.smem_bytes, st>>>(tm_x, tm_b, tm_c, tm_h, tm_y, p);
    return cudaGetLastError();
}

}  // namespace m2
