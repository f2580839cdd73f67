// k_ssd_fused_tc.cu — the state pass and the chunk output in one kernel
// (bf16, 5th-generation tensor cores), so the carried states never leave the
// chip and x is read from HBM once.
//
// "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in NVIDIA
// CUDA Tile" computes the chunk-start states in one kernel (§Kernel 2) and the
// outputs from them in another (§Kernel 3), with the states in global memory
// in between.  Here one CTA owns a pair of heads of one batch row (both read
// the same B, C group) and walks the sequence in blocks of 128 tokens, keeping
// the fp32 state h of both heads in tensor memory.  A chunk of T = 128 is one
// block; a chunk of T = 256 is two, and the second block reads the first one's
// contribution through the state at the block boundary, an exact regrouping of
// the chunk's output formula:
//   y_i = exp2(G_i - G_s) C_i^T h_blk + sum_{j in block, j <= i} (C_i . B_j) exp2(G_i - G_j) dt_j x_j + D x_i
//   h_next = exp2(G_l - G_s) h_blk + sum_{j in block} exp2(G_l - G_j) dt_j B_j x_j^T
// where G is stage 1's chunk-local cumsum (log2 units), G_s its value just
// before the block (0 at a chunk start) and G_l its value at the block's last
// token.  Per block, with the pair's two heads a and b side by side as N:
//   CB  = C B^T                        tcgen05, 128 x 128, K = state
//   Z   = C [h_a | h_b]                tcgen05, N = 128; h in bf16 from the scan
//   Z  <- f_i Z                        epilogue warps, in TMEM
//   P   = CB . w (causal)              P warps, to TMEM as bf16, per head
//   Y   = Z + P X                      tcgen05 accumulating onto Z, A from TMEM
//   y   = u_i Y + D x                  epilogue
//   h  <- exp2(G_l - G_s) h + B^T [w_a . X_a | w_b . X_b]    scan, then tcgen05
// The decay of each P row is split at the column r before its 32-row quadrant:
// exp2(G_i - G_j) dt_j = u_i w_j, u_i = exp2(G_i - G_r) <= 1, w_j =
// exp2(G_r - G_j) dt_j, and exp2(G_i - G_s) = u_i exp2(G_r - G_s); so for such
// rows f_i = exp2(G_r - G_s) <= 1 and u_i Y = exp2(G_i - G_s) Z + (exact P) X.
// Rows whose u_i would fall below 2^-96 take exp2(G_i - G_j) dt_j per entry,
// f_i = exp2(G_i - G_s) and u_i = 1.  With Z rescaled in place the output needs
// one accumulator, so the C B^T product of the next block can start as soon as
// this block's P warps have read CB.  Roles (30 warps):
//   warp 0      X producer: TMA of both heads' X block into a double buffer;
//               its lanes gather G, dt, D and G_s of both heads by cp.async;
//               before refilling a buffer it stores the y the epilogue wrote
//               over that buffer's X (TMA store)
//   warp 1      TMEM allocator; issues CB and the TMA loads of C (one buffer)
//               and B (two buffers)
//   warp 2      issues Z and the state update (the state chain)
//   warp 3      issues P X of head a, then of head b
//   warps 4-19  P formation: (head, column half, TMEM lane quadrant); the
//               first half covers column groups 0-1, the second groups 2-3
//   warps 20-23 epilogue: Z rescaling, then y written over X in shared memory
//   warps 24-27 scan, then fold: h -> bf16 tile for Z and h <- exp2(G_l - G_s) h
//               in TMEM; once Z has read that tile, w . X into the same buffer
// Tensor memory (512 columns): CB fp32 [0,128), Z / Y [128,256) (head a |
// head b), P' bf16 [256,384), h fp32 [384,512).  Every wait is bounded; a
// timeout sets the status word and the CTA unwinds.
#include "common.cuh"
#include "tc_ptx.cuh"
#include "tmap_host.cuh"

namespace m2 {
namespace {

constexpr int kBlk = 128;  // tokens per block
constexpr int kS = 128;    // state rows
constexpr int kH = 64;     // head dim
constexpr int kThreads = 28 * 32;
constexpr int kWarpP0 = 4, kWarpEpi0 = 20, kWarpScan0 = 24;
constexpr int kSmemLimit = 232448;

constexpr uint32_t kColCB = 0, kColZ = 128, kColP = 256, kColH = 384;

// Shared memory (offsets from the 1024-aligned base).  Tiles are 128-byte
// swizzled boxes of 128 rows x 64 bf16 (16 KB).
constexpr uint32_t kBox = 16384;
constexpr uint32_t kOffC = 0;              // C block: states 0-63 | 64-127
constexpr uint32_t kOffB = 2 * kBox;       // B double buffer: [2][states 0-63 | 64-127]
constexpr uint32_t kOffX = 6 * kBox;       // X double buffer: [2][head a | head b]
constexpr uint32_t kOffHW = 10 * kBox;     // h in bf16 (rows = states), then w . X (rows = tokens): head a | b
constexpr uint32_t kOffVec = 12 * kBox;    // per X buffer: G[2][128], dt[2][128], misc[16]
constexpr uint32_t kVecBytes = 2304;
constexpr uint32_t kOffWv = kOffVec + 2 * kVecBytes;  // P warps' column weights [16][64]
constexpr uint32_t kOffBar = kOffWv + 16 * 64 * 4;
// misc: D_a, D_b, G_s of a, b
constexpr int kMiscD = 0, kMiscGs = 2;

enum : int {
    kBarCFull = 0,
    kBarCFree,
    kBarCbDone,
    kBarZDone,
    kBarZScaled,
    kBarY2Done,
    kBarEpiDone,
    kBarHReady,
    kBarWxReady,
    kBarUDone,
    kBarDrainA,
    kBarDrainB,
    kBarDrainC,
    kBarCbRead,                 // the P warps have read CB
    kBarPReady,                 // [2] per head
    kBarBFull = kBarPReady + 2, // [2]
    kBarBFree = kBarBFull + 2,  // [2]
    kBarXFull = kBarBFree + 2,  // [2] X buffer filled (TMA + gathers)
    kBarXRead = kBarXFull + 2,  // [2] the fold warps have read the buffer's X
    kBarYReady = kBarXRead + 2, // [2] the epilogue has written y over the buffer's X
    kNumBars = kBarYReady + 2
};
constexpr uint32_t kSmemBytes = kOffBar + kNumBars * 8 + 64 + 1024;  // + ctl + alignment slack
static_assert(kSmemBytes <= (uint32_t)kSmemLimit, "shared-memory plan too large");

struct FusedParams {
    Geom g;
    const float* dt;
    const float* G;
    const float* D;
    const float* init;
    float* final_state;
    unsigned int* status;
};

struct SharedCtl {
    uint32_t tmem_base;
    int abort;
    int never;  // stays 0: for the bounded drain waits that must not stop at an abort
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

struct Vec {  // one X buffer's gathered per-token values
    float G[2][kBlk];
    float dt[2][kBlk];
    float misc[16];
};
static_assert(sizeof(Vec) <= kVecBytes, "per-buffer vector area too small");

// Issues Y += P_hh X_hh for one head (A: P in TMEM; B: the head's X box,
// MN-major); the accumulator already holds the rescaled Z.
__device__ __forceinline__ void issue_pv(uint32_t tmem, uint64_t dXhead, int hh) {
    const uint32_t id_y = tc::idesc_bf16(128, kH, false, true);
#pragma unroll
    for (int k16 = 0; k16 < kBlk / 16; ++k16)
        tc::mma_bf16_ts(tmem + kColZ + hh * kH, tmem + kColP + hh * 64 + k16 * 8, dXhead + 128 * k16, id_y, 1u);
}

__global__ void __launch_bounds__(kThreads, 1)
k_ssd_fused_tc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
               const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_y,
               const FusedParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const Geom& g = p.g;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int h0 = 2 * (int)blockIdx.x;  // heads h0, h0 + 1
    const int64_t b = blockIdx.y;
    const int grp = (int)(h0 / g.heads_per_group);
    const int T = (int)g.chunk;
    const int nblk = (int)((g.seqlen + kBlk - 1) / kBlk);

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
    SharedCtl* ctl = reinterpret_cast<SharedCtl*>(smem + kOffBar + kNumBars * 8);
    Vec* vecs = reinterpret_cast<Vec*>(smem + kOffVec);

    if (threadIdx.x == 0) {
        tc::mbar_init(&bars[kBarCFull], 1);
        tc::mbar_init(&bars[kBarCFree], 2);     // after the CB and Z products
        tc::mbar_init(&bars[kBarCbDone], 1);
        tc::mbar_init(&bars[kBarZDone], 1);
        tc::mbar_init(&bars[kBarZScaled], 4);
        tc::mbar_init(&bars[kBarY2Done], 1);
        tc::mbar_init(&bars[kBarEpiDone], 4);
        tc::mbar_init(&bars[kBarHReady], 4);
        tc::mbar_init(&bars[kBarWxReady], 4);
        tc::mbar_init(&bars[kBarUDone], 1);
        tc::mbar_init(&bars[kBarDrainA], 1);
        tc::mbar_init(&bars[kBarDrainB], 1);
        tc::mbar_init(&bars[kBarDrainC], 1);
        tc::mbar_init(&bars[kBarCbRead], 16);
        for (int u = 0; u < 2; ++u) {
            tc::mbar_init(&bars[kBarPReady + u], 8);
            tc::mbar_init(&bars[kBarBFull + u], 1);
            tc::mbar_init(&bars[kBarBFree + u], 2);  // after the CB product and the state update
            tc::mbar_init(&bars[kBarXFull + u], 1 + 32);  // expect-tx + one cp.async arrival per lane
            tc::mbar_init(&bars[kBarXRead + u], 4);       // the fold warps
            tc::mbar_init(&bars[kBarYReady + u], 4);      // the epilogue warps
        }
        ctl->abort = 0;
        ctl->never = 0;
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
    volatile int* never = &ctl->never;

    if (warp == 0) {
        // ===================== X producer + per-token gathers =====================
        if (lane == 0) {
            tc::tma_prefetch_desc(&tm_x);
            tc::tma_prefetch_desc(&tm_y);
        }
        tc::griddep_wait();  // G comes from stage 1
        bool ok = true;
        int fills0 = 0, fills1 = 0;  // fills issued per buffer
        for (int k = 0; ok && k < nblk; ++k) {
            const int u = k & 1, v = k >> 1;
            if (k >= 2) {
                // y of block k - 2 sits over this buffer's X: store it, then refill
                bool w_ok = true;
                if (lane == 0) {
                    w_ok = tc::mbar_wait(&bars[kBarYReady + u], (v - 1) & 1, abort_flag);
                    if (w_ok) {
                        for (int hh = 0; hh < 2; ++hh)
                            tc::tma_store_4d(&tm_y, smem + kOffX + u * 2 * kBox + hh * kBox, 0, h0 + hh,
                                             (k - 2) * kBlk, (int)b);
                        tc::bulk_commit();
                        tc::bulk_wait_read_all();
                    }
                }
                if (!__shfl_sync(0xffffffffu, (int)w_ok, 0)) {
                    ok = false;
                    break;
                }
            }
            const int64_t t0 = (int64_t)k * kBlk;
            const int nvalid = (int)imin64(kBlk, g.seqlen - t0);
            const int pos = (int)(t0 % T);  // position of the block in its chunk
            uint8_t* sX = smem + kOffX + u * 2 * kBox;
            Vec* vec = vecs + u;
            uint64_t* full = &bars[kBarXFull + u];
            if (lane == 0) {
                tc::mbar_arrive_expect_tx(full, 2 * kBox);
                for (int hh = 0; hh < 2; ++hh)
                    tc::tma_load_4d(sX + hh * kBox, &tm_x, full, 0, h0 + hh, (int)t0, (int)b);
            }
            // G (past the last valid token: G of the last one), dt (zero there)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const float* Gh = p.G + (b * g.nheads + h0 + hh) * g.seqlen + t0;
                const float* dth = p.dt + (b * g.seqlen + t0) * g.nheads + h0 + hh;
#pragma unroll
                for (int r = 0; r < kBlk / 32; ++r) {
                    const int j = lane + 32 * r;
                    const int jv = j < nvalid ? j : nvalid - 1;
                    tc::cp_async4(&vec->G[hh][j], Gh + jv, 4);
                    tc::cp_async4(&vec->dt[hh][j], dth + (int64_t)jv * g.nheads, j < nvalid ? 4u : 0u);
                }
            }
            if (lane < 2) {
                const int hh = lane;
                // D (zero when absent) and G just before the block (zero at a chunk start)
                tc::cp_async4(&vec->misc[kMiscD + hh], p.D ? p.D + h0 + hh : p.dt, p.D ? 4u : 0u);
                const float* gs = p.G + (b * g.nheads + h0 + hh) * g.seqlen + (pos ? t0 - 1 : t0);
                tc::cp_async4(&vec->misc[kMiscGs + hh], gs, pos ? 4u : 0u);
            }
            tc::cp_async_mbar_arrive_noinc(full);
            if (u) ++fills1; else ++fills0;
        }
        // the last (up to) two blocks' y
        for (int k = nblk - 2 < 0 ? 0 : nblk - 2; ok && k < nblk; ++k) {
            if (lane == 0) {
                const int u = k & 1, v = k >> 1;
                ok = tc::mbar_wait(&bars[kBarYReady + u], v & 1, abort_flag);
                if (ok) {
                    for (int hh = 0; hh < 2; ++hh)
                        tc::tma_store_4d(&tm_y, smem + kOffX + u * 2 * kBox + hh * kBox, 0, h0 + hh, k * kBlk, (int)b);
                    tc::bulk_commit();
                }
            }
            ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
        }
        if (!ok && lane == 0) set_abort(ctl, p.status);
        // no copy of this warp may still be landing or reading when the CTA exits
        if (lane == 0) {
            tc::bulk_wait_all();
            if (fills0 > 0) (void)tc::mbar_wait(&bars[kBarXFull + 0], (fills0 - 1) & 1, never);
            if (fills1 > 0) (void)tc::mbar_wait(&bars[kBarXFull + 1], (fills1 - 1) & 1, never);
        }
    } else if (warp == 1) {
        // ============== issuer of CB, and the C and B loads (TMA) ==============
        if (lane == 0) {
            tc::tma_prefetch_desc(&tm_b);
            tc::tma_prefetch_desc(&tm_c);
            bool ok = true;
            int cfills = 0, bfills0 = 0, bfills1 = 0;
            auto load_b = [&](int k) {
                const int u = k & 1;
                tc::mbar_arrive_expect_tx(&bars[kBarBFull + u], 2 * kBox);
                for (int kb = 0; kb < 2; ++kb)
                    tc::tma_load_4d(smem + kOffB + u * 2 * kBox + kb * kBox, &tm_b, &bars[kBarBFull + u], kb * 64,
                                    grp, k * kBlk, (int)b);
                if (u) ++bfills1; else ++bfills0;
            };
            auto load_c = [&](int k) {
                tc::mbar_arrive_expect_tx(&bars[kBarCFull], 2 * kBox);
                for (int kb = 0; kb < 2; ++kb)
                    tc::tma_load_4d(smem + kOffC + kb * kBox, &tm_c, &bars[kBarCFull], kb * 64, grp, k * kBlk, (int)b);
                ++cfills;
            };
            if (nblk > 0) {
                load_b(0);
                load_c(0);
            }
            const uint32_t aC = tc::smem_u32(smem + kOffC), aB0 = tc::smem_u32(smem + kOffB);
            const uint32_t id_cb = tc::idesc_bf16(128, 128, false, false);
            for (int k = 0; ok && k < nblk; ++k) {
                const int u = k & 1, v = k >> 1;
                if (!tc::mbar_wait(&bars[kBarCFull], k & 1, abort_flag)) { ok = false; break; }
                if (!tc::mbar_wait(&bars[kBarBFull + u], v & 1, abort_flag)) { ok = false; break; }
                // CB of block k - 1 has been read by every P warp
                if (k >= 1 && !tc::mbar_wait(&bars[kBarCbRead], (k - 1) & 1, abort_flag)) { ok = false; break; }
                tc::tc_fence_after();
                // CB = C B^T: both K-major over the state (two boxes of 64)
                const uint32_t aB = aB0 + u * 2 * kBox;
#pragma unroll
                for (int k16 = 0; k16 < kS / 16; ++k16) {
                    const uint32_t off = (k16 >> 2) * kBox + (k16 & 3) * 32;
                    tc::mma_bf16_ss(tmem + kColCB, tc::sdesc_sw128(aC + off, 16, 1024),
                                    tc::sdesc_sw128(aB + off, 16, 1024), id_cb, k16 > 0);
                }
                tc::mma_commit(&bars[kBarCbDone]);
                tc::mma_commit(&bars[kBarCFree]);
                tc::mma_commit(&bars[kBarBFree + u]);
                if (k + 1 < nblk) {
                    // B of block k + 1 into the buffer block k - 1's CB and state update read
                    if (k >= 1 && !tc::mbar_wait(&bars[kBarBFree + (u ^ 1)], ((k - 1) >> 1) & 1, abort_flag)) {
                        ok = false;
                        break;
                    }
                    load_b(k + 1);
                    // C of block k + 1 once block k's CB and Z products read it
                    if (!tc::mbar_wait(&bars[kBarCFree], k & 1, abort_flag)) { ok = false; break; }
                    load_c(k + 1);
                }
            }
            // every MMA this thread issued has completed, and no copy is still
            // landing, before TMEM is freed and the CTA exits
            tc::mma_commit(&bars[kBarDrainA]);
            (void)tc::mbar_wait(&bars[kBarDrainA], 0, never);
            if (cfills > 0) (void)tc::mbar_wait(&bars[kBarCFull], (cfills - 1) & 1, never);
            if (bfills0 > 0) (void)tc::mbar_wait(&bars[kBarBFull + 0], (bfills0 - 1) & 1, never);
            if (bfills1 > 0) (void)tc::mbar_wait(&bars[kBarBFull + 1], (bfills1 - 1) & 1, never);
            if (!ok) set_abort(ctl, p.status);
        }
    } else if (warp == 3) {
        // ============ issuer of P X onto the rescaled Z, head a then head b ============
        if (lane == 0) {
            bool ok = true;
            const uint64_t dX0 = tc::sdesc_sw128(tc::smem_u32(smem + kOffX), kBox, 1024);
            for (int k = 0; ok && k < nblk; ++k) {
                const int u = k & 1, v = k >> 1;
                if (!tc::mbar_wait(&bars[kBarZScaled], k & 1, abort_flag)) { ok = false; break; }
                if (!tc::mbar_wait(&bars[kBarXFull + u], v & 1, abort_flag)) { ok = false; break; }
                for (int hh = 0; hh < 2 && ok; ++hh) {
                    if (!tc::mbar_wait(&bars[kBarPReady + hh], k & 1, abort_flag)) { ok = false; break; }
                    tc::tc_fence_after();
                    issue_pv(tmem, dX0 + (uint64_t)u * ((2 * kBox) >> 4) + (uint64_t)hh * (kBox >> 4), hh);
                }
                if (ok) tc::mma_commit(&bars[kBarY2Done]);
            }
            tc::mma_commit(&bars[kBarDrainC]);
            (void)tc::mbar_wait(&bars[kBarDrainC], 0, never);
            if (!ok) set_abort(ctl, p.status);
        }
    } else if (warp == 2) {
        // ============ issuer of the state chain: Z, state update ============
        if (lane == 0) {
            bool ok = true;
            const uint32_t aC = tc::smem_u32(smem + kOffC);
            const uint32_t id_z = tc::idesc_bf16(128, 2 * kH, false, true);
            const uint32_t id_u = tc::idesc_bf16(128, 2 * kH, true, true);
            // B operands: h (rows = states = K) for Z, then w . X (rows = tokens =
            // K) for the update, both in the shared buffer, MN-major with the two
            // heads' boxes kBox apart; the update's A = B^T, MN-major: rows =
            // tokens = K, the two 64-state boxes kBox apart
            const uint64_t dHW = tc::sdesc_sw128(tc::smem_u32(smem + kOffHW), kBox, 1024);
            const uint64_t dBt0 = tc::sdesc_sw128(tc::smem_u32(smem + kOffB), kBox, 1024);
            for (int k = 0; ok && k < nblk; ++k) {
                const int u = k & 1, v = k >> 1;
                if (!tc::mbar_wait(&bars[kBarCFull], k & 1, abort_flag)) { ok = false; break; }
                if (!tc::mbar_wait(&bars[kBarHReady], k & 1, abort_flag)) { ok = false; break; }
                if (k >= 1 && !tc::mbar_wait(&bars[kBarEpiDone], (k - 1) & 1, abort_flag)) { ok = false; break; }
                tc::tc_fence_after();
                // Z = C [h_a | h_b]   (K = state)
#pragma unroll
                for (int k16 = 0; k16 < kS / 16; ++k16)
                    tc::mma_bf16_ss(tmem + kColZ,
                                    tc::sdesc_sw128(aC + (k16 >> 2) * kBox + (k16 & 3) * 32, 16, 1024),
                                    dHW + 128 * k16, id_z, k16 > 0);
                tc::mma_commit(&bars[kBarZDone]);
                tc::mma_commit(&bars[kBarCFree]);
                // h += B^T [w_a . X_a | w_b . X_b]   (K = token; h already scaled by the scan)
                if (!tc::mbar_wait(&bars[kBarBFull + u], v & 1, abort_flag)) { ok = false; break; }
                if (!tc::mbar_wait(&bars[kBarWxReady], k & 1, abort_flag)) { ok = false; break; }
                tc::tc_fence_after();
                const uint64_t dBt = dBt0 + (uint64_t)u * ((2 * kBox) >> 4);
#pragma unroll
                for (int k16 = 0; k16 < kBlk / 16; ++k16)
                    tc::mma_bf16_ss(tmem + kColH, dBt + 128 * k16, dHW + 128 * k16, id_u, 1u);
                tc::mma_commit(&bars[kBarUDone]);
                tc::mma_commit(&bars[kBarBFree + u]);
            }
            tc::mma_commit(&bars[kBarDrainB]);
            (void)tc::mbar_wait(&bars[kBarDrainB], 0, never);
            if (!ok) set_abort(ctl, p.status);
        }
    } else if (warp < kWarpEpi0) {
        // ======== P formation (warps 4-19: head, column half, lane quadrant) ========
        const int q = warp & 3;
        const int role = (warp - kWarpP0) >> 2;  // 0..3
        const int hh = role & 1, part = role >> 1;
        const int i = 32 * q + lane;  // row of the block = TMEM lane
        const int g_lo = 2 * part, g_hi = imin64(2 * part + 1, q);  // column groups with entries
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        const uint32_t tp = tmem + kColP + hh * 64 + lane_base;
        float* wv = reinterpret_cast<float*>(smem + kOffWv) + (warp - kWarpP0) * 64;  // w of groups g_lo, g_lo + 1
        bool ok = true;
        for (int k = 0; k < nblk; ++k) {
            const int u = k & 1, v = k >> 1;
            if (ok) ok = tc::mbar_wait(&bars[kBarCbDone], k & 1, abort_flag);
            if (ok) ok = tc::mbar_wait(&bars[kBarXFull + u], v & 1, abort_flag);
            if (ok && k >= 1) ok = tc::mbar_wait(&bars[kBarY2Done], (k - 1) & 1, abort_flag);  // P free
            if (!ok) break;
            tc::tc_fence_after();
            const Vec* vec = vecs + u;
            const float grow = vec->G[hh][i];
            const float gref = q == 0 ? vec->misc[kMiscGs + hh] : vec->G[hh][32 * q - 1];
            const bool mild = gref - grow <= kMildSpan;  // false for NaN
            const bool all_mild = __all_sync(0xffffffffu, mild);
            for (int gi = g_lo; gi <= g_hi; ++gi) {
                const int j = 32 * gi + lane;
                const float wj = exp2f(fminf(gref - vec->G[hh][j], kMildSpan)) * vec->dt[hh][j];
                wv[32 * (gi - g_lo) + lane] = wj > kWMax ? kWMax : wj;
            }
            __syncwarp();
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                const int gi = g_lo + t;
                if (gi > g_hi) {
                    uint32_t z[8];
#pragma unroll
                    for (int x = 0; x < 8; ++x) z[x] = 0u;
                    tc::tmem_st8(tp + 16 * gi, z);
                    tc::tmem_st8(tp + 16 * gi + 8, z);
                    continue;
                }
                uint32_t r[2][16];
                tc::tmem_ld16_nowait(tmem + kColCB + lane_base + 32 * gi, r[0]);
                tc::tmem_ld16_nowait(tmem + kColCB + lane_base + 32 * gi + 16, r[1]);
                tc::tmem_wait_ld16(r[0]);
                tc::tmem_tie16(r[1]);
                if (gi == g_hi) {
                    // this warp's last read of CB: the next block's CB may be written
                    tc::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(&bars[kBarCbRead]);
                }
                if (gi == q) {  // causal mask inside the diagonal 32 x 32 group
#pragma unroll
                    for (int x = 0; x < 16; ++x) {
                        if (x > lane) r[0][x] = 0u;
                        if (16 + x > lane) r[1][x] = 0u;
                    }
                }
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int col = 32 * gi + 16 * half;
                    const float* w = wv + 32 * t + 16 * half;
                    const uint32_t* rr = r[half];
                    uint32_t pk[8];
                    if (all_mild) {
#pragma unroll
                        for (int e4 = 0; e4 < 4; ++e4) {
                            const float4 v4 = *reinterpret_cast<const float4*>(w + 4 * e4);
                            const int o = 4 * e4;
                            const float2 p0 = tc::mul_f32x2(
                                make_float2(__uint_as_float(rr[o]), __uint_as_float(rr[o + 1])), make_float2(v4.x, v4.y));
                            const float2 p1 = tc::mul_f32x2(
                                make_float2(__uint_as_float(rr[o + 2]), __uint_as_float(rr[o + 3])), make_float2(v4.z, v4.w));
                            pk[2 * e4] = tc::pack_bf16x2(p0.x, p0.y);
                            pk[2 * e4 + 1] = tc::pack_bf16x2(p1.x, p1.y);
                        }
                    } else {
                        // per row: the split weight (mild rows, the same products
                        // as above) or the direct one
                        const float* gj = &vec->G[hh][col];
                        const float* dj = &vec->dt[hh][col];
#pragma unroll
                        for (int e4 = 0; e4 < 4; ++e4) {
                            const float4 v4 = *reinterpret_cast<const float4*>(w + 4 * e4);
                            const float4 g4 = *reinterpret_cast<const float4*>(gj + 4 * e4);
                            const float4 d4 = *reinterpret_cast<const float4*>(dj + 4 * e4);
                            const int o = 4 * e4;
                            const float f0 = mild ? v4.x : exact_weight(grow, g4.x, d4.x);
                            const float f1 = mild ? v4.y : exact_weight(grow, g4.y, d4.y);
                            const float f2 = mild ? v4.z : exact_weight(grow, g4.z, d4.z);
                            const float f3 = mild ? v4.w : exact_weight(grow, g4.w, d4.w);
                            pk[2 * e4] = tc::pack_bf16x2(__uint_as_float(rr[o]) * f0, __uint_as_float(rr[o + 1]) * f1);
                            pk[2 * e4 + 1] =
                                tc::pack_bf16x2(__uint_as_float(rr[o + 2]) * f2, __uint_as_float(rr[o + 3]) * f3);
                        }
                    }
                    tc::tmem_st8(tp + col / 2, pk);
                }
            }
            if (g_hi < g_lo) {
                // no column group of this warp has entries (second half, quadrants 0-1)
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&bars[kBarCbRead]);
            }
            tc::tmem_wait_st();
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[kBarPReady + hh]);
        }
        if (!ok) set_abort(ctl, p.status);
    } else if (warp < kWarpScan0) {
        // ========================= epilogue (warps 20-23) =========================
        const int q = warp & 3;
        const int i = 32 * q + lane;
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        bool ok = true;
        for (int k = 0; ok && k < nblk; ++k) {
            const int u = k & 1, v = k >> 1;
            const Vec* vec = vecs + u;
            // row factors of both heads: Z <- f_i Z now, y = u_i Y + D x later
            float fz[2] = {0.f, 0.f}, fu[2] = {1.f, 1.f};
            if (ok) ok = tc::mbar_wait(&bars[kBarXFull + u], v & 1, abort_flag);
            if (ok) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const float grow = vec->G[hh][i];
                    const float gs = vec->misc[kMiscGs + hh];
                    const float gref = q == 0 ? gs : vec->G[hh][32 * q - 1];
                    const bool mild = gref - grow <= kMildSpan;
                    fz[hh] = mild ? exp2f(gref - gs) : exp2f(grow - gs);
                    fu[hh] = mild ? exp2f(grow - gref) : 1.f;
                }
            }
            if (ok) ok = tc::mbar_wait(&bars[kBarZDone], k & 1, abort_flag);
            tc::tc_fence_after();
            if (ok) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
                    for (int m = 0; m < kH / 32; ++m) {
                        uint32_t za[2][16];
                        const uint32_t ta = tmem + kColZ + hh * kH + lane_base + 32 * m;
                        tc::tmem_ld16_nowait(ta, za[0]);
                        tc::tmem_ld16_nowait(ta + 16, za[1]);
                        tc::tmem_wait_ld16(za[0]);
                        tc::tmem_tie16(za[1]);
#pragma unroll
                        for (int t = 0; t < 2; ++t)
#pragma unroll
                            for (int x = 0; x < 16; ++x) za[t][x] = __float_as_uint(fz[hh] * __uint_as_float(za[t][x]));
                        tc::tmem_st16(ta, za[0]);
                        tc::tmem_st16(ta + 16, za[1]);
                    }
                }
                tc::tmem_wait_st();
            }
            tc::tc_fence_before();
            __syncwarp();
            if (ok && lane == 0) tc::mbar_arrive(&bars[kBarZScaled]);
            // ---- y = u_i Y + D x, written over x in the stage
            if (ok) ok = tc::mbar_wait(&bars[kBarY2Done], k & 1, abort_flag);
            if (ok) ok = tc::mbar_wait(&bars[kBarXRead + u], v & 1, abort_flag);  // y goes over X
            tc::tc_fence_after();
            uint8_t* sX = smem + kOffX + u * 2 * kBox;
            if (ok) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const float dh = vec->misc[kMiscD + hh];
                    const float2 d2 = make_float2(dh, dh), u2 = make_float2(fu[hh], fu[hh]);
                    uint8_t* xrow = sX + hh * kBox + i * 128;
#pragma unroll
                    for (int m = 0; m < kH / 32; ++m) {
                        // 32 columns of Y and the four 16-byte x chunks under one wait
                        uint32_t ya[4][8];
                        uint4* px[4];
                        uint4 xv[4];
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const int kk = 32 * m + 8 * t;
                            tc::tmem_ld8_nowait(tmem + kColZ + hh * kH + lane_base + kk, ya[t]);
                            px[t] = reinterpret_cast<uint4*>(xrow + (((kk >> 3) ^ (i & 7)) << 4));
                        }
#pragma unroll
                        for (int t = 0; t < 4; ++t) xv[t] = *px[t];
                        tc::tmem_wait_ld8(ya[0]);
                        tc::tmem_tie8(ya[1]);
                        tc::tmem_tie8(ya[2]);
                        tc::tmem_tie8(ya[3]);
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            const uint32_t xw[4] = {xv[t].x, xv[t].y, xv[t].z, xv[t].w};
                            uint32_t yw[4];
#pragma unroll
                            for (int x = 0; x < 4; ++x) {
                                const float2 a2 = tc::fma_f32x2(
                                    d2, make_float2(tc::bf16_lo(xw[x]), tc::bf16_hi(xw[x])),
                                    tc::mul_f32x2(u2, make_float2(__uint_as_float(ya[t][2 * x]),
                                                                  __uint_as_float(ya[t][2 * x + 1]))));
                                yw[x] = tc::pack_bf16x2(a2.x, a2.y);
                            }
                            *px[t] = make_uint4(yw[0], yw[1], yw[2], yw[3]);
                        }
                    }
                }
            }
            // Y has been read: Z of the next block may be written.  y is in
            // shared memory for the X producer's TMA store.
            tc::tc_fence_before();
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (ok && lane == 0) {
                tc::mbar_arrive(&bars[kBarEpiDone]);
                tc::mbar_arrive(&bars[kBarYReady + u]);
            }
        }
        if (!ok) set_abort(ctl, p.status);
    } else {
        // ==================== scan, then fold (warps 16-19) ====================
        const int q = warp & 3;
        const int s = 32 * q + lane;       // scan: state row = TMEM lane
        const int t = (warp - kWarpScan0) * 32 + lane;  // fold: token row of the block
        const uint32_t lane_base = static_cast<uint32_t>(32 * q) << 16;
        // h <- initial state (or zeros)
#pragma unroll 1
        for (int hh = 0; hh < 2; ++hh) {
            const float* src = p.init ? p.init + ((b * g.nheads + h0 + hh) * kS + s) * kH : nullptr;
#pragma unroll 1
            for (int m = 0; m < kH / 16; ++m) {
                uint32_t r[16];
#pragma unroll
                for (int e = 0; e < 16; e += 4) {
                    const float4 f = src ? *reinterpret_cast<const float4*>(src + 16 * m + e) : make_float4(0.f, 0.f, 0.f, 0.f);
                    r[e] = __float_as_uint(f.x);
                    r[e + 1] = __float_as_uint(f.y);
                    r[e + 2] = __float_as_uint(f.z);
                    r[e + 3] = __float_as_uint(f.w);
                }
                tc::tmem_st16(tmem + kColH + hh * kH + lane_base + 16 * m, r);
            }
        }
        tc::tmem_wait_st();
        bool ok = true;
        for (int k = 0; k < nblk; ++k) {
            const int u = k & 1, v = k >> 1;
            // ---- scan: h -> bf16 tile (rows = states), then h <- exp2(G_l - G_s) h
            if (ok && k >= 1) ok = tc::mbar_wait(&bars[kBarUDone], (k - 1) & 1, abort_flag);
            if (ok) ok = tc::mbar_wait(&bars[kBarXFull + u], v & 1, abort_flag);
            if (!ok) break;
            tc::tc_fence_after();
            const Vec* vec = vecs + u;
#pragma unroll 1
            for (int hh = 0; hh < 2; ++hh) {
                const float alpha = exp2f(vec->G[hh][kBlk - 1] - vec->misc[kMiscGs + hh]);
                uint8_t* row = smem + kOffHW + hh * kBox + s * 128;
#pragma unroll
                for (int m = 0; m < kH / 16; ++m) {
                    uint32_t hv[16];
                    tc::tmem_ld16(tmem + kColH + hh * kH + lane_base + 16 * m, hv);
#pragma unroll
                    for (int c2 = 0; c2 < 2; ++c2) {
                        const int e = 8 * c2, c = 2 * m + c2;  // 16-byte chunk of the row
                        *reinterpret_cast<uint4*>(row + ((c ^ (s & 7)) << 4)) = make_uint4(
                            tc::pack_bf16x2(__uint_as_float(hv[e]), __uint_as_float(hv[e + 1])),
                            tc::pack_bf16x2(__uint_as_float(hv[e + 2]), __uint_as_float(hv[e + 3])),
                            tc::pack_bf16x2(__uint_as_float(hv[e + 4]), __uint_as_float(hv[e + 5])),
                            tc::pack_bf16x2(__uint_as_float(hv[e + 6]), __uint_as_float(hv[e + 7])));
                    }
#pragma unroll
                    for (int e = 0; e < 16; ++e) hv[e] = __float_as_uint(alpha * __uint_as_float(hv[e]));
                    tc::tmem_st16(tmem + kColH + hh * kH + lane_base + 16 * m, hv);
                }
            }
            tc::tmem_wait_st();
            tc::fence_proxy_async_smem();
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[kBarHReady]);
            // ---- fold: once Z has read the h tile, w . X into the same buffer
            ok = tc::mbar_wait(&bars[kBarZDone], k & 1, abort_flag);
            if (!ok) break;
            const uint8_t* sX = smem + kOffX + u * 2 * kBox;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const float w = vec->dt[hh][t] * exp2f(vec->G[hh][kBlk - 1] - vec->G[hh][t]);
                const uint8_t* src = sX + hh * kBox + t * 128;
                uint8_t* dst = smem + kOffHW + hh * kBox + t * 128;
#pragma unroll
                for (int c0 = 0; c0 < 8; c0 += 4) {
                    uint4 a[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) a[c] = *reinterpret_cast<const uint4*>(src + (((c0 + c + t) & 7) << 4));
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint4 r = a[c];
                        r.x = tc::pack_bf16x2(tc::bf16_lo(r.x) * w, tc::bf16_hi(r.x) * w);
                        r.y = tc::pack_bf16x2(tc::bf16_lo(r.y) * w, tc::bf16_hi(r.y) * w);
                        r.z = tc::pack_bf16x2(tc::bf16_lo(r.z) * w, tc::bf16_hi(r.z) * w);
                        r.w = tc::pack_bf16x2(tc::bf16_lo(r.w) * w, tc::bf16_hi(r.w) * w);
                        *reinterpret_cast<uint4*>(dst + (((c0 + c + t) & 7) << 4)) = r;
                    }
                }
            }
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tc::mbar_arrive(&bars[kBarWxReady]);
                tc::mbar_arrive(&bars[kBarXRead + u]);
            }
        }
        // the last state update has landed: write the final state
        if (ok && nblk > 0) ok = tc::mbar_wait(&bars[kBarUDone], (nblk - 1) & 1, abort_flag);
        if (ok && p.final_state) {
            tc::tc_fence_after();
#pragma unroll 1
            for (int hh = 0; hh < 2; ++hh) {
                float* dst = p.final_state + ((b * g.nheads + h0 + hh) * kS + s) * kH;
#pragma unroll 1
                for (int m = 0; m < kH / 16; ++m) {
                    uint32_t hv[16];
                    tc::tmem_ld16(tmem + kColH + hh * kH + lane_base + 16 * m, hv);
#pragma unroll
                    for (int e = 0; e < 16; e += 4)
                        *reinterpret_cast<float4*>(dst + 16 * m + e) =
                            make_float4(__uint_as_float(hv[e]), __uint_as_float(hv[e + 1]),
                                        __uint_as_float(hv[e + 2]), __uint_as_float(hv[e + 3]));
                }
            }
        }
        if (!ok) set_abort(ctl, p.status);
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

}  // namespace

// Shapes the fused kernel covers: bf16, head dim 64, state 128, chunks of 128
// or 256 tokens, heads in pairs of one group.
bool ssd_fused_fits(const Geom& g) {
    if (g.headdim != kH || g.dstate != kS) return false;
    if (g.chunk != 128 && g.chunk != 256) return false;
    if (g.nheads % 2 != 0 || g.heads_per_group % 2 != 0) return false;
    if (g.nheads / 2 > 65535 || g.batch > 65535) return false;
    if (g.batch * g.seqlen >= (int64_t(1) << 31)) return false;
    return g.seqlen >= 1 && g.batch >= 1;
}

cudaError_t launch_ssd_fused(const Geom& g, const FusedArgs& a, cudaStream_t st) {
    if (!ssd_fused_fits(g)) return cudaErrorInvalidConfiguration;
    FusedParams p{};
    p.g = g;
    p.dt = a.dt;
    p.G = a.G;
    p.D = a.D;
    p.init = a.init;
    p.final_state = a.final_state;
    p.status = device_status_word();
    const uint64_t H = g.headdim, S = g.dstate, nh = g.nheads, L = g.seqlen, G = g.ngroups;
    CUtensorMap tm_x, tm_b, tm_c, tm_y;
    {
        const uint64_t dims[4] = {H, nh, L, (uint64_t)g.batch};
        const uint64_t strides[3] = {H * 2, nh * H * 2, L * nh * H * 2};
        const uint32_t box[4] = {64, 1, kBlk, 1};
        if (!make_tmap_bf16(&tm_x, a.x, 4, dims, strides, box)) return cudaErrorInvalidValue;
        if (!make_tmap_bf16(&tm_y, a.y, 4, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[4] = {S, G, L, (uint64_t)g.batch};
        const uint64_t strides[3] = {S * 2, G * S * 2, L * G * S * 2};
        const uint32_t box[4] = {64, 1, kBlk, 1};
        if (!make_tmap_bf16(&tm_b, a.B, 4, dims, strides, box)) return cudaErrorInvalidValue;
        if (!make_tmap_bf16(&tm_c, a.C, 4, dims, strides, box)) return cudaErrorInvalidValue;
    }
    cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(k_ssd_fused_tc), (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(g.nheads / 2), (unsigned)g.batch);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_ssd_fused_tc, tm_x, tm_b, tm_c, tm_y, p);
}

}  // namespace m2
