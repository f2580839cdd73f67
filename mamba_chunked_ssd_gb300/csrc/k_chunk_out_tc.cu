// k_chunk_out_tc.cu — stage 3 on the 5th-generation tensor cores (bf16).
//
// "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in NVIDIA
// CUDA Tile", §Kernel 3, computes per chunk and head
//     Y = exp2(G) (C h_c) + ((C B^T) . exp2(G_i - G_j) . dt_j . causal M) X + D X.
// GB300 design.  One CTA owns (batch, chunk, 128-row block I of the chunk,
// a block of heads sharing one B/C group); T = 128 has one row block, T = 256
// two.  Rows of block I see columns j < 128 (I + 1); the interaction matrix
// is split along j into the block on the diagonal (j in block I) and, for
// I = 1, the block below it (j in block 0).
//   warp 0       producer: TMA of C and B once, then per head X (rows of
//                blocks 0 .. I) and h_c into a ring of stages; its 32 lanes
//                gather the head's G, dt and D into the same stage with
//                cp.async, so the epilogue never waits on a global load;
//                before refilling a stage it stores (TMA) the y that the
//                epilogue wrote over the stage's X, so no epilogue warp waits
//                on a store;
//   warp 1       TMEM allocator; one thread issues the C B^T products and
//                the tcgen05.mma of head stream 0;
//   warps 2..17  epilogue, split into head streams (two when H = 64, one when
//                H = 128) that take alternate heads, each stream with its own
//                TMEM accumulators so one stream's arithmetic overlaps the
//                other's tensor-core work;
//   warp 18      one thread issues the tcgen05.mma of head stream 1 (idle with
//                one stream).
// Once per CTA (per group, shared by every head):
//   CB_II = C_I B_I^T -> TMEM, causally masked in place;  for I = 1 also
//   CB_10 = C_1 B_0^T, converted to bf16 into shared memory as an MMA operand.
// Per head, with a = exp2(G_ref) and v_j = exp2(G_ref - G_j) dt_j for I = 1,
// G_ref = G_127 for heads that decay by more than 2^-64 over the first 128
// tokens and 0 otherwise (a = 1 and no second term for I = 0):
//   Z  = C_I (a h_c) + CB_10 (v . X_0)     tcgen05; a h_c (a != 1) and v . X_0
//                                          are scaled in place in the stage
//   P  = CB_II . w_j                       epilogue, written to TMEM as bf16 and
//                                          consumed there as operand A
//   Y2 = P X_I                             tcgen05, A from TMEM
//   y_i = exp2(G_i - G_ref) Z + u_i Y2 + D x_i  (G_ref = 0 for I = 0)
// with the decay of each row split at r, the last column before the row's
// 32-row quadrant:  exp2(G_i - G_j) dt_j = u_i w_j,  u_i = exp2(G_i - G_r),
// w_j = exp2(G_r - G_j) dt_j.  Both splits are exact identities; a_t <= 0
// keeps G non-increasing inside a chunk, so u_i <= 1 and w_j <= dt_j left of
// the quadrant.  A row whose u_i would fall below 2^-96 (a very strong decay
// inside its quadrant) takes exp2(G_i - G_j) per entry and u_i = 1.  Every
// row's arithmetic depends only on its own and earlier tokens.  Masked
// entries are zero in CB before any weight multiplies them.  The T x T matrix
// never reaches global memory.
// Chunks of 64 tokens run in pairs: a CTA's 128 rows are chunks 2c' and
// 2c' + 1, each with its own cumsum and its own state.  The state term takes
// both states in one product over K = 2S,
//   Z = [C_top | C_bot] [h_2c' ; h_2c'+1],
// where C_top is C with the rows of the second chunk zeroed and C_bot with
// those of the first (both built once per CTA; CB = C_top B^T + C_bot B^T),
// and P is block-diagonal: rows of the second chunk see no column of the
// first, and their quadrant 2 takes the chunk start as its reference.
// Every wait is bounded; a timeout sets the status word and the CTA unwinds.
#include <stdlib.h>
#include <string.h>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "tmap_host.cuh"

namespace m2 {
namespace {

constexpr int kEpiWarps = 16;
constexpr int kIssuer2 = 2 + kEpiWarps;  // warp 18: MMA issuer of head stream 1 (two streams)
constexpr int kStoreWarp = kIssuer2 + 1;  // warp 19: TMA stores of y (deep rings)
constexpr int kThreads = (kStoreWarp + 1) * 32;
// Chunks of one row block (T = 128, and chunk pairs) with at least this many
// stages send y out through a warp of its own as soon as it is written, and
// the producer refills a stage once that store has read it.  Otherwise the
// producer stores y itself, just before it refills the stage.  Measured on
// GB300: the store warp makes stage 3 4-8 % faster for 128-token chunks
// (state 64 or 128, 4-5 stages) and 1.5-2 % slower for 256-token chunks,
// even when only their first row block uses it.
constexpr int kStoreWarpMinStages = 4;
constexpr int kSmemLimit = 232448;
constexpr int kMaxStages = 5;
constexpr int kMaxStreams = 2;
// Fill barriers of the stages.  Head k fills stage k % nst and is read by
// stream k % nstr; its fill is signalled on barrier k % nfill with
// nfill = lcm(nst, nstr), so that each barrier's fills all go to one stage and
// one stream and every waiter sees each phase of it in order (a waiter that
// skipped a phase would take the next-but-one phase parity for its own).
constexpr int kMaxFill = 10;  // lcm(5, 2)
// Arrivals that complete a fill: the producer's expect-tx, then one per lane
// when that lane's cp.async gathers have landed.
constexpr int kFillArrivals = 1 + 32;

// TMEM columns (512 allocated): CB_II fp32 at [0, 128); P of stream s (bf16,
// 64 columns) at 128 + 64 s; Z and Y2 of stream s (fp32, H columns each) at
// 256 + 2 H s.  CB_10 is staged at [256, 384) before any stream uses it.
constexpr uint32_t kColCB = 0;
__host__ __device__ constexpr uint32_t col_p(int s) { return 128u + 64u * (uint32_t)s; }
__host__ __device__ constexpr uint32_t col_z(int s, int H) { return 256u + 2u * (uint32_t)H * (uint32_t)s; }

// Shared-memory layout of a CTA of row block I: C_I (for chunk pairs C_top
// and C_bot), (I = 1) CB_10, then the stages; a stage holds
// X [128 (I + 1) rows x H] | h_c [S x H] (two states for chunk pairs) |
// G[T] dt[T] D.  Block 0 needs neither X_1 nor CB_10, so it fits more stages.
struct CoLayout {
    int nst;    // pipeline stages
    int nfill;  // stage-fill barriers, lcm(nst, nstr)
    // B (read only by the C B^T products) overlays the first `rot` stage
    // slots; ring stage i lives in slot (i + rot) % nst, so the first
    // nst - rot heads fill slots B never touches, without waiting for C B^T
    // (rot = 0: every fill waits for C B^T)
    int rot;
    uint32_t off_stage, stage_bytes, off_h_in_stage, off_vec_in_stage, off_small, off_bar, smem_bytes;
};

struct CoTcParams {
    Geom g;           // geometry of the row blocks: chunk 128 or 256 (64-token chunks in pairs)
    int T;            // tokens a CTA's rows span (128 or 256)
    int64_t h_chunks; // chunk states per (batch, head): the caller's chunk count
    int nhb;          // heads per CTA (all in one group)
    int nstr;         // epilogue head streams (2 for H = 64, 1 for H = 128)
    int head_blocks;  // nheads / nhb
    int persistent;   // one CTA per SM takes an equal share of the work (one row block per chunk)
    uint32_t off_C, off_CB10, smem_bytes;
    CoLayout lay[2];  // by row block I
    const float* dt;
    const float* G;
    const float* D;
    unsigned int* status;
};

enum : int {
    kBarCbFull = 0,
    kBarCbDone,
    kBarCb10Ready,
    kBarOpsReady,                              // [kMaxStreams]
    kBarPReady = kBarOpsReady + kMaxStreams,   // [kMaxStreams]
    kBarYDone = kBarPReady + kMaxStreams,      // [kMaxStreams]
    kBarYFree = kBarYDone + kMaxStreams,       // [kMaxStreams]
    kBarFull = kBarYFree + kMaxStreams,        // [kMaxFill]
    kBarStored = kBarFull + kMaxFill,          // [kMaxStages] y's store has read the stage (store warp)
    kBarYReady = kBarStored + kMaxStages,      // [kMaxStages] y is written over the stage's X
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

// Largest exponent (log2 units) either factor of the split decay may carry:
// P entries then stay below 2^96 |CB| dt, far from the bf16 / fp32 range.
constexpr float kMildSpan = 96.f;
// Upper clamp of a column weight: keeps 0 x weight = 0 for the masked entries
// whatever dt is (a NaN weight is kept: the comparison is false for NaN).
constexpr float kWMax = 0x1p120f;

// exp2(G_i - G_j) dt_j for the direct path, exponent clamped at kMildSpan so
// that masked entries (j > i) multiply a finite weight.
__device__ __forceinline__ float exact_weight(float gi, float gj, float dtj) {
    const float w = exp2f(fminf(gi - gj, kMildSpan)) * dtj;
    return w > kWMax ? kWMax : w;
}

// Scales, in place, four consecutive 16-byte bf16 chunks [c_begin, c_begin + 4)
// of one 128-byte-swizzled row by f, rounded once to bf16 per element (bf16x2
// multiplies by f rounded to bf16).  c_begin is a multiple of 4, so the four
// chunks lie in one box of 64 columns; boxes sit box_stride bytes apart.  The
// chunks are visited in physical order, rotated by the row to spread banks.
__device__ __forceinline__ void scale_row4(uint8_t* base, uint32_t box_stride, int row, int c_begin, float f) {
    const uint32_t f2 = tc::pack_bf16x2(f, f);
    uint8_t* rowp = base + (c_begin >> 3) * box_stride + row * 128;
    const int c0 = (c_begin & 7) + row;
    uint4 v[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) v[t] = *reinterpret_cast<const uint4*>(rowp + (((c0 + t) & 7) << 4));
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        v[t].x = tc::mul_bf16x2(v[t].x, f2);
        v[t].y = tc::mul_bf16x2(v[t].y, f2);
        v[t].z = tc::mul_bf16x2(v[t].z, f2);
        v[t].w = tc::mul_bf16x2(v[t].w, f2);
    }
#pragma unroll
    for (int t = 0; t < 4; ++t) *reinterpret_cast<uint4*>(rowp + (((c0 + t) & 7) << 4)) = v[t];
}

// H (the head width one MMA covers) and T (chunk) are compile-time, so the
// stream / part / box counts and most swizzle offsets fold into constants.
// VS = 2 splits every head of width 2 H into two virtual heads of width H that
// share the head's decays (its P is formed once per virtual head): the stages
// then hold half of the head's X and h_c, which lets a head of 128 columns
// with a 256-wide state and a 256-token chunk fit, and gives such heads two
// streams.  VS = 1: virtual and real heads coincide.  PAIR: the 128 rows are
// two chunks of 64 tokens (T = 128).
template <int H, int T, int VS, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
k_chunk_out_tc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
               const __grid_constant__ CUtensorMap tm_c, const __grid_constant__ CUtensorMap tm_h,
               const __grid_constant__ CUtensorMap tm_y, const CoTcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const Geom& g = p.g;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    // Work items.  Without persistence each CTA takes the one item its
    // blockIdx names: x index hb + head_blocks (I + (T / 128) c) (the chunk
    // index rides in x, whose range covers every chunk count the library
    // accepts) and the batch row, nhb heads from head hb * nhb.  With it (one
    // row block per chunk, so every item has the same shared-memory layout)
    // one CTA per SM takes an equal share of the (batch, chunk, virtual head)
    // triples, in that order, and runs it as items of consecutive heads that
    // share one chunk and one group: so C, B and their product are formed
    // once per chunk and group rather than once per 16 heads, and the CTAs'
    // shares differ by one head at most.  Every item starts with fresh
    // barriers and ends with the CTA quiescent, so items are independent, and
    // the CTA keeps its tensor memory and skips the turnover between CTAs.
    // (The counts fit in 32 bits: the host caps b nh nc S below 2^31.)
    const int gx = p.head_blocks * (T / 128) * (int)g.nchunks;
    const int vh_all = (int)g.nheads * VS;           // virtual heads per chunk
    const int vh_grp = (int)g.heads_per_group * VS;  // virtual heads per group
    // persistent: this CTA's triples [f, f_end); else its one item f
    int f, f_end;
    if (p.persistent) {
        const int64_t n_units = g.batch * g.nchunks * vh_all;
        f = (int)(n_units * blockIdx.x / gridDim.x);
        f_end = (int)(n_units * (blockIdx.x + 1) / gridDim.x);
    } else {
        f = (int)blockIdx.x + gx * (int)blockIdx.y;
        f_end = f + 1;
    }
    bool tmem_held = false;
    uint32_t tmem = 0;
    while (f < f_end) {
    int64_t b, c;
    int I, vh0, nvh;
    if (p.persistent) {
        const int bc = f / vh_all;
        const int vh = f % vh_all;
        nvh = min(f_end - f, (vh / vh_grp + 1) * vh_grp - vh);
        vh0 = vh;
        b = bc / (int)g.nchunks;
        c = bc % (int)g.nchunks;
        I = 0;
        f += nvh;
    } else {
        const int xi = f % gx;
        const int hb = xi % p.head_blocks;
        const int rest = xi / p.head_blocks;
        I = rest % (T / 128);  // row block inside the chunk
        c = rest / (T / 128);
        b = f / gx;
        vh0 = hb * p.nhb * VS;
        nvh = p.nhb * VS;
        f = f_end;
    }
    const int64_t t0 = c * T;
    const int tc = (int)imin64(T, g.seqlen - t0);  // valid tokens of the chunk
    if (128 * I >= tc) continue;                         // ragged tail: no valid row here
    const int grp = (int)(vh0 / VS / g.heads_per_group);
    const int Tj = 128 * (I + 1);  // columns j that rows of block I can see
    const int S = (int)g.dstate;
    constexpr int nstr = (H == 64) ? 2 : 1;
    const int wps = kEpiWarps / nstr;  // warps per stream

    static_assert(!PAIR || T == 128, "chunk pairs span 128 rows");
    uint8_t* sC = smem + p.off_C;
    uint8_t* sC1 = sC + 128 * S * 2;  // C_bot (chunk pairs)
    uint8_t* sCB10 = smem + p.off_CB10;
    const CoLayout lay = I ? p.lay[1] : p.lay[0];
    uint8_t* sStage = smem + lay.off_stage;
    uint8_t* sB = sCB10;  // B overlays CB_10 and the first stage slots until the CB products are done
    // shared-memory slot of ring stage i
    auto slot_of = [&](int i) { return i + lay.rot >= lay.nst ? i + lay.rot - lay.nst : i + lay.rot; };
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.off_bar);
    SharedCtl* ctl = reinterpret_cast<SharedCtl*>(smem + lay.off_bar + kNumBars * 8);

    if (threadIdx.x == 0) {
        tc::mbar_init(&bars[kBarCbFull], 1);
        tc::mbar_init(&bars[kBarCbDone], 1);
        tc::mbar_init(&bars[kBarCb10Ready], kEpiWarps);
        for (int i = 0; i < kMaxStreams; ++i) {
            tc::mbar_init(&bars[kBarOpsReady + i], wps);
            tc::mbar_init(&bars[kBarPReady + i], wps);
            tc::mbar_init(&bars[kBarYDone + i], 1);
            tc::mbar_init(&bars[kBarYFree + i], wps);
        }
        for (int i = 0; i < kMaxFill; ++i) tc::mbar_init(&bars[kBarFull + i], kFillArrivals);
        // a stage is refilled once the y the epilogue wrote over X_I in it has
        // been stored (the epilogue read Z and Y2 first, so the MMAs are done
        // with the stage too)
        for (int i = 0; i < kMaxStages; ++i) {
            tc::mbar_init(&bars[kBarStored + i], 1);
            tc::mbar_init(&bars[kBarYReady + i], wps);
        }
        if (!tmem_held) ctl->abort = 0;
        tc::fence_barrier_init();
    }
    if (PAIR && !tmem_held) {
        // zero rows 64..127 of C_top and rows 0..63 of C_bot (the TMA fills
        // the other halves); the MMAs read them through the async proxy
        const int nbox = S / 64;
        for (int u = threadIdx.x; u < nbox * 512; u += kThreads) {
            const int kb = u >> 9, r = u & 511;  // 512 x 16 bytes per half box
            *reinterpret_cast<uint4*>(sC + kb * 16384 + 8192 + r * 16) = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(sC1 + kb * 16384 + r * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        tc::fence_proxy_async_smem();
    }
    if (warp == 1 && !tmem_held) {
        tc::tmem_alloc(&ctl->tmem_base, 512);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (!tmem_held) tmem = ctl->tmem_base;
    tmem_held = true;
    volatile int* abort_flag = &ctl->abort;
    const uint32_t x_bytes = (uint32_t)Tj * H * 2;
    const uint32_t h_bytes = (uint32_t)S * H * 2;
    const bool store_warp = T == 128 && lay.nst >= kStoreWarpMinStages;
    // y of virtual head k leaves ring stage st through TMA stores; rows past
    // the sequence end are clipped
    auto issue_y_store = [&](int k, int st) {
        const uint8_t* sY = sStage + slot_of(st) * lay.stage_bytes;
        for (int cb = 0; cb < H / 64; ++cb)
            tc::tma_store_4d(&tm_y, sY + cb * (Tj * 128) + I * 16384, ((vh0 + k) % VS) * H + cb * 64, (vh0 + k) / VS,
                             (int)(t0 + 128 * I), (int)b);
        tc::bulk_commit();
    };

    if (warp == 0) {
        // ============== TMA producer + per-head G / dt / D gather ==============
        if (lane == 0) {
            tc::tma_prefetch_desc(&tm_x);
            tc::tma_prefetch_desc(&tm_b);
            tc::tma_prefetch_desc(&tm_c);
            tc::tma_prefetch_desc(&tm_h);
            tc::mbar_arrive_expect_tx(&bars[kBarCbFull], (uint32_t)(128 * S * 2 + Tj * S * 2));
            for (int kb = 0; kb < S / 64; ++kb) {
                if (PAIR) {
                    // 64-row boxes: rows of chunk 2c' into C_top, of 2c' + 1 into C_bot
                    tc::tma_load_4d(sC + kb * 16384, &tm_c, &bars[kBarCbFull], kb * 64, grp, (int)t0, (int)b);
                    tc::tma_load_4d(sC1 + kb * 16384 + 8192, &tm_c, &bars[kBarCbFull], kb * 64, grp,
                                    (int)(t0 + 64), (int)b);
                } else {
                    tc::tma_load_4d(sC + kb * 16384, &tm_c, &bars[kBarCbFull], kb * 64, grp, (int)(t0 + 128 * I),
                                    (int)b);
                }
                for (int rb = 0; rb < Tj / 128; ++rb)
                    tc::tma_load_4d(sB + kb * (Tj * 128) + rb * 16384, &tm_b, &bars[kBarCbFull], kb * 64, grp,
                                    (int)(t0 + 128 * rb), (int)b);
            }
        }
        // h_c and G come from the previous kernels
        tc::griddep_wait();
        bool ok = true;
        bool b_free = false;  // the slots under B may be filled (C B^T done)
        // stage, its reuse phase and the fill barrier as counters (no divisions)
        int st = 0, fill = 0;
        uint32_t slot_phase = 1;  // phase of the previous use of the stage
        // without the store warp: y of head kp (ring stage st_kp, its use of
        // phase ph) is stored here, just before the stage is refilled
        auto store_y = [&](int kp, int st_kp, uint32_t ph) -> bool {
            if (!tc::mbar_wait(&bars[kBarYReady + st_kp], ph, abort_flag)) return false;
            issue_y_store(kp, st_kp);
            return true;
        };
        for (int k = 0; ok && k < nvh; ++k) {
            if (k >= lay.nst) {
                bool w_ok = true;
                if (lane == 0) {
                    if (store_warp) {
                        w_ok = tc::mbar_wait(&bars[kBarStored + st], slot_phase, abort_flag);
                    } else {
                        w_ok = store_y(k - lay.nst, st, slot_phase);
                        tc::bulk_wait_read_all();  // the stage may be overwritten
                    }
                }
                if (!__shfl_sync(0xffffffffu, (int)w_ok, 0)) {
                    ok = false;
                    break;
                }
            }
            if (!b_free && (lay.rot == 0 || slot_of(st) < lay.rot)) {
                // this slot lies under B: wait until the C B^T products have read it
                if (lane == 0) ok = tc::mbar_wait(&bars[kBarCbDone], 0, abort_flag);
                if (!__shfl_sync(0xffffffffu, (int)ok, 0)) {
                    ok = false;
                    break;
                }
                b_free = true;
            }
            uint8_t* sX = sStage + slot_of(st) * lay.stage_bytes;
            uint8_t* sH = sX + lay.off_h_in_stage;
            float* vG = reinterpret_cast<float*>(sX + lay.off_vec_in_stage);  // G[T], dt[T], D
            float* vDt = vG + T;
            uint64_t* full = &bars[kBarFull + fill];
            const int h = (vh0 + k) / VS;          // real head
            const int col0 = ((vh0 + k) % VS) * H;  // its first column in this virtual head
            if (lane == 0) {
                tc::mbar_arrive_expect_tx(full, x_bytes + (PAIR ? 2 : 1) * h_bytes);
                // state rows of the chunk (of both chunks of a pair; past the
                // last chunk the pair's second state repeats the first, whose
                // rows then multiply zeros of C_bot or fall past the end)
                const int64_t hrow = (b * g.nheads + h) * p.h_chunks + (PAIR ? 2 * c : c);
                const int64_t hrow1 = (PAIR && 2 * c + 1 < p.h_chunks) ? hrow + 1 : hrow;
                for (int cb = 0; cb < H / 64; ++cb) {
                    for (int rb = 0; rb < Tj / 128; ++rb)
                        tc::tma_load_4d(sX + cb * (Tj * 128) + rb * 16384, &tm_x, full, col0 + cb * 64, h,
                                        (int)(t0 + 128 * rb), (int)b);
                    tc::tma_load_2d(sH + cb * (S * 128), &tm_h, full, col0 + cb * 64, (int)(hrow * S));
                    if (PAIR)
                        tc::tma_load_2d(sH + h_bytes + cb * (S * 128), &tm_h, full, col0 + cb * 64,
                                        (int)(hrow1 * S));
                }
            }
            // G_j (past the last valid token: G of the last one) and dt_j (zero there)
            const float* Gh = p.G + (b * g.nheads + h) * g.seqlen + t0;
            const float* dth = p.dt + (b * g.seqlen + t0) * g.nheads + h;
            for (int j = lane; j < Tj; j += 32) {
                const int jv = j < tc ? j : tc - 1;
                tc::cp_async4(vG + j, Gh + jv, 4);
                tc::cp_async4(vDt + j, dth + (int64_t)jv * g.nheads, j < tc ? 4u : 0u);
            }
            if (lane == 0) tc::cp_async4(vDt + T, p.D ? p.D + h : p.dt, p.D ? 4u : 0u);
            tc::cp_async_mbar_arrive_noinc(full);
            if (++st == lay.nst) {
                st = 0;
                slot_phase ^= 1u;
            }
            if (++fill == lay.nfill) fill = 0;
        }
        // the y of the last heads still sits in the stages
        if (lane == 0 && !store_warp) {
            for (int kp = nvh > lay.nst ? nvh - lay.nst : 0; ok && kp < nvh; ++kp)
                ok = store_y(kp, kp % lay.nst, (uint32_t)(kp / lay.nst) & 1u);
            tc::bulk_wait_all();
        }
        if (!ok && lane == 0) set_abort(ctl, p.status);
    } else if (warp == kStoreWarp) {
        // ============ y stores (TMA) in head order, for deep rings ============
        // y of head k leaves as soon as the epilogue has written it; once the
        // store has read the stage, the producer may refill it.
        if (lane == 0 && store_warp) {
            bool ok = true;
            int st = 0;
            uint32_t ph = 0;
            for (int k = 0; k < nvh; ++k) {
                if (!tc::mbar_wait(&bars[kBarYReady + st], ph, abort_flag)) {
                    ok = false;
                    break;
                }
                issue_y_store(k, st);
                tc::bulk_wait_read_all();  // this warp only stores, so it waits here
                tc::mbar_arrive(&bars[kBarStored + st]);
                if (++st == lay.nst) {
                    st = 0;
                    ph ^= 1u;
                }
            }
            tc::bulk_wait_all();
            if (!ok) set_abort(ctl, p.status);
        }
    } else if (warp == 1 || (nstr == 2 && warp == kIssuer2)) {
        // ========================= MMA issuers (one per stream) =========================
        // Warp 1 issues the C B^T products and the per-head products of stream
        // 0, warp 18 those of stream 1, so neither stream waits behind the other.
        if (lane == 0) {
            const int sid0 = (warp == 1) ? 0 : 1;
            bool ok = tc::mbar_wait(&bars[kBarCbFull], 0, abort_flag);
            const uint32_t aC = tc::smem_u32(sC), aB = tc::smem_u32(sB);
            if (ok && sid0 == 1) {
                // stream 1 reads C_I (and for I = 1 the bf16 CB_10) from shared memory
                if (I == 1) ok = tc::mbar_wait(&bars[kBarCb10Ready], 0, abort_flag);
            } else if (ok) {
                tc::tc_fence_after();
                // CB_II = C_I B_I^T (both K-major over S); for I = 1 also CB_10 = C_1 B_0^T.
                const uint32_t id_cb = tc::idesc_bf16(128, 128, false, false);
                for (int k16 = 0; k16 < S / 16; ++k16) {
                    const uint64_t da = tc::sdesc_sw128(aC + (k16 >> 2) * 16384 + (k16 & 3) * 32, 16, 1024);
                    const uint32_t bbase = aB + (k16 >> 2) * (Tj * 128) + (k16 & 3) * 32;
                    tc::mma_bf16_ss(tmem + kColCB, da, tc::sdesc_sw128(bbase + I * 16384, 16, 1024), id_cb, k16 > 0);
                    if (I == 1) tc::mma_bf16_ss(tmem + 256, da, tc::sdesc_sw128(bbase, 16, 1024), id_cb, k16 > 0);
                }
                if (PAIR) {
                    // CB = C_top B^T + C_bot B^T
                    const uint32_t aC1 = tc::smem_u32(sC1);
                    for (int k16 = 0; k16 < S / 16; ++k16) {
                        const uint64_t da = tc::sdesc_sw128(aC1 + (k16 >> 2) * 16384 + (k16 & 3) * 32, 16, 1024);
                        const uint32_t bbase = aB + (k16 >> 2) * (Tj * 128) + (k16 & 3) * 32;
                        tc::mma_bf16_ss(tmem + kColCB, da, tc::sdesc_sw128(bbase, 16, 1024), id_cb, 1);
                    }
                }
                tc::mma_commit(&bars[kBarCbDone]);
                if (I == 1) ok = tc::mbar_wait(&bars[kBarCb10Ready], 0, abort_flag);
            }
            const uint32_t id_y = tc::idesc_bf16(128, H, false, true);
            // Each issuing thread paces its stream, so its loop is kept short: stage and fill-barrier indices and phases are counters, and
            // every descriptor is a base built once plus a constant offset in
            // its 14-bit address field (16-byte units; shared memory is below
            // 256 KB, so the field cannot carry).  K-major A tiles (C_I, CB_10)
            // advance 32 bytes per 16 columns inside a 64-column box and 16 KB
            // per box; MN-major B tiles (h_c, X) advance 2 KB per 16 rows.
            const uint64_t dC0 = tc::sdesc_sw128(aC, 16, 1024);
            const uint64_t dC1 = tc::sdesc_sw128(tc::smem_u32(sC1), 16, 1024);  // C_bot (chunk pairs)
            const uint64_t dCB10 = tc::sdesc_sw128(tc::smem_u32(sCB10), 16, 1024);
            const uint64_t dH0 = tc::sdesc_sw128(tc::smem_u32(sStage + lay.off_h_in_stage), S * 128, 1024);
            const uint64_t dX0 = tc::sdesc_sw128(tc::smem_u32(sStage), Tj * 128, 1024);
            const uint64_t stage_step = lay.stage_bytes >> 4;
            int st = sid0 % lay.nst, fill = sid0 % lay.nfill;
            int pst = slot_of(st);  // its shared-memory slot
            uint32_t fill_phase = (sid0 / lay.nfill) & 1;
            uint64_t dstage = pst * stage_step;  // slot offset, in descriptor units
            for (int k = sid0; ok && k < nvh; k += nstr) {
                const int s = k % nstr, n = k / nstr;
                const uint32_t tz = tmem + col_z(s, H), ty2 = tz + H;
                if (!tc::mbar_wait(&bars[kBarFull + fill], fill_phase, abort_flag)) { ok = false; break; }
                if (n >= 1 && !tc::mbar_wait(&bars[kBarYFree + s], (n - 1) & 1, abort_flag)) { ok = false; break; }
                if (I == 1 && !tc::mbar_wait(&bars[kBarOpsReady + s], n & 1, abort_flag)) { ok = false; break; }
                tc::tc_fence_after();
                const uint64_t dH = dH0 + dstage, dX = dX0 + dstage;
                // Z = C_I (a h_c)   (B operand: rows s = K, columns H = N, MN-major)
                for (int k16 = 0; k16 < S / 16; ++k16)
                    tc::mma_bf16_ss(tz, dC0 + (k16 >> 2) * 1024 + (k16 & 3) * 2, dH + 128 * k16, id_y, k16 > 0);
                if (PAIR) {
                    // Z += C_bot h_2c'+1   (the second state follows the first in the stage)
                    const uint64_t dH1 = dH + (h_bytes >> 4);
                    for (int k16 = 0; k16 < S / 16; ++k16)
                        tc::mma_bf16_ss(tz, dC1 + (k16 >> 2) * 1024 + (k16 & 3) * 2, dH1 + 128 * k16, id_y, 1);
                }
                if (I == 1) {
                    // Z += CB_10 (v . X_0)   (A: CB_10 bf16, K-major over j; B: rows 0..127 of
                    // the stage's X, scaled in place, MN-major)
#pragma unroll
                    for (int k16 = 0; k16 < 8; ++k16)
                        tc::mma_bf16_ss(tz, dCB10 + (k16 >> 2) * 1024 + (k16 & 3) * 2, dX + 128 * k16, id_y, 1);
                }
                // Y2 = P X_I   (A: P in TMEM; B: rows 128I.. of X, MN-major)
                if (!tc::mbar_wait(&bars[kBarPReady + s], n & 1, abort_flag)) { ok = false; break; }
                tc::tc_fence_after();
#pragma unroll
                for (int k16 = 0; k16 < 8; ++k16)
                    tc::mma_bf16_ts(ty2, tmem + col_p(s) + k16 * 8, dX + I * 1024 + 128 * k16, id_y, k16 > 0);
                tc::mma_commit(&bars[kBarYDone + s]);
#pragma unroll
                for (int i = 0; i < nstr; ++i) {
                    if (++st == lay.nst) st = 0;
                    if (++pst == lay.nst) {
                        pst = 0;
                        dstage = 0;
                    } else {
                        dstage += stage_step;
                    }
                    if (++fill == lay.nfill) {
                        fill = 0;
                        fill_phase ^= 1u;
                    }
                }
            }
            if (!ok) set_abort(ctl, p.status);
        }
    } else if (warp < kIssuer2) {
        // ============================== epilogue ==============================
        const int e = warp - 2;                 // 0..15
        const int sid = e / wps;                // head stream of this warp
        const int q = warp & 3;                 // TMEM lane quadrant this warp may access
        const int nparts = wps / 4;             // warps per quadrant within a stream
        const int part = (e % wps) >> 2;        // column part handled by this warp
        const int gpw = 4 / nparts;             // 32-column groups of P per warp
        const int ncoly = H / nparts;           // output columns per thread (32)
        // the folds give each thread 8 (H/64) / nparts = 4 chunks of 16 bytes per row
        const int il = q * 32 + lane;           // row inside the block = TMEM lane
        const int i = 128 * I + il;             // row inside the chunk
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        const uint32_t tz = tmem + col_z(sid, H), ty2 = tz + H, tp = tmem + col_p(sid);
        float* wv = reinterpret_cast<float*>(smem + lay.off_small) + e * 64;  // per warp: w of 2 column groups
        // the column before this quadrant (-1: before the chunk; quadrant 2
        // of a chunk pair starts the pair's second chunk)
        const int rq = (PAIR && q == 2) ? -1 : 128 * I + 32 * q - 1;
        // 32-column groups of the diagonal block this quadrant's rows see
        // (a chunk pair's second chunk sees none of the first's)
        auto visible = [&](int gi) { return gi <= q && !(PAIR && q >= 2 && gi < 2); };

        bool ok = tc::mbar_wait(&bars[kBarCbDone], 0, abort_flag);
        tc::tc_fence_after();
        if (ok && I == 1) {
            // CB_10 (staged in TMEM) -> bf16 [128 rows i x 128 columns j], K-major, 128B swizzle
            const int cg = e >> 2;  // 32-column group 0..3
            uint8_t* row = sCB10 + (cg >> 1) * 16384 + il * 128;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                uint32_t r[16];
                tc::tmem_ld16(tmem + 256 + lane_base + 32 * cg + 16 * hh, r);
                const int c0 = (cg & 1) * 4 + 2 * hh;
#pragma unroll
                for (int s4 = 0; s4 < 2; ++s4) {
                    const int x = 8 * s4;
                    *reinterpret_cast<uint4*>(row + (((c0 + s4) ^ (il & 7)) << 4)) = make_uint4(
                        tc::pack_bf16x2(__uint_as_float(r[x]), __uint_as_float(r[x + 1])),
                        tc::pack_bf16x2(__uint_as_float(r[x + 2]), __uint_as_float(r[x + 3])),
                        tc::pack_bf16x2(__uint_as_float(r[x + 4]), __uint_as_float(r[x + 5])),
                        tc::pack_bf16x2(__uint_as_float(r[x + 6]), __uint_as_float(r[x + 7])));
                }
            }
            tc::fence_proxy_async_smem();
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[kBarCb10Ready]);
        }
        if (ok && e < 4) {
            // Causal mask, once for every head: zero CB_II above the diagonal
            // inside this quadrant's diagonal 32 x 32 group (the groups right
            // of it are never read).
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
        // Every epilogue warp sees the masked CB before it forms P.
        tc::tc_fence_before();
        asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
        tc::tc_fence_after();

        // stage and fill barrier of head k as counters, advanced by nstr heads
        int st = sid % lay.nst, fill = sid % lay.nfill;
        uint32_t fill_phase = (sid / lay.nfill) & 1;
        for (int k = sid; ok && k < nvh; k += nstr) {
            const int n = k / nstr;
            if (ok) ok = tc::mbar_wait(&bars[kBarFull + fill], fill_phase, abort_flag);
            uint8_t* sX = sStage + slot_of(st) * lay.stage_bytes;
          if (ok) {
            const float* vG = reinterpret_cast<const float*>(sX + lay.off_vec_in_stage);
            const float* vDt = vG + T;
            const float grow = vG[i];
            const float gref = rq < 0 ? 0.f : vG[rq];

            // Decays of this quadrant's rows split at r = rq (see the file
            // comment).  mild: u_i >= 2^-kMildSpan, so w_j <= dt_j / u_i stays
            // in range for every column the row uses.  The test reads only G_r
            // and G_i, so a row's path never depends on later tokens; the
            // warp-wide fast loop gives mild rows the same products as the
            // mixed loop.
            const bool mild = gref - grow <= kMildSpan;  // false for NaN
            const bool all_mild = __all_sync(0xffffffffu, mild);
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                if (t >= gpw) break;
                const int gi = part * gpw + t;
                if (!visible(gi)) continue;
                const int j = 128 * I + 32 * gi + lane;
                const float wj = exp2f(fminf(gref - vG[j], kMildSpan)) * vDt[j];
                wv[32 * t + lane] = wj > kWMax ? kWMax : wj;
            }
            __syncwarp();

            // Row block 1 takes the carried state and the first 128 tokens in one
            // product, relative to a reference G_ref: Z = C_1 (exp2(G_ref) h_c) +
            // CB_10 (v . X_0), v_j = exp2(G_ref - G_j) dt_j, and the rows' factor
            // is exp2(G_i - G_ref).  G_ref = G_127 keeps every factor <= 1 but
            // rescales h_c in place; when G_127 >= -64, G_ref = 0 leaves h_c as
            // it is (v stays below 2^64 dt, far inside the bf16 range).
            const float g127 = I == 1 ? vG[127] : 0.f;
            const bool scale_h = I == 1 && !(g127 >= -64.f);  // NaN: the safe branch
            const float gref_z = scale_h ? g127 : 0.f;
            if (I == 1) {
                // (exp2(G_ref) h_c and) v . X_0, in place in the stage
                if (scale_h) {
                    uint8_t* sH = sX + lay.off_h_in_stage;
                    const float a = exp2f(g127);
                    for (int r = il; r < S; r += 128) scale_row4(sH, S * 128, r, part * 4, a);
                }
                const float vj = exp2f(gref_z - vG[il]) * vDt[il];
                scale_row4(sX, Tj * 128, il, part * 4, vj);
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&bars[kBarOpsReady + sid]);
            }

            // ---- P on the diagonal block -> TMEM as bf16 (CB is masked already),
            // one 32-column group at a time: both 16-column halves are loaded
            // under one wait
#pragma unroll
            for (int t = 0; t < 2; ++t) {
                if (t >= gpw) break;
                const int gi = part * gpw + t;  // 32-column group 0..3 of the diagonal block
                if (!visible(gi)) {
                    uint32_t z[8];
#pragma unroll
                    for (int x = 0; x < 8; ++x) z[x] = 0u;
                    tc::tmem_st8(tp + lane_base + 16 * gi, z);
                    tc::tmem_st8(tp + lane_base + 16 * gi + 8, z);
                    continue;
                }
                uint32_t r[2][16];
                tc::tmem_ld16_nowait(tmem + kColCB + lane_base + 32 * gi, r[0]);
                tc::tmem_ld16_nowait(tmem + kColCB + lane_base + 32 * gi + 16, r[1]);
                tc::tmem_wait_ld16(r[0]);
                tc::tmem_tie16(r[1]);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const uint32_t col = 32 * gi + 16 * hh;  // first column of this piece
                    const float* w = wv + 32 * t + 16 * hh;
                    const float* gj = vG + 128 * I + col;
                    const float* dj = vDt + 128 * I + col;
                    const uint32_t* rr = r[hh];
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
                    tc::tmem_st8(tp + lane_base + col / 2, pk);
                }
            }
            tc::tmem_wait_st();
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[kBarPReady + sid]);

            // ---- y = exp2(G_i - G_ref) Z + u_i Y2 + D x_i   (G_ref above; 0 for I = 0),
            // written over x_i in the stage (each thread rewrites exactly the
            // 16-byte pieces it reads; Y2, the last reader of X_I, is done)
            const float si = exp2f(grow - gref_z);
            const float ui = mild ? exp2f(grow - gref) : 1.f;
            const float dh = vDt[T];
            const float2 si2 = make_float2(si, si), ui2 = make_float2(ui, ui), d2 = make_float2(dh, dh);
            uint8_t* xrow = sX + i * 128;
            ok = tc::mbar_wait(&bars[kBarYDone + sid], n & 1, abort_flag);
            tc::tc_fence_after();
            if (ok) {
                // two 8-column slices of Z and Y2 (and their x chunks) per wait
#pragma unroll
                for (int mp = 0; mp < 2; ++mp) {
                    if (mp >= ncoly / 16) break;
                    uint32_t za[2][8], yb[2][8];
                    uint4* px[2];
                    uint4 xv[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int kk = part * ncoly + 16 * mp + 8 * u;
                        tc::tmem_ld8_nowait(tz + lane_base + kk, za[u]);
                        tc::tmem_ld8_nowait(ty2 + lane_base + kk, yb[u]);
                        px[u] = reinterpret_cast<uint4*>(xrow + (kk >> 6) * (Tj * 128) +
                                                         ((((kk & 63) >> 3) ^ (i & 7)) << 4));
                    }
                    xv[0] = *px[0];
                    xv[1] = *px[1];
                    tc::tmem_wait_ld8(za[0]);
                    tc::tmem_tie8(yb[0]);
                    tc::tmem_tie8(za[1]);
                    tc::tmem_tie8(yb[1]);
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        // y = si Z + ui Y2 + D x, in fp32, rounded once to bf16
                        const uint32_t xw[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
                        uint32_t yw[4];
#pragma unroll
                        for (int x = 0; x < 4; ++x) {
                            const float2 t2 = tc::fma_f32x2(
                                d2, make_float2(tc::bf16_lo(xw[x]), tc::bf16_hi(xw[x])),
                                tc::mul_f32x2(ui2, make_float2(__uint_as_float(yb[u][2 * x]), __uint_as_float(yb[u][2 * x + 1]))));
                            const float2 a2 = tc::fma_f32x2(
                                si2, make_float2(__uint_as_float(za[u][2 * x]), __uint_as_float(za[u][2 * x + 1])), t2);
                            yw[x] = tc::pack_bf16x2(a2.x, a2.y);
                        }
                        *px[u] = make_uint4(yw[0], yw[1], yw[2], yw[3]);
                    }
                }
            }
          }
            // Z and Y2 have been read (the stream's accumulators may be
            // rewritten), and y is in the stage for the producer's TMA store
            tc::tc_fence_before();
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (ok && lane == 0) {
                tc::mbar_arrive(&bars[kBarYFree + sid]);
                tc::mbar_arrive(&bars[kBarYReady + st]);
            }
#pragma unroll
            for (int i = 0; i < nstr; ++i) {
                if (++st == lay.nst) st = 0;
                if (++fill == lay.nfill) {
                    fill = 0;
                    fill_phase ^= 1u;
                }
            }
        }
        if (!ok) set_abort(ctl, p.status);
    }

    tc::tc_fence_before();
    __syncthreads();
    // the item's barriers have completed their last phases: retire them
    if (threadIdx.x == 0)
        for (int i = 0; i < kNumBars; ++i) tc::mbar_inval(&bars[i]);
    if (*abort_flag) break;  // read after the barrier: the same for every thread
    }
    if (tmem_held && warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

// Real heads per CTA: the largest divisor of the heads per group with at most
// 16 virtual heads.
int pick_heads_per_cta(const Geom& g, int vs) {
    const int r = (int)g.heads_per_group;
    for (int n = 16 / vs; n >= 1; --n)
        if (r % n == 0) return n;
    return 1;
}

int lcm_small(int a, int b) {
    int m = a;
    while (m % b != 0) m += a;
    return m;
}

// Chunks of 64 tokens run as pairs spanning 128 rows.
bool is_pair(const Geom& g) { return g.chunk == 64; }
int row_blocks(const Geom& g) { return is_pair(g) ? 1 : (int)(g.chunk / 128); }

bool plan_layout(const Geom& g, int I, int vs, int nstr, uint32_t off_CB10, CoLayout& L) {
    const int T = 128 * row_blocks(g), S = (int)g.dstate, H = (int)g.headdim / vs, Tj = 128 * (I + 1);
    const int nh_tiles = is_pair(g) ? 2 : 1;  // states per stage
    L.off_stage = off_CB10 + (I == 1 ? 32768u : 0u);
    L.off_h_in_stage = (uint32_t)(Tj * H * 2);
    L.off_vec_in_stage = L.off_h_in_stage + (uint32_t)(nh_tiles * S * H * 2);
    const uint32_t vec_bytes = (uint32_t)(2 * T + 4) * 4;
    L.stage_bytes = (L.off_vec_in_stage + vec_bytes + 1023) / 1024 * 1024;  // swizzled tiles: 1024-aligned
    for (int nst = kMaxStages; nst >= 1; --nst) {
        // B (for the CB products) overlays CB_10, the stages and, if it is
        // longer, the per-warp area: all are written only after CB is done.
        const uint32_t stages_end = L.off_stage + nst * L.stage_bytes;
        const uint32_t b_end = off_CB10 + (uint32_t)(Tj * S * 2);
        const uint32_t off_small = stages_end > b_end ? stages_end : b_end;
        const uint32_t off_bar = off_small + kEpiWarps * 64 * 4;
        const uint32_t total = off_bar + kNumBars * 8 + 64 + 1024;  // + ctl + alignment slack
        if (total <= (uint32_t)kSmemLimit) {
            L.nst = nst;
            L.nfill = lcm_small(nst, nstr);
            // stage slots that B overlaps
            const int64_t over = (int64_t)b_end - (int64_t)L.off_stage;
            L.rot = over <= 0 ? 0 : (int)((over + L.stage_bytes - 1) / L.stage_bytes);
            if (L.rot >= nst) L.rot = 0;  // B covers every slot
            L.off_small = off_small;
            L.off_bar = off_bar;
            L.smem_bytes = total;
            return L.nfill <= kMaxFill;
        }
    }
    return false;
}

// Shared-memory plan for virtual-head split vs (1, or 2 for 128-wide heads).
bool plan_smem(const Geom& g, int vs, CoTcParams& p) {
    if (vs != 1 && !(vs == 2 && g.headdim == 128)) return false;
    p.nstr = (g.headdim / vs == 64) ? 2 : 1;
    p.off_C = 0;
    p.off_CB10 = p.off_C + (is_pair(g) ? 2u : 1u) * 128 * (uint32_t)g.dstate * 2;
    p.smem_bytes = 0;
    for (int I = 0; I < row_blocks(g); ++I) {
        if (!plan_layout(g, I, vs, p.nstr, p.off_CB10, p.lay[I])) return false;
        if (p.lay[I].smem_bytes > p.smem_bytes) p.smem_bytes = p.lay[I].smem_bytes;
    }
    if (row_blocks(g) == 1) p.lay[1] = p.lay[0];  // unused
    return true;
}

// The virtual-head split used for a shape (0: none fits).  Heads of 128
// columns are split in two when the state is 128 or wider, and stay whole
// with state 64; whichever fits is taken when the preferred one does not.
// Measured on GB300 (stage-3 time, whole vs split, µs, every sweep length
// within 1 %): state 64: 424 vs 523 (chunk 128), 539 vs 611 (chunk 256);
// state 128: 571 vs 555 (128), 837 vs 677 (256); state 256: 974 vs 714
// (128), split only (256, 1297).
// MAMBA2_CHUNK_OUT_HEAD_SPLIT=1 or =2 forces that variant, for timing both on
// one shape; where the forced variant does not fit, stage 3 runs on the
// CUDA-core kernel.
int pick_vs(const Geom& g) {
    CoTcParams p;
    const char* env = getenv("MAMBA2_CHUNK_OUT_HEAD_SPLIT");
    if (env && (env[0] == '1' || env[0] == '2') && env[1] == 0) {
        const int want = env[0] - '0';
        return plan_smem(g, want, p) ? want : 0;
    }
    const bool split = plan_smem(g, 2, p);
    const bool whole = plan_smem(g, 1, p);
    if (g.dstate >= 128 && split) return 2;
    if (whole) return 1;
    return split ? 2 : 0;
}

// The geometry of the CTAs' row blocks: a pair of 64-token chunks is one
// block of 128 rows.
Geom block_geom(const Geom& g) {
    Geom gb = g;
    if (is_pair(g)) {
        gb.chunk = 128;
        gb.nchunks = (g.seqlen + 127) / 128;
    }
    return gb;
}

}  // namespace

// Shapes the tensor-core stage-3 kernel covers; others use the CUDA-core kernel.
bool chunk_out_tc_fits(const Geom& g) {
    if (g.chunk != 64 && g.chunk != 128 && g.chunk != 256) return false;
    if (g.headdim != 64 && g.headdim != 128) return false;
    if (g.dstate != 64 && g.dstate != 128 && g.dstate != 256) return false;
    if (g.batch * g.nheads * g.nchunks * g.dstate >= (int64_t(1) << 31)) return false;
    if (g.batch * g.seqlen >= (int64_t(1) << 31)) return false;
    // grid.x = head blocks x row blocks x row-block chunks (at most nheads * 2 * nchunks)
    const Geom gb = block_geom(g);
    if (g.nheads * row_blocks(g) * gb.nchunks >= (int64_t(1) << 31)) return false;
    return pick_vs(g) != 0;
}

cudaError_t launch_chunk_out_tc(const Geom& g, const ChunkOutArgs& a, cudaStream_t st) {
    CoTcParams p{};
    p.g = block_geom(g);
    p.T = 128 * row_blocks(g);
    p.h_chunks = g.nchunks;
    const int vs = pick_vs(g);
    if (vs == 0 || !plan_smem(g, vs, p)) return cudaErrorInvalidConfiguration;
    p.nhb = pick_heads_per_cta(g, vs);
    p.head_blocks = (int)(g.nheads / p.nhb);
    p.dt = a.dt;
    p.G = a.G;
    p.D = a.D;
    p.status = device_status_word();
    const uint64_t H = g.headdim, S = g.dstate, nh = g.nheads, L = g.seqlen, G = g.ngroups;
    CUtensorMap tm_x, tm_b, tm_c, tm_h, tm_y;
    {
        const uint64_t dims[4] = {H, nh, L, (uint64_t)g.batch};
        const uint64_t strides[3] = {H * 2, nh * H * 2, L * nh * H * 2};
        const uint32_t box[4] = {64, 1, 128, 1};
        if (!make_tmap_bf16(&tm_x, a.x, 4, dims, strides, box)) return cudaErrorInvalidValue;
        if (!make_tmap_bf16(&tm_y, a.y, 4, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[4] = {S, G, L, (uint64_t)g.batch};
        const uint64_t strides[3] = {S * 2, G * S * 2, L * G * S * 2};
        const uint32_t box[4] = {64, 1, 128, 1};
        const uint32_t box_c[4] = {64, 1, is_pair(g) ? 64u : 128u, 1};  // C of a pair: one chunk per box
        if (!make_tmap_bf16(&tm_b, a.B, 4, dims, strides, box)) return cudaErrorInvalidValue;
        if (!make_tmap_bf16(&tm_c, a.C, 4, dims, strides, box_c)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t rows = (uint64_t)g.batch * nh * g.nchunks * S;
        const uint64_t dims[2] = {H, rows};
        const uint64_t strides[1] = {H * 2};
        const uint32_t box[2] = {64, (uint32_t)S};
        if (!make_tmap_bf16(&tm_h, a.chunk_states, 2, dims, strides, box)) return cudaErrorInvalidValue;
    }
    auto kern = is_pair(g)
                    ? (g.headdim == 64 ? k_chunk_out_tc<64, 128, 1, true>
                                       : (vs == 2 ? k_chunk_out_tc<64, 128, 2, true> : k_chunk_out_tc<128, 128, 1, true>))
                : (g.headdim == 64)
                    ? (p.T == 256 ? k_chunk_out_tc<64, 256, 1, false> : k_chunk_out_tc<64, 128, 1, false>)
                    : (vs == 2 ? (p.T == 256 ? k_chunk_out_tc<64, 256, 2, false> : k_chunk_out_tc<64, 128, 2, false>)
                               : (p.T == 256 ? k_chunk_out_tc<128, 256, 1, false> : k_chunk_out_tc<128, 128, 1, false>));
    cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(kern), (int)p.smem_bytes);
    if (e != cudaSuccess) return e;
    // One row block per chunk: one CTA per SM takes an equal share (unless
    // MAMBA2_CHUNK_OUT_PERSISTENT=0); else one CTA per item.
    const int64_t gx = (int64_t)p.head_blocks * (p.T / 128) * p.g.nchunks, n_items = gx * g.batch;
    const char* pe = getenv("MAMBA2_CHUNK_OUT_PERSISTENT");
    p.persistent = (row_blocks(g) == 1 && !(pe && strcmp(pe, "0") == 0)) ? 1 : 0;
    const int nsm = sm_count();
    if (p.persistent && nsm <= 0) return cudaErrorInvalidValue;
    dim3 grid = p.persistent ? dim3((unsigned)(n_items < nsm ? n_items : nsm))
                             : dim3((unsigned)gx, (unsigned)g.batch);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = p.smem_bytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = a.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, tm_x, tm_b, tm_c, tm_h, tm_y, p);
}

}  // namespace m2
