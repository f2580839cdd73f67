// k_state_pass_tc.cu — stage 2 on the 5th-generation tensor cores (bf16).
//
// [blog §Kernel 2]: for c = 0 .. nc-1 store h_c, then
//     h_{c+1} = exp2(G_last) h_c + (w . B_c)^T X_c,   w_t = dt_t exp2(G_last - G_t).
// GB300 design.  One CTA owns (batch, head, 128-row tile of the S x H state)
// and walks the chunks in order:
//   warp 0      producer: TMA of 64- or 128-token sub-blocks of B (the tile's 128
//               state columns) and of X into a ring of shared-memory stages;
//               its lanes also gather the sub-block's G_t and dt_t and the
//               chunk's G_last into the stage with cp.async, so the other
//               warps never wait on a global load;
//   warp 1      TMEM allocator and single-thread tcgen05.mma issuer:
//               U_c = B_c^T (w . X_c) accumulated over the chunk's sub-blocks
//               into one of two TMEM buffers (A = B_c^T and B = w . X_c are
//               both read "MN-major" straight from the TMA layout);
//   warps 2..9  form w_t = dt_t exp2(G_last - G_t) and fold it into the X rows
//               in shared memory (so the weighted operand is formed once, on
//               chip), and run the scan:
//               the state h lives in TMEM next to U; per chunk each thread
//               (one state row, half of the columns) stores h_c, then sets
//               h <- exp2(G_last) h + U_c.
// Heads of 64 columns may run in pairs (HP below): a pair's x rows are
// adjacent, so the two heads load as one 128-column head and share B's tile
// and one product per sub-block.
// The weighted-operand fold applies the blog's "pre-multiplied operand" to X
// instead of B (same product; X is the smaller per-head tile).  States past
// dstate (when dstate = 64) are zero-filled by TMA and never stored.
//
// Sequence segments.  When there are too few (batch, head) pairs to fill the
// GPU, the forward pass splits each sequence into segments of whole chunks
// and runs this kernel twice around a short carry (k_state_carry below):
//   summary pass  every segment but the last walks its chunks from a zero
//                 state (segment 0 from the initial state) and writes only its
//                 end state;
//   carry         H_1 = end state of segment 0, and for k >= 1
//                 H_{k+1} = exp2(D_k) H_k + (end state of segment k),
//                 D_k being the sum of G_last over segment k's chunks: the
//                 state entering each segment, by the jump formula;
//   segment pass  every segment walks its chunks from its entering state,
//                 storing the chunk states; the last one writes final_state.
// The chunk states are those of one pass over the whole sequence; only the
// order of the fp32 sums at segment boundaries differs.
#include <stdlib.h>

#include "common.cuh"
#include "tc_ptx.cuh"
#include "tmap_host.cuh"

namespace m2 {
namespace {

constexpr int kFoldWarps = 4;  // warps 2..5
constexpr int kScanWarps = 4;  // warps 6..9, one per TMEM lane quadrant
constexpr int kThreads = (2 + kFoldWarps + kScanWarps) * 32;
// Tokens per sub-block (KB): 64, or 128 where one CTA runs per SM and the
// chunk has at least 128 tokens.  Measured on GB300 (state pass alone):
// 128-token sub-blocks are 11-14 % faster with one CTA per SM (4 stages of
// 128 against 8 of 64), 9 % slower with two CTAs per SM (2 stages against 4);
// 32-token sub-blocks were 25-70 % slower than 64 (the per-sub-block
// hand-offs cost more than a deeper ring gains).
constexpr int kMaxStages = 8;
constexpr int kSmemLimit = 232448;

// What a launch computes (sequence segments: see above).
enum SpMode : int { kWholeSequence = 0, kSegmentSummary = 1, kSegmentPass = 2 };

struct SpTcParams {
    Geom g;
    int mode;           // SpMode
    int nseg;           // segments of a sequence (1 for kWholeSequence)
    int cps;            // chunks per segment
    int seg_grid;       // segments this launch covers: nseg, or nseg - 1 for the summary
    float* seg_states;  // [b, nh, nseg - 1, S, H] fp32: segment end states, then entering states
    int kb;             // tokens per sub-block (64 or 128)
    int nsb;            // sub-blocks per chunk = chunk / kb
    int nst;            // ring stages
    int stg_tiles;      // 64-row staging tiles for the chunk-state stores (1 or 2)
    // stage: B [2 boxes] (split: B_hi, B_lo) | X [H / 64 boxes] (split: X_hi, X_lo) | G, dt, G_last
    uint32_t stage_bytes, off_blo_in_stage, off_x_in_stage, off_xlo_in_stage, off_w_in_stage, off_stg, off_bar,
        smem_bytes, tmem_cols;
    const float* dt;
    const float* G;
    const float* init;
    __nv_bfloat16* chunk_states;
    float* final_state;
    unsigned int* status;
};

enum : int {
    kBarUDone = 0,     // [2]
    kBarUFree = 2,     // [2]
    kBarFull = 4,      // [kMaxStages]
    kBarXform = 4 + kMaxStages,
    kBarSlotFree = 4 + 2 * kMaxStages,
    kNumBars = 4 + 3 * kMaxStages
};

struct SharedCtl {
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ void set_abort(SharedCtl* ctl, unsigned int* status) {
    ctl->abort = 1;
    if (status) atomicExch(status, kStatusTimeout);
}

// H (head dim), T (chunk) and KB (tokens per sub-block) are compile-time, so
// the sub-block count and the box and chunk offsets fold into constants.
// SPLIT: an fp32 problem.  x arrives as fp32 (boxes of 32 columns) and B as
// bf16 hi/lo planes ([b, L, 2 G, S], group 2g hi and 2g + 1 lo); the fold
// forms w x in fp32 and leaves it in place as a hi/lo pair (each 64-column
// group's two fp32 boxes become its hi box and its lo box), U takes three
// products (B_hi (w x)_hi + B_hi (w x)_lo + B_lo (w x)_hi), and the chunk
// states leave as fp32, rows [b, nh, nc, S] x H.
// HP: a pair of heads 2 h', 2 h' + 1 of 64 columns each, whose x rows are
// adjacent in memory, runs as one head of 128 columns (H = 128): one B tile
// and one 128 x 128 x KB product per sub-block serve both heads.  The fold
// takes each half's own weights, the scan each half's own decay, and the
// halves' states come from and go to their own heads' rows.
template <int H, int T, int KB, bool SPLIT, bool HP = false>
__global__ void __launch_bounds__(kThreads, 2)
k_state_pass_tc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_b,
                const __grid_constant__ CUtensorMap tm_cs, const SpTcParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const Geom& g = p.g;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int mt = blockIdx.x;              // 128-row tile of the state
    const int h = blockIdx.y;               // head (HP: head pair; x's view has nheads / 2 heads of 128)
    const int64_t b = blockIdx.z / (unsigned)p.seg_grid;
    const int seg = (int)(blockIdx.z % (unsigned)p.seg_grid);
    const int hr = HP ? 2 * h : h;          // the (first) real head
    const int64_t bh = b * g.nheads + hr;
    const int grp = (int)(hr / g.heads_per_group);
    static_assert(!HP || (H == 128 && !SPLIT), "head pairs: two bf16 heads of 64 columns");
    constexpr int HH = HP ? 64 : H;         // columns of a real head
    constexpr int NV = HP ? 2 : 1;          // real heads of this CTA
    const int S = (int)g.dstate;
    constexpr int kKb = KB;
    static_assert(KB == 64 || KB == 128, "sub-blocks of 64 or 128 tokens");
    static_assert(T % KB == 0, "whole sub-blocks per chunk");
    static_assert(!SPLIT || KB == 64, "split: two fold threads per token row");
    constexpr int nsb = T / kKb;              // sub-blocks per chunk
    // this CTA's chunks [c_begin, c_begin + nchl)
    const int c_begin = seg * p.cps;
    const int nchl = (int)imin64(p.cps, g.nchunks - c_begin);
    const int nsub = nchl * nsb;  // sub-blocks of those chunks

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.off_bar);
    SharedCtl* ctl = reinterpret_cast<SharedCtl*>(smem + p.off_bar + kNumBars * 8);

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&bars[kBarUDone + i], 1);
            tc::mbar_init(&bars[kBarUFree + i], kScanWarps);
        }
        for (int i = 0; i < kMaxStages; ++i) {
            tc::mbar_init(&bars[kBarFull + i], 1 + 32);  // expect-tx + one cp.async arrival per lane
            tc::mbar_init(&bars[kBarXform + i], kFoldWarps);
            tc::mbar_init(&bars[kBarSlotFree + i], 1);
        }
        ctl->abort = 0;
        tc::fence_barrier_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(&ctl->tmem_base, p.tmem_cols);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    const uint32_t tm_u0 = tmem;           // U buffers: [0, H), [H, 2H)
    const uint32_t tm_h = tmem + 2 * H;    // running state, two buffers: [2H, 3H), [3H, 4H)
    volatile int* abort_flag = &ctl->abort;
    const uint32_t x_box_bytes = kKb * 128;

    tc::griddep_launch_dependents();  // stage 3 may start; it waits for this grid
    if (warp == 0) {
        // ===================== TMA producer + weight gather =====================
        if (lane == 0) {
            tc::tma_prefetch_desc(&tm_x);
            tc::tma_prefetch_desc(&tm_b);
        }
        tc::griddep_wait();  // G comes from the previous kernel
        const float* Gbh = p.G + bh * g.seqlen;
        bool ok = true;
        int st = 0;
        uint32_t slot_phase = 1;  // phase of the previous use of the stage (counters, no divisions)
        for (int u = 0; u < nsub; ++u, st = (st + 1 == p.nst) ? (slot_phase ^= 1u, 0) : st + 1) {
            if (u >= p.nst) {
                bool w_ok = true;
                if (lane == 0) w_ok = tc::mbar_wait(&bars[kBarSlotFree + st], slot_phase, abort_flag);
                if (!__shfl_sync(0xffffffffu, (int)w_ok, 0)) { ok = false; break; }
            }
            const int c = c_begin + u / nsb, sb = u % nsb;
            const int64_t t0 = (int64_t)c * T;
            const int tc = (int)imin64(T, g.seqlen - t0);
            const int tok = (int)(t0 + sb * kKb);
            uint8_t* sB = smem + st * p.stage_bytes;
            uint8_t* sX = sB + p.off_x_in_stage;
            float* sV = reinterpret_cast<float*>(sB + p.off_w_in_stage);  // G[kKb], dt[kKb], G_last
            if (lane == 0) {
                // split: B as two planes, x as fp32 (the same bytes as its hi/lo pair)
                constexpr int planes = SPLIT ? 2 : 1;
                tc::mbar_arrive_expect_tx(&bars[kBarFull + st], planes * (2 + H / 64) * x_box_bytes);
                for (int pl = 0; pl < planes; ++pl)
                    for (int kb = 0; kb < 2; ++kb)
                        tc::tma_load_4d(sB + pl * p.off_blo_in_stage + kb * x_box_bytes, &tm_b, &bars[kBarFull + st],
                                        mt * 128 + kb * 64, SPLIT ? 2 * grp + pl : grp, tok, (int)b);
                constexpr int xcols = SPLIT ? 32 : 64;  // columns per box
                for (int cb = 0; cb < H / xcols; ++cb)
                    tc::tma_load_4d(sX + cb * x_box_bytes, &tm_x, &bars[kBarFull + st], cb * xcols, h, tok, (int)b);
            }
            // G_t and dt_t of the sub-block's tokens (past the last valid token:
            // G of the last one and dt = 0) and G_last of the chunk, gathered
            // straight into the stage; each lane arrives on the stage barrier
            // once its copies have landed.
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                // head hr + v: its G row follows the previous head's
                float* sVv = sV + v * (2 * kKb + 1);
                const float* Gv = Gbh + v * g.seqlen;
#pragma unroll
                for (int r = 0; r < kKb / 32; ++r) {
                    const int tl = sb * kKb + lane + 32 * r;
                    const int tv = tl < tc ? tl : tc - 1;
                    tc::cp_async4(sVv + lane + 32 * r, Gv + t0 + tv, 4);
                    tc::cp_async4(sVv + kKb + lane + 32 * r, p.dt + (b * g.seqlen + t0 + tv) * g.nheads + hr + v,
                                  tl < tc ? 4u : 0u);
                }
                if (lane == 0) tc::cp_async4(sVv + 2 * kKb, Gv + t0 + tc - 1, 4);
            }
            tc::cp_async_mbar_arrive_noinc(&bars[kBarFull + st]);
        }
        if (!ok && lane == 0) set_abort(ctl, p.status);
    } else if (warp == 1) {
        // ============================ MMA issuer ============================
        if (lane == 0) {
            bool ok = true;
            // A = B_c^T (rows of the box are tokens = K, columns are states = M),
            // B = w . X_c (rows tokens = K, columns head dim = N): both MN-major.
            const uint32_t idesc = tc::idesc_bf16(128, H, true, true);
            // This one thread paces the kernel, so its loop is kept short: the
            // stage index and phase are counters, and the descriptors of a
            // stage are the first stage's advanced by whole stages (the 14-bit
            // address field, in 16-byte units, cannot carry: shared memory is
            // below 256 KB) and by 2 KB (128 units) per 16 tokens.
            const uint64_t desc0 = tc::sdesc_sw128(tc::smem_u32(smem), x_box_bytes, 1024);
            // split: w x's 64-column hi boxes are two boxes apart (its lo
            // boxes in between)
            const uint64_t xdesc0 = tc::sdesc_sw128(tc::smem_u32(smem), (SPLIT ? 2 : 1) * x_box_bytes, 1024);
            const uint64_t stage_step = p.stage_bytes >> 4, x_step = p.off_x_in_stage >> 4;
            const uint64_t blo_step = p.off_blo_in_stage >> 4, xlo_step = p.off_xlo_in_stage >> 4;
            uint64_t dstage = desc0, xstage = xdesc0;
            int st = 0;
            uint32_t phase = 0;
            for (int u = 0; u < nsub; ++u) {
                const int c = u / nsb, sb = u % nsb, ub = c & 1;
                if (sb == 0 && c >= 2 && !tc::mbar_wait(&bars[kBarUFree + ub], ((c >> 1) - 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                if (!tc::mbar_wait(&bars[kBarXform + st], phase, abort_flag)) {
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
                const uint32_t tu = tm_u0 + ub * H;
                if (SPLIT) {
                    // B_hi (w x)_hi + B_hi (w x)_lo + B_lo (w x)_hi
                    const uint64_t pa[3] = {0, 0, blo_step}, pb[3] = {x_step, xlo_step, x_step};
                    for (int ps = 0; ps < 3; ++ps)
#pragma unroll
                        for (int k16 = 0; k16 < kKb / 16; ++k16)
                            tc::mma_bf16_ss(tu, dstage + pa[ps] + 128 * k16, xstage + pb[ps] + 128 * k16, idesc,
                                            (sb > 0 || ps > 0 || k16 > 0) ? 1u : 0u);
                } else {
#pragma unroll
                    for (int k16 = 0; k16 < kKb / 16; ++k16)
                        tc::mma_bf16_ss(tu, dstage + 128 * k16, dstage + x_step + 128 * k16, idesc,
                                        (sb > 0 || k16 > 0) ? 1u : 0u);
                }
                tc::mma_commit(&bars[kBarSlotFree + st]);
                if (sb == nsb - 1) tc::mma_commit(&bars[kBarUDone + ub]);
                if (++st == p.nst) {
                    st = 0;
                    phase ^= 1u;
                    dstage = desc0;
                    xstage = xdesc0;
                } else {
                    dstage += stage_step;
                    xstage += stage_step;
                }
            }
            if (!ok) set_abort(ctl, p.status);
        }
    } else {
        bool ok = true;
        if (warp < 2 + kFoldWarps) {
            // ================= weight fold (warps 2..5) =================
            // 128 / kKb threads per token row of a sub-block, each taking an
            // equal share of the row's 16-byte chunks (rotated to spread banks).
            constexpr int tpr = 128 / kKb;
            const int ft = (warp - 2) * 32 + lane;  // 0..127
            const int frow = ft / tpr, fh = ft % tpr;
            const int per = 8 * (H / 64) / tpr;     // chunks per thread (2 to 8)
            int st = 0;
            uint32_t full_phase = 0;
            for (int u = 0; ok && u < nsub; ++u, st = (st + 1 == p.nst) ? (full_phase ^= 1u, 0) : st + 1) {
                if (!tc::mbar_wait(&bars[kBarFull + st], full_phase, abort_flag)) { ok = false; break; }
                const float* sV = reinterpret_cast<const float*>(smem + st * p.stage_bytes + p.off_w_in_stage);
                const float w = sV[kKb + frow] * exp2f(sV[2 * kKb] - sV[frow]);  // w_t = dt_t exp2(G_last - G_t)
                // HP: the second head's weight, for the row's second 64-column box
                const float w1 = HP ? sV[(2 * kKb + 1) + kKb + frow] *
                                          exp2f(sV[(2 * kKb + 1) + 2 * kKb] - sV[(2 * kKb + 1) + frow])
                                    : w;
                uint8_t* rowp = smem + st * p.stage_bytes + p.off_x_in_stage + frow * 128;
                if (SPLIT) {
                    // fp32 x -> w x as a hi/lo pair, one 64-column group at a
                    // time: this thread reads its 32-column box of the row,
                    // and after both threads of the row have read, writes its
                    // 32 columns into the group's hi box (the first of the two)
                    // and lo box (the second)
#pragma unroll 1
                    for (int cg = 0; cg < H / 64; ++cg) {
                        uint8_t* grow = rowp + 2 * cg * x_box_bytes;
                        float v[32];
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float4 f = *reinterpret_cast<const float4*>(grow + fh * x_box_bytes +
                                                                              ((j ^ (frow & 7)) << 4));
                            v[4 * j] = f.x * w;
                            v[4 * j + 1] = f.y * w;
                            v[4 * j + 2] = f.z * w;
                            v[4 * j + 3] = f.w * w;
                        }
                        __syncwarp();
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint32_t off = (((4 * fh + j) ^ (frow & 7)) << 4);
                            uint32_t oh[4], ol[4];
#pragma unroll
                            for (int x = 0; x < 4; ++x) {
                                const float a0 = v[8 * j + 2 * x], a1 = v[8 * j + 2 * x + 1];
                                oh[x] = tc::pack_bf16x2(a0, a1);
                                ol[x] = tc::pack_bf16x2(a0 - tc::bf16_lo(oh[x]), a1 - tc::bf16_hi(oh[x]));
                            }
                            *reinterpret_cast<uint4*>(grow + off) = make_uint4(oh[0], oh[1], oh[2], oh[3]);
                            *reinterpret_cast<uint4*>(grow + x_box_bytes + off) = make_uint4(ol[0], ol[1], ol[2], ol[3]);
                        }
                    }
                }
#pragma unroll
                for (int f0 = 0; f0 < 16; f0 += 2) {  // two chunks in flight
                    if (SPLIT) break;
                    if (f0 >= per) break;
                    uint4 v[2];
#pragma unroll
                    for (int f = 0; f < 2; ++f) {
                        const int flat = fh * per + f0 + f;  // 0 .. 8 (H/64) - 1
                        v[f] = *reinterpret_cast<const uint4*>(rowp + (flat >> 3) * x_box_bytes +
                                                               ((((flat & 7) + frow) & 7) << 4));
                    }
#pragma unroll
                    for (int f = 0; f < 2; ++f) {
                        const int flat = fh * per + f0 + f;
                        const float wf = (HP && (flat >> 3)) ? w1 : w;
                        uint4 a = v[f];
                        a.x = tc::pack_bf16x2(tc::bf16_lo(a.x) * wf, tc::bf16_hi(a.x) * wf);
                        a.y = tc::pack_bf16x2(tc::bf16_lo(a.y) * wf, tc::bf16_hi(a.y) * wf);
                        a.z = tc::pack_bf16x2(tc::bf16_lo(a.z) * wf, tc::bf16_hi(a.z) * wf);
                        a.w = tc::pack_bf16x2(tc::bf16_lo(a.w) * wf, tc::bf16_hi(a.w) * wf);
                        *reinterpret_cast<uint4*>(rowp + (flat >> 3) * x_box_bytes +
                                                  ((((flat & 7) + frow) & 7) << 4)) = a;
                    }
                }
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&bars[kBarXform + st]);
            }
        } else {
            // ============ scan (warps 6..9): one state row per thread ============
            const int q = warp & 3;  // TMEM lane quadrant
            const int s = mt * 128 + q * 32 + lane;
            const bool valid = s < S;
            const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
            const float* Gbh = p.G + bh * g.seqlen;
            // G_last of chunk c for real head hr + v
            auto glast_of = [&](int c, int v) -> float {
                const int64_t t0 = (int64_t)c * T;
                return Gbh[v * g.seqlen + t0 + imin64(T, g.seqlen - t0) - 1];
            };
            // h <- initial state (segment 0), the segment's entering state
            // (segment pass), or zeros; 32 columns (eight 16-byte loads) per
            // round.  The initial state is the caller's input, so its loads
            // start before the wait for the previous kernel; the entering
            // state of a later segment comes from the carry kernel.
            // (hstride: elements from one head's state to the next head's)
            auto load_h = [&](const float* h_in, int64_t hstride) {
#pragma unroll 1
                for (int m = 0; m < H / 32; ++m) {
                    // columns 32 m .. of the CTA's state: real head hr + (32 m) / HH
                    const float* src = h_in + ((32 * m) / HH) * hstride + s * HH + (32 * m) % HH;
                    float4 f[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        f[j] = (valid && h_in) ? *reinterpret_cast<const float4*>(src + 4 * j)
                                               : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {
                        uint32_t r[16];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            r[4 * j] = __float_as_uint(f[4 * hf + j].x);
                            r[4 * j + 1] = __float_as_uint(f[4 * hf + j].y);
                            r[4 * j + 2] = __float_as_uint(f[4 * hf + j].z);
                            r[4 * j + 3] = __float_as_uint(f[4 * hf + j].w);
                        }
                        tc::tmem_st16(tm_h + lane_base + 32 * m + 16 * hf, r);
                    }
                }
                tc::tmem_wait_st();
            };
            if (seg == 0) {
                load_h(p.init ? p.init + bh * S * HH : nullptr, (int64_t)S * HH);
                tc::griddep_wait();
            } else {
                tc::griddep_wait();
                load_h(p.mode == kSegmentPass ? p.seg_states + (bh * (p.nseg - 1) + seg - 1) * S * HH : nullptr,
                       (int64_t)(p.nseg - 1) * S * HH);
            }
            // Per chunk: h_{c+1} = exp2(G_last) h_c + U_c into the other h
            // buffer (then U_c's buffer is released to the MMA), then h_c is
            // stored; G_last of the next chunk is fetched while this one waits
            // for its U.  h_c leaves through 64-row shared-memory tiles
            // (128-byte swizzle; quadrants 0-1 fill the first half's, 2-3 the
            // second's) and TMA stores.
            uint8_t* stg = smem + p.off_stg;
            const int hrow = (q & 1) * 32 + lane;  // row inside the 64-row tile
            const bool leader = (q == 0 && lane == 0);
            const bool store = p.mode != kSegmentSummary;  // the summary keeps only the end state
            // 64-row halves of this CTA's state rows (one for dstate 64) and
            // the staging passes per chunk; a tile is 64 x H (bf16: boxes of
            // 64 columns; split, fp32: boxes of 32)
            const int nhalf = (S - mt * 128 >= 128) ? 2 : 1;
            const int npass = p.stg_tiles >= nhalf ? 1 : nhalf;
            constexpr uint32_t tile_bytes = (SPLIT ? H / 32 : H / 64) * 8192;
            float gl_next = glast_of(c_begin, 0), gl_next1 = HP ? glast_of(c_begin, 1) : 0.f;
            // Every scan warp runs every iteration and every named barrier below,
            // whatever its own waits return, so no warp is left at a barrier;
            // after a failed wait a warp only skips the work.
            for (int cl = 0; cl < nchl; ++cl) {
                const int c = c_begin + cl, ub = cl & 1;
                const float alpha = exp2f(gl_next), alpha1 = HP ? exp2f(gl_next1) : alpha;
                if (cl + 1 < nchl) {
                    gl_next = glast_of(c + 1, 0);
                    if (HP) gl_next1 = glast_of(c + 1, 1);
                }
                if (ok) ok = tc::mbar_wait(&bars[kBarUDone + ub], (cl >> 1) & 1, abort_flag);
                tc::tc_fence_after();
                const int64_t row0 = (bh * g.nchunks + c) * S + mt * 128;  // first state row of the tile
                // h_{c+1} = exp2(G_last) h_c + U_c into the other h buffer;
                // U_c's buffer is free once read
                const uint32_t h_cur = tm_h + (cl & 1) * H, h_nxt = tm_h + ((cl + 1) & 1) * H;
                if (ok) {
#pragma unroll 1
                    for (int m = 0; m < H / 16; ++m) {
                        uint32_t hv[16], uv[16];
                        const float am = (HP && 16 * m >= HH) ? alpha1 : alpha;  // this column group's head
                        tc::tmem_ld16_nowait(h_cur + lane_base + 16 * m, hv);
                        tc::tmem_ld16_nowait(tm_u0 + ub * H + lane_base + 16 * m, uv);
                        tc::tmem_wait_ld16(hv);
                        tc::tmem_wait_ld16(uv);
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            hv[e] = __float_as_uint(fmaf(am, __uint_as_float(hv[e]), __uint_as_float(uv[e])));
                        tc::tmem_st16(h_nxt + lane_base + 16 * m, hv);
                    }
                }
                tc::tmem_wait_st();
                tc::tc_fence_before();
                __syncwarp();
                if (ok && lane == 0) tc::mbar_arrive(&bars[kBarUFree + ub]);
                // h_c, still in h_cur, leaves through the staging tiles: one
                // pass when every 64-row half has its own tile (both quadrant
                // pairs fill at once), else one pass per half through the one
                // tile.  Each pass first waits until the stores before it have
                // read the tiles (usually long done).
                for (int pass = 0; store && pass < npass; ++pass) {
                    if (leader) tc::bulk_wait_read_all();
                    asm volatile("bar.sync 1, %0;" ::"r"(kScanWarps * 32) : "memory");
                    const int hq = q >> 1;  // this quadrant pair's half
                    if (ok && (npass == 1 ? hq < nhalf : hq == pass)) {
                        uint8_t* tile = stg + (npass == 1 ? hq : 0) * tile_bytes;
#pragma unroll 1
                        for (int m = 0; m < H / 16; ++m) {
                            uint32_t hv[16];
                            tc::tmem_ld16(h_cur + lane_base + 16 * m, hv);
                            if (SPLIT) {
                                // fp32: columns 16m .. 16m + 15 are 16-byte
                                // chunks 4 (m & 1) .. + 3 of box m / 2
                                uint8_t* rowp = tile + (m >> 1) * 8192 + hrow * 128;
#pragma unroll
                                for (int j = 0; j < 4; ++j)
                                    *reinterpret_cast<uint4*>(rowp + (((4 * (m & 1) + j) ^ (hrow & 7)) << 4)) =
                                        make_uint4(hv[4 * j], hv[4 * j + 1], hv[4 * j + 2], hv[4 * j + 3]);
                            } else {
                                uint8_t* rowp = tile + (m >> 2) * 8192 + hrow * 128;
#pragma unroll
                                for (int s4 = 0; s4 < 2; ++s4) {
                                    const int e = 8 * s4, j = 2 * (m & 3) + s4;  // 16-byte chunk in the row
                                    uint32_t wh[4];
#pragma unroll
                                    for (int x = 0; x < 4; ++x)
                                        wh[x] = tc::pack_bf16x2(__uint_as_float(hv[e + 2 * x]),
                                                                __uint_as_float(hv[e + 2 * x + 1]));
                                    *reinterpret_cast<uint4*>(rowp + ((j ^ (hrow & 7)) << 4)) =
                                        make_uint4(wh[0], wh[1], wh[2], wh[3]);
                                }
                            }
                        }
                        tc::fence_proxy_async_smem();
                    }
                    asm volatile("bar.sync 1, %0;" ::"r"(kScanWarps * 32) : "memory");
                    if (leader && ok) {
                        constexpr int scols = SPLIT ? 32 : 64;  // columns per box (fp32 / bf16)
                        for (int hf = (npass == 1 ? 0 : pass); hf < (npass == 1 ? nhalf : pass + 1); ++hf)
                            for (int cb = 0; cb < H / scols; ++cb)
                                // HP: box cb is head hr + cb's 64 columns, in its own rows
                                tc::tma_store_2d(&tm_cs, stg + (npass == 1 ? hf : 0) * tile_bytes + cb * 8192,
                                                 HP ? 0 : cb * scols,
                                                 (int)(row0 + 64 * hf + (HP ? cb * g.nchunks * S : 0)));
                        tc::bulk_commit();
                    }
                }
            }
            if (leader) tc::bulk_wait_all();
            // the end state: a summary's into its segment slot, the last
            // segment's into final_state
            float* h_out = nullptr;
            int64_t out_stride = (int64_t)S * HH;  // from one head's end state to the next head's
            if (p.mode == kSegmentSummary) {
                h_out = p.seg_states + (bh * (p.nseg - 1) + seg) * S * HH;
                out_stride = (int64_t)(p.nseg - 1) * S * HH;
            } else if (seg == p.nseg - 1 && p.final_state) {
                h_out = p.final_state + bh * S * HH;
            }
            if (ok && h_out && valid) {
#pragma unroll 1
                for (int m = 0; m < H / 16; ++m) {
                    uint32_t hv[16];
                    tc::tmem_ld16(tm_h + (nchl & 1) * H + lane_base + 16 * m, hv);  // h after the last chunk
                    float4* d4 = reinterpret_cast<float4*>(h_out + ((16 * m) / HH) * out_stride + s * HH + (16 * m) % HH);
#pragma unroll
                    for (int s4 = 0; s4 < 4; ++s4)
                        d4[s4] = make_float4(__uint_as_float(hv[4 * s4]), __uint_as_float(hv[4 * s4 + 1]),
                                             __uint_as_float(hv[4 * s4 + 2]), __uint_as_float(hv[4 * s4 + 3]));
                }
            }
        }
        if (!ok) set_abort(ctl, p.status);
    }

    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, p.tmem_cols);
    }
}

// Carry over segments (see the file comment): one thread per state element
// of one (batch, head); slot k of seg_states holds segment k's end state on
// entry and the state entering segment k + 1 on exit.
__global__ void __launch_bounds__(256) k_state_carry(const float* __restrict__ G, float* seg_states, Geom g,
                                                    int nseg, int cps) {
    __shared__ float decay[64];  // exp2(D_k), k < nseg - 1
    const int64_t bh = blockIdx.y;
    const int64_t SH = g.dstate * g.headdim;
    tc::griddep_launch_dependents();  // the segment pass may start; it waits for this grid
    tc::griddep_wait();               // G and the end states come from the previous kernels
    {
        // D_k = sum of G_last over the chunks of segment k (all whole chunks:
        // only the last segment, which is never carried out of, can be ragged);
        // warp w sums segments w, w + 8, ..., its lanes over strided chunks
        const float* Gbh = G + bh * g.seqlen;
        const int w = threadIdx.x / 32, lane = threadIdx.x % 32;
        for (int k = w; k < nseg - 1; k += 8) {
            float d = 0.f;
            for (int c = k * cps + lane; c < (k + 1) * cps; c += 32) d += Gbh[(int64_t)c * g.chunk + g.chunk - 1];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
            if (lane == 0) decay[k] = exp2f(d);
        }
    }
    __syncthreads();
    const int64_t e = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (e >= SH) return;
    float* slot = seg_states + bh * (nseg - 1) * SH + e;
    float hk = slot[0];  // H_1: segment 0 started from the initial state
    // eight end states are loaded before any is overwritten, so the loads
    // overlap instead of waiting behind the stores
    for (int k0 = 1; k0 < nseg - 1; k0 += 8) {
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = (k0 + i < nseg - 1) ? slot[(k0 + i) * SH] : 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (k0 + i < nseg - 1) {
                hk = fmaf(decay[k0 + i], hk, v[i]);
                slot[(k0 + i) * SH] = hk;
            }
        }
    }
}

// Ring plan.  Two CTAs share an SM when TMEM allows and the grid has enough
// CTAs to use them; a grid of at most one CTA per SM (ctas_per_sm_cap = 1)
// gets the whole shared memory, i.e. a deeper ring.
// A split (fp32) problem's stages hold B's hi and lo tiles and fp32 x (the
// bytes of x's hi/lo pair): one CTA per SM with a ring of 64-token
// sub-blocks.
bool plan(const Geom& g, SpTcParams& p, int ctas_per_sm_cap = 2, bool split = false, bool hp = false) {
    const int H = hp ? 128 : (int)g.headdim;  // head pairs run as one head of 128 columns
    p.tmem_cols = (4 * H <= 256) ? 256 : 512;  // U x 2, h x 2
    const bool two = p.tmem_cols == 256 && ctas_per_sm_cap >= 2 && !split;
    const int kKb = (!two && g.chunk >= 128 && !split) ? 128 : 64;
    const uint32_t planes = split ? 2 : 1;
    p.kb = kKb;
    p.nsb = (int)(g.chunk / kKb);
    p.off_blo_in_stage = 2 * kKb * 128;
    p.off_x_in_stage = planes * 2 * kKb * 128;
    // split: a 64-column group's lo box follows its hi box
    p.off_xlo_in_stage = p.off_x_in_stage + kKb * 128;
    p.off_w_in_stage = p.off_x_in_stage + planes * (H / 64) * kKb * 128;
    // G[kKb], dt[kKb], G_last (of each head of a pair); padded to keep stages 1 KB aligned
    p.stage_bytes = p.off_w_in_stage + ((hp ? 2 : 1) * (2 * kKb + 1) * 4 + 1023) / 1024 * 1024;
    const uint32_t budget = two ? (kSmemLimit / 2 - 2048) : kSmemLimit;
    const uint32_t fixed = kNumBars * 8 + 64 + 1024;
    // Staging tiles of 64 rows x H: bf16 (boxes of 64 columns), or fp32
    // (split; boxes of 32).  A tile per 64-row half (the two halves of a
    // chunk leave at once), except at two CTAs per SM with more than two
    // sub-blocks per chunk, where one tile keeps a ring stage more (each
    // measured faster where it is used).
    p.stg_tiles = (g.dstate >= 128 && (!two || p.nsb <= 2)) ? 2 : 1;
    const uint32_t stg_bytes = p.stg_tiles * planes * (uint32_t)(H / 64) * 8192;
    int nst = (int)((budget - fixed - stg_bytes) / p.stage_bytes);
    if (nst > kMaxStages) nst = kMaxStages;
    if (nst < 2) return false;
    p.nst = nst;
    p.off_stg = nst * p.stage_bytes;
    p.off_bar = p.off_stg + stg_bytes;
    p.smem_bytes = p.off_bar + fixed;
    return true;
}

}  // namespace

// SMs of the GPU the library is built for (GB300); sets how many segments
// fill it.  A pure function of the shape, so the workspace size is too.
constexpr int kTargetSms = 152;

int state_pass_segments(const Geom& g) {
    SpTcParams p;
    if (!state_pass_tc_fits(g) || !plan(g, p)) return 1;
    // MAMBA2_STATE_SEGMENTS=1 forces one pass over each sequence (for timing
    // both on one shape)
    const char* env = getenv("MAMBA2_STATE_SEGMENTS");
    if (env && env[0] == '1' && env[1] == 0) return 1;
    const int64_t per_sm = (p.tmem_cols == 256) ? 2 : 1;  // resident CTAs per SM
    const int64_t base = g.batch * g.nheads * ((g.dstate + 127) / 128);
    int64_t nseg = kTargetSms * per_sm / base;
    // at least 4 chunks a segment, at most 64 segments; worth it from 3
    // segments on (the summary and segment passes each walk one segment)
    nseg = imin64(imin64(nseg, g.nchunks / 4), 64);
    if (nseg < 3) return 1;
    const int64_t cps = (g.nchunks + nseg - 1) / nseg;
    return (int)((g.nchunks + cps - 1) / cps);
}

int64_t state_pass_segment_bytes(const Geom& g) {
    const int nseg = state_pass_segments(g);
    return nseg > 1 ? g.batch * g.nheads * (nseg - 1) * g.dstate * g.headdim * 4 : 0;
}

// The split (fp32) state pass: chunks of 128, one pass.
bool state_pass_split_fits(const Geom& g) {
    SpTcParams p;
    return g.chunk == 128 && state_pass_tc_fits(g) && plan(g, p, 1, true);
}

bool state_pass_tc_fits(const Geom& g) {
    if (g.chunk != 64 && g.chunk != 128 && g.chunk != 256) return false;
    if (g.headdim != 64 && g.headdim != 128) return false;
    if (g.dstate != 64 && g.dstate != 128 && g.dstate != 256) return false;
    if (g.batch * g.seqlen >= (int64_t(1) << 31)) return false;
    // chunk-state rows are TMA coordinates (32-bit)
    if (g.batch * g.nheads * g.nchunks * g.dstate >= (int64_t(1) << 31)) return false;
    SpTcParams p;
    return plan(g, p);
}

cudaError_t launch_state_pass_tc(const Geom& g, const StatePassArgs& a, cudaStream_t st) {
    SpTcParams p{};
    p.g = g;
    const bool hp = use_head_pairs(g, a);  // the rule lives with the other per-shape choices
    const int mtiles = (int)((g.dstate + 127) / 128);
    const int seg_grid = a.segments > 1 ? (a.summary ? a.segments - 1 : a.segments) : 1;
    const int64_t heads = hp ? g.nheads / 2 : g.nheads;  // CTAs along the heads
    const int64_t ctas = (int64_t)mtiles * heads * g.batch * seg_grid;
    const bool split = a.split;
    if (split && (a.segments > 1 || g.chunk != 128)) return cudaErrorInvalidConfiguration;
    if (!plan(g, p, ctas <= kTargetSms ? 1 : 2, split, hp)) return cudaErrorInvalidConfiguration;
    p.mode = kWholeSequence;
    p.nseg = 1;
    p.cps = (int)g.nchunks;
    p.seg_grid = 1;
    p.seg_states = nullptr;
    if (a.segments > 1) {
        p.mode = a.summary ? kSegmentSummary : kSegmentPass;
        p.nseg = a.segments;
        p.cps = (int)((g.nchunks + a.segments - 1) / a.segments);
        p.seg_grid = a.summary ? a.segments - 1 : a.segments;
        p.seg_states = a.seg_states;
    }
    p.dt = a.dt;
    p.G = a.G;
    p.init = a.init;
    p.chunk_states = static_cast<__nv_bfloat16*>(a.chunk_states);
    p.final_state = a.final_state;
    p.status = device_status_word();
    const uint64_t H = g.headdim, S = g.dstate, nh = g.nheads, L = g.seqlen, G = g.ngroups;
    const int kKb = p.kb;
    const uint64_t planes = split ? 2 : 1;  // split: B's hi/lo planes as twice the groups
    const uint64_t xe = split ? 4 : 2;       // bytes of an x and chunk-state element
    const uint32_t xcols = split ? 32 : 64;  // columns of their boxes
    CUtensorMap tm_x, tm_b;
    {
        // head pairs: x viewed as nh / 2 heads of 128 columns (a pair's rows are adjacent)
        const uint64_t Hx = hp ? 2 * H : H, nhx = hp ? nh / 2 : nh;
        const uint64_t dims[4] = {Hx, nhx, L, (uint64_t)g.batch};
        const uint64_t strides[3] = {Hx * xe, nhx * Hx * xe, L * nhx * Hx * xe};
        const uint32_t box[4] = {xcols, 1, (uint32_t)kKb, 1};
        if (!make_tmap(&tm_x, split ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, 4,
                       dims, strides, box))
            return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[4] = {S, planes * G, L, (uint64_t)g.batch};
        const uint64_t strides[3] = {S * 2, planes * G * S * 2, L * planes * G * S * 2};
        const uint32_t box[4] = {64, 1, kKb, 1};
        if (!make_tmap_bf16(&tm_b, a.B, 4, dims, strides, box)) return cudaErrorInvalidValue;
    }
    CUtensorMap tm_cs;
    {
        const uint64_t rows = (uint64_t)g.batch * nh * g.nchunks * S;
        const uint64_t dims[2] = {H, rows};
        const uint64_t strides[1] = {H * xe};
        const uint32_t box[2] = {xcols, 64};
        if (!make_tmap(&tm_cs, split ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                       a.chunk_states, 2, dims, strides, box))
            return cudaErrorInvalidValue;
    }
    auto kern = split ? (g.headdim == 64 ? k_state_pass_tc<64, 128, 64, true> : k_state_pass_tc<128, 128, 64, true>)
                : hp ? (g.chunk == 256 ? k_state_pass_tc<128, 256, 128, false, true>
                        : g.chunk == 128 ? k_state_pass_tc<128, 128, 128, false, true>
                                         : k_state_pass_tc<128, 64, 64, false, true>)
                : (g.headdim == 64)
                    ? (g.chunk == 256 ? (kKb == 128 ? k_state_pass_tc<64, 256, 128, false> : k_state_pass_tc<64, 256, 64, false>)
                       : g.chunk == 128 ? (kKb == 128 ? k_state_pass_tc<64, 128, 128, false> : k_state_pass_tc<64, 128, 64, false>)
                                        : k_state_pass_tc<64, 64, 64, false>)
                    : (g.chunk == 256 ? k_state_pass_tc<128, 256, 128, false>
                       : g.chunk == 128 ? k_state_pass_tc<128, 128, 128, false> : k_state_pass_tc<128, 64, 64, false>);
    cudaError_t e = ensure_max_dynamic_smem(reinterpret_cast<const void*>(kern), (int)p.smem_bytes);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)mtiles, (unsigned)heads, (unsigned)(g.batch * p.seg_grid));
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
    return cudaLaunchKernelEx(&cfg, kern, tm_x, tm_b, tm_cs, p);
}

cudaError_t launch_state_carry(const Geom& g, const float* G, float* seg_states, int nseg, bool pdl,
                               cudaStream_t st) {
    const int cps = (int)((g.nchunks + nseg - 1) / nseg);
    dim3 grid((unsigned)((g.dstate * g.headdim + 255) / 256), (unsigned)(g.batch * g.nheads));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k_state_carry, G, seg_states, g, nseg, cps);
}

}  // namespace m2
