/*
 * ssd_oracle.c — plain fp64 CPU oracle for the Mamba-2 chunked SSD forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
 * and its Python binding) may include, link, load or call this file.  Only the
 * tests, the package's smoke check and the CPU-baseline leg of the benchmark
 * use it.  It shares no code, header, table or constant generator with the
 * CUDA path.
 *
 * Source: "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in
 * NVIDIA CUDA Tile" (NVIDIA technical blog), cited below as [blog §section].
 *
 * What it computes
 * ----------------
 *   a_t = A[h] * dt_t                         [blog §Mamba-2 architecture]
 *   h_t = exp(a_t) h_{t-1} + dt_t B_t x_t^T   (h is S x H)
 *   y_t = C_t^T h_t + D[h] x_t                (inclusive state: the output at
 *                                              token t sees h_t, i.e. the
 *                                              diagonal term j = t; this is the
 *                                              reading of the expanded output
 *                                              formula and of the i >= j mask)
 *
 * Four entry points:
 *   oracle_ssd_recurrence  token-by-token recurrence, the definition itself;
 *   oracle_chunk_cumsum    stage 1: G = log2(e) * intra-chunk inclusive cumsum
 *                          of a_t                   [blog §Kernel 1]
 *   oracle_state_pass      stage 2: chunk-start states by the decayed jump
 *                          formula                  [blog §Kernel 2]
 *   oracle_chunk_out       stage 3: per-chunk outputs from the chunk-start
 *                          states                   [blog §Kernel 3]
 * Stages 1-3 follow the blog's order and notation with no blocking, fusion or
 * reordering; chained, they must agree with the recurrence (the chunked
 * formulas are exact rewrites of it).  A ragged last chunk (L % T != 0) is
 * handled with G_last taken at the last valid token.
 *
 * Layouts (row-major, contiguous):
 *   x  [batch, L, nheads, H]      dt [batch, L, nheads]     A, D [nheads]
 *   B, C [batch, L, ngroups, S]   group of head h = h / (nheads / ngroups)
 *   state / init / final [batch, nheads, S, H]
 *   chunk_states [batch, nheads, nchunks, S, H]  (state at the start of chunk c)
 *   G [batch, nheads, L]          (log2 units)
 *
 * Work is split over (batch, head) pairs with POSIX threads; each pair's
 * arithmetic is sequential, so the result does not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int64_t batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size;
} oracle_dims;

/* ---------------------------------------------------------------- helpers */

static inline int64_t idx_x(const oracle_dims* d, int64_t b, int64_t t, int64_t h) {
    return ((b * d->seqlen + t) * d->nheads + h) * d->headdim;
}
static inline int64_t idx_dt(const oracle_dims* d, int64_t b, int64_t t, int64_t h) {
    return (b * d->seqlen + t) * d->nheads + h;
}
static inline int64_t idx_bc(const oracle_dims* d, int64_t b, int64_t t, int64_t g) {
    return ((b * d->seqlen + t) * d->ngroups + g) * d->dstate;
}
static inline int64_t idx_state(const oracle_dims* d, int64_t b, int64_t h) {
    return (b * d->nheads + h) * d->dstate * d->headdim;
}
static inline int64_t nchunks_of(const oracle_dims* d) {
    return (d->seqlen + d->chunk_size - 1) / d->chunk_size;
}
static inline int64_t idx_chunk_state(const oracle_dims* d, int64_t b, int64_t h, int64_t c) {
    return ((b * d->nheads + h) * nchunks_of(d) + c) * d->dstate * d->headdim;
}
static inline int64_t group_of(const oracle_dims* d, int64_t h) {
    return h / (d->nheads / d->ngroups);
}

/* A work item is one (batch, head) pair.  `pairs` lists them as
 * (b0, h0, b1, h1, ...); NULL means every pair in order. */
typedef void (*pair_fn)(const void* ctx, int64_t b, int64_t h);

typedef struct {
    pair_fn fn;
    const void* ctx;
    const int64_t* pairs;
    int64_t npairs;
    int64_t nheads;
    int64_t next; /* shared work counter */
} pool_job;

static void run_item(pool_job* job, int64_t i) {
    int64_t b, h;
    if (job->pairs) {
        b = job->pairs[2 * i];
        h = job->pairs[2 * i + 1];
    } else {
        b = i / job->nheads;
        h = i % job->nheads;
    }
    job->fn(job->ctx, b, h);
}

static void* pool_worker(void* arg) {
    pool_job* job = (pool_job*)arg;
    for (;;) {
        int64_t i = __atomic_fetch_add(&job->next, 1, __ATOMIC_RELAXED);
        if (i >= job->npairs) break;
        run_item(job, i);
    }
    return NULL;
}

static int run_pairs(pair_fn fn, const void* ctx, const oracle_dims* d,
                     const int64_t* pairs, int64_t npairs, int nthreads) {
    pool_job job;
    job.fn = fn;
    job.ctx = ctx;
    job.pairs = pairs;
    job.npairs = pairs ? npairs : d->batch * d->nheads;
    job.nheads = d->nheads;
    job.next = 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (nthreads > job.npairs) nthreads = (int)(job.npairs > 0 ? job.npairs : 1);
    pthread_t tids[256];
    int started = 0;
    for (int i = 1; i < nthreads; ++i) {
        if (pthread_create(&tids[started], NULL, pool_worker, &job) != 0) break;
        ++started;
    }
    pool_worker(&job);
    for (int i = 0; i < started; ++i) pthread_join(tids[i], NULL);
    return 0;
}

static int dims_ok(const oracle_dims* d) {
    if (!d) return 0;
    if (d->batch < 0 || d->seqlen < 0 || d->nheads < 1 || d->headdim < 1 || d->dstate < 1 ||
        d->ngroups < 1 || d->nheads % d->ngroups != 0)
        return 0;
    return 1;
}

/* ------------------------------------------------ token-by-token recurrence */

typedef struct {
    const oracle_dims* d;
    const double *x, *dt, *A, *B, *C, *D, *init;
    double *y, *final_state, *chunk_states;
} rec_ctx;

/* [blog §Mamba-2 architecture]: h_t = exp(A dt_t) h_{t-1} + dt_t B_t x_t^T,
 * y_t = C_t^T h_t + D x_t, with h_0 = init (zeros when absent). */
static void rec_pair(const void* vctx, int64_t b, int64_t h) {
    const rec_ctx* c = (const rec_ctx*)vctx;
    const oracle_dims* d = c->d;
    const int64_t S = d->dstate, H = d->headdim, g = group_of(d, h);
    double* st = (double*)calloc((size_t)(S * H), sizeof(double));
    double* yacc = (double*)malloc((size_t)H * sizeof(double));
    if (c->init) memcpy(st, c->init + idx_state(d, b, h), (size_t)(S * H) * sizeof(double));
    const double Dh = c->D ? c->D[h] : 0.0;
    for (int64_t t = 0; t < d->seqlen; ++t) {
        if (c->chunk_states && d->chunk_size > 0 && t % d->chunk_size == 0)
            memcpy(c->chunk_states + idx_chunk_state(d, b, h, t / d->chunk_size), st,
                   (size_t)(S * H) * sizeof(double));
        const double dtt = c->dt[idx_dt(d, b, t, h)];
        const double decay = exp(c->A[h] * dtt);
        const double* xt = c->x + idx_x(d, b, t, h);
        const double* Bt = c->B + idx_bc(d, b, t, g);
        const double* Ct = c->C + idx_bc(d, b, t, g);
        for (int64_t k = 0; k < H; ++k) yacc[k] = 0.0;
        for (int64_t s = 0; s < S; ++s) {
            const double bs = dtt * Bt[s];
            const double cs = Ct[s];
            double* row = st + s * H;
            for (int64_t k = 0; k < H; ++k) {
                row[k] = decay * row[k] + bs * xt[k];
                yacc[k] += cs * row[k];
            }
        }
        double* yt = c->y + idx_x(d, b, t, h);
        for (int64_t k = 0; k < H; ++k) yt[k] = yacc[k] + Dh * xt[k];
    }
    if (c->final_state) memcpy(c->final_state + idx_state(d, b, h), st, (size_t)(S * H) * sizeof(double));
    free(yacc);
    free(st);
}

/* Returns 0 on success, -1 on invalid dims.  `init`, `D`, `final_state` and
 * `chunk_states` may be NULL.  chunk_states (when given, with chunk_size > 0)
 * receives the state at the start of every chunk: chunk 0 holds `init`. */
int oracle_ssd_recurrence(const oracle_dims* d, const double* x, const double* dt, const double* A,
                          const double* B, const double* C, const double* D, const double* init,
                          double* y, double* final_state, double* chunk_states,
                          const int64_t* pairs, int64_t npairs, int nthreads) {
    if (!dims_ok(d) || !x || !dt || !A || !B || !C || !y) return -1;
    if (chunk_states && d->chunk_size < 1) return -1;
    rec_ctx c = {d, x, dt, A, B, C, D, init, y, final_state, chunk_states};
    return run_pairs(rec_pair, &c, d, pairs, npairs, nthreads);
}

/* ------------------------------------------------------ stage 1: cumsum G */

typedef struct {
    const oracle_dims* d;
    const double *dt, *A;
    double* G;
} cumsum_ctx;

/* [blog §Kernel 1]: the effective decay a[h] * dt[t, h] is summed along the
 * token axis inside each chunk (the sum restarts at every chunk start), then
 * scaled by log2(e) so that later stages can use exp2. */
static void cumsum_pair(const void* vctx, int64_t b, int64_t h) {
    const cumsum_ctx* c = (const cumsum_ctx*)vctx;
    const oracle_dims* d = c->d;
    double* Gbh = c->G + (b * d->nheads + h) * d->seqlen;
    double run = 0.0;
    for (int64_t t = 0; t < d->seqlen; ++t) {
        if (t % d->chunk_size == 0) run = 0.0;
        run += c->A[h] * c->dt[idx_dt(d, b, t, h)];
        Gbh[t] = run * M_LOG2E;
    }
}

int oracle_chunk_cumsum(const oracle_dims* d, const double* dt, const double* A, double* G,
                        const int64_t* pairs, int64_t npairs, int nthreads) {
    if (!dims_ok(d) || d->chunk_size < 1 || !dt || !A || !G) return -1;
    cumsum_ctx c = {d, dt, A, G};
    return run_pairs(cumsum_pair, &c, d, pairs, npairs, nthreads);
}

/* ------------------------------------------------ stage 2: chunk-start states */

typedef struct {
    const oracle_dims* d;
    const double *x, *dt, *B, *G, *init;
    double *chunk_states, *final_state;
} state_ctx;

/* [blog §Kernel 2 / §Mamba-2 architecture, decayed jump formula]:
 *   store h (the state entering chunk c), then
 *   h <- exp2(G_last) h + sum_t exp2(G_last - G_t) dt_t B_t x_t^T,
 * where G is stage 1's output (log2 units) and G_last is G at the chunk's last
 * token.  After the last chunk h is the final state. */
static void state_pair(const void* vctx, int64_t b, int64_t h) {
    const state_ctx* c = (const state_ctx*)vctx;
    const oracle_dims* d = c->d;
    const int64_t S = d->dstate, H = d->headdim, g = group_of(d, h), T = d->chunk_size;
    const double* Gbh = c->G + (b * d->nheads + h) * d->seqlen;
    double* st = (double*)calloc((size_t)(S * H), sizeof(double));
    if (c->init) memcpy(st, c->init + idx_state(d, b, h), (size_t)(S * H) * sizeof(double));
    const int64_t nc = nchunks_of(d);
    for (int64_t ch = 0; ch < nc; ++ch) {
        if (c->chunk_states)
            memcpy(c->chunk_states + idx_chunk_state(d, b, h, ch), st, (size_t)(S * H) * sizeof(double));
        const int64_t t0 = ch * T;
        const int64_t t1 = (t0 + T < d->seqlen) ? t0 + T : d->seqlen;
        const double g_last = Gbh[t1 - 1];
        const double carry = exp2(g_last);
        for (int64_t i = 0; i < S * H; ++i) st[i] *= carry;
        for (int64_t t = t0; t < t1; ++t) {
            const double w = exp2(g_last - Gbh[t]) * c->dt[idx_dt(d, b, t, h)];
            const double* Bt = c->B + idx_bc(d, b, t, g);
            const double* xt = c->x + idx_x(d, b, t, h);
            for (int64_t s = 0; s < S; ++s) {
                const double bw = Bt[s] * w;
                double* row = st + s * H;
                for (int64_t k = 0; k < H; ++k) row[k] += bw * xt[k];
            }
        }
    }
    if (c->final_state) memcpy(c->final_state + idx_state(d, b, h), st, (size_t)(S * H) * sizeof(double));
    free(st);
}

int oracle_state_pass(const oracle_dims* d, const double* x, const double* dt, const double* B,
                      const double* G, const double* init, double* chunk_states, double* final_state,
                      const int64_t* pairs, int64_t npairs, int nthreads) {
    if (!dims_ok(d) || d->chunk_size < 1 || !x || !dt || !B || !G) return -1;
    state_ctx c = {d, x, dt, B, G, init, chunk_states, final_state};
    return run_pairs(state_pair, &c, d, pairs, npairs, nthreads);
}

/* ------------------------------------------------------ stage 3: outputs */

typedef struct {
    const oracle_dims* d;
    const double *x, *dt, *B, *C, *D, *G, *chunk_states;
    double* y;
} out_ctx;

/* [blog §Kernel 3, Phases 1 and 2]: for each token i of chunk c,
 *   y_i = exp2(G_i) (C_i . h_c) + sum_{j in chunk, j <= i} (C_i . B_j) exp2(G_i - G_j) dt_j x_j
 *         + D x_i,
 * h_c being the state entering the chunk.  Terms with j > i are the ones the
 * causal mask removes; they are never formed here. */
static void out_pair(const void* vctx, int64_t b, int64_t h) {
    const out_ctx* c = (const out_ctx*)vctx;
    const oracle_dims* d = c->d;
    const int64_t S = d->dstate, H = d->headdim, g = group_of(d, h), T = d->chunk_size;
    const double* Gbh = c->G + (b * d->nheads + h) * d->seqlen;
    const double Dh = c->D ? c->D[h] : 0.0;
    double* acc = (double*)malloc((size_t)H * sizeof(double));
    const int64_t nc = nchunks_of(d);
    for (int64_t ch = 0; ch < nc; ++ch) {
        const double* hc = c->chunk_states + idx_chunk_state(d, b, h, ch);
        const int64_t t0 = ch * T;
        const int64_t t1 = (t0 + T < d->seqlen) ? t0 + T : d->seqlen;
        for (int64_t i = t0; i < t1; ++i) {
            const double* Ci = c->C + idx_bc(d, b, i, g);
            /* carried-state term: exp2(G_i) * C_i^T h_c */
            for (int64_t k = 0; k < H; ++k) acc[k] = 0.0;
            for (int64_t s = 0; s < S; ++s) {
                const double cs = Ci[s];
                const double* row = hc + s * H;
                for (int64_t k = 0; k < H; ++k) acc[k] += cs * row[k];
            }
            const double carry = exp2(Gbh[i]);
            for (int64_t k = 0; k < H; ++k) acc[k] *= carry;
            /* decayed, causally masked interaction term */
            for (int64_t j = t0; j <= i; ++j) {
                const double* Bj = c->B + idx_bc(d, b, j, g);
                double cb = 0.0;
                for (int64_t s = 0; s < S; ++s) cb += Ci[s] * Bj[s];
                const double p = cb * exp2(Gbh[i] - Gbh[j]) * c->dt[idx_dt(d, b, j, h)];
                const double* xj = c->x + idx_x(d, b, j, h);
                for (int64_t k = 0; k < H; ++k) acc[k] += p * xj[k];
            }
            /* skip connection */
            const double* xi = c->x + idx_x(d, b, i, h);
            double* yi = c->y + idx_x(d, b, i, h);
            for (int64_t k = 0; k < H; ++k) yi[k] = acc[k] + Dh * xi[k];
        }
    }
    free(acc);
}

int oracle_chunk_out(const oracle_dims* d, const double* x, const double* dt, const double* B,
                     const double* C, const double* D, const double* G, const double* chunk_states,
                     double* y, const int64_t* pairs, int64_t npairs, int nthreads) {
    if (!dims_ok(d) || d->chunk_size < 1 || !x || !dt || !B || !C || !G || !chunk_states || !y) return -1;
    out_ctx c = {d, x, dt, B, C, D, G, chunk_states, y};
    return run_pairs(out_pair, &c, d, pairs, npairs, nthreads);
}
