/*
 * gdn_oracle.c -- fp64 CPU oracle for the gated delta rule (GDN) forward and its reverse mode.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load or call this file.  It shares no code, header,
 * table or helper with the CUDA library; neither includes nor links the other.
 *
 * Sources (web pages, cited by title and section):
 *   [CP]   "Add context parallelism to the Gated Delta Net (Qwen3-Next / Qwen3.5)",
 *          MaxText pull request #5040.
 *            - section "Why": the chunked rule is affine in the incoming state,
 *              h_out = (gamma I - k_tilde^T w) h + k_tilde^T u = M h + U and
 *              o = (q_g - attn_i w) h + attn_i u; affine maps compose associatively.
 *            - section "Implementation": the three phases (zero-state pass carrying M_r,
 *              exclusive prefix scan over (M_r, U_r), re-emit from the true state reusing
 *              the WY factors), the low-rank composition M_new = gamma M - k_tilde^T (w M),
 *              and the chunk-padding bullet (g = 0, q = k = v = 0 is a no-op).
 *            - section "Limitation: load balancing must be off": segments are contiguous
 *              and in sequence order.
 *   [TP]   "RFC(qwen35): TP Phase2", pegainfer issue #694, "Partition Contract": the
 *          recurrent state is [Hv, K, V] in f32 (here widened to f64).
 *
 * The per-token recurrence (the plain definition everything else must reproduce):
 *     h_t = exp(g_t) (I - beta_t k_t k_t^T) h_{t-1} + beta_t k_t v_t^T,   o_t = h_t^T q_t
 * with h a K x V matrix per value head.  [CP] "Why" names the chunk factors w, u, attn_i,
 * k_tilde, q_g and gamma without defining them; their definitions below are derived from
 * the recurrence (readings listed in the design notes):
 *     G_t      = sum_{s<=t} g_s (inclusive, within the chunk)    gamma = exp(G_L)
 *     A[t][j]  = beta_t exp(G_t - G_j) (k_t . k_j)  for j < t, else 0
 *     Tm       = (I + A)^{-1}        (forward substitution; Tm is unit lower triangular)
 *     w        = Tm diag(beta_t exp(G_t)) K        u = Tm diag(beta_t) V
 *     k_tilde_j= exp(G_L - G_j) k_j                q_g_t = exp(G_t) q_t
 *     attn_i[t][j] = exp(G_t - G_j) (q_t . k_j)  for j <= t, else 0
 *
 * Array layouts (row-major, all double unless stated):
 *     q, k [T, hk, K]    v [T, hv, V]    g, beta [T, hv]
 *     h0, h_final [N, hv, K, V] (h0 may be NULL = zeros)     out [T, hv, V]
 *     cu_seqlens int64 [N+1], cu[0] = 0, non-decreasing, cu[N] = T
 * Value head j reads key head j / (hv / hk) (grouped order, as the Ulysses page
 * "Ulysses attention: repeat KV heads when there are fewer than context ranks" repeats
 * KV heads: [kv0, kv0, kv1, kv1]).
 *
 * Segments: each sequence's Nc = ceil(L / C) chunks are split into P contiguous,
 * in-order segments; the first (Nc mod P) segments get one extra chunk; segments past
 * Nc are empty (identity transition).  Segment (n, r) has global index n * P + r.
 *
 * Every function returns 0 on success and a negative number on bad arguments.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ thread pool */

typedef void (*item_fn)(void* ctx, int64_t item);

typedef struct {
    item_fn fn;
    void* ctx;
    int64_t n_items;
    int64_t next; /* atomically incremented */
} pool_job;

static void* pool_worker(void* arg) {
    pool_job* job = (pool_job*)arg;
    for (;;) {
        int64_t i = __atomic_fetch_add(&job->next, 1, __ATOMIC_RELAXED);
        if (i >= job->n_items) break;
        job->fn(job->ctx, i);
    }
    return NULL;
}

/* Runs fn(ctx, i) for i in [0, n_items) on up to nthreads threads (the caller included). */
static void run_items(item_fn fn, void* ctx, int64_t n_items, int nthreads) {
    pool_job job = {fn, ctx, n_items, 0};
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (nthreads > n_items) nthreads = (int)(n_items > 0 ? n_items : 1);
    pthread_t tid[256];
    int started = 0;
    for (int i = 1; i < nthreads; ++i) {
        if (pthread_create(&tid[started], NULL, pool_worker, &job) == 0) ++started;
    }
    pool_worker(&job);
    for (int i = 0; i < started; ++i) pthread_join(tid[i], NULL);
}

static int check_geometry(int64_t T, int N, const int64_t* cu, int hk, int hv, int K, int V) {
    if (T < 0 || N < 1 || !cu || hk < 1 || hv < 1 || K < 1 || V < 1) return -1;
    if (hv % hk != 0) return -2;
    if (cu[0] != 0 || cu[N] != T) return -3;
    for (int n = 0; n < N; ++n)
        if (cu[n + 1] < cu[n]) return -4;
    return 0;
}

/* ------------------------------------------------- 1. the per-token recurrence */

typedef struct {
    const double *q, *k, *v, *g, *beta, *h0;
    const int64_t* cu;
    int N, hk, hv, K, V, ncb, cb;
    double *out, *h_final;
} token_ctx;

/* One work item = (sequence n, value head j, block of state columns).  State columns
 * are independent: column c of h only ever meets column c of v, so a block of them
 * runs on its own. */
static void token_item(void* vctx, int64_t item) {
    const token_ctx* c = (const token_ctx*)vctx;
    const int K = c->K, V = c->V, hk = c->hk, hv = c->hv;
    const int blk = (int)(item % c->ncb);
    const int j = (int)((item / c->ncb) % hv);
    const int n = (int)(item / ((int64_t)c->ncb * hv));
    const int kh = j / (hv / hk);
    const int c0 = blk * c->cb;
    const int c1 = (c0 + c->cb < V) ? c0 + c->cb : V;
    const int w = c1 - c0;
    double* h = (double*)malloc(sizeof(double) * (size_t)K * (size_t)w);
    double* p = (double*)malloc(sizeof(double) * (size_t)w);
    for (int i = 0; i < K; ++i)
        for (int cc = 0; cc < w; ++cc)
            h[(size_t)i * w + cc] =
                c->h0 ? c->h0[(((size_t)n * hv + j) * K + i) * V + c0 + cc] : 0.0;
    for (int64_t t = c->cu[n]; t < c->cu[n + 1]; ++t) {
        const double* kt = c->k + ((size_t)t * hk + kh) * K;
        const double* qt = c->q + ((size_t)t * hk + kh) * K;
        const double* vt = c->v + ((size_t)t * hv + j) * V + c0;
        const double alpha = exp(c->g[(size_t)t * hv + j]);
        const double b = c->beta[(size_t)t * hv + j];
        /* p = h^T k_t */
        for (int cc = 0; cc < w; ++cc) p[cc] = 0.0;
        for (int i = 0; i < K; ++i) {
            const double ki = kt[i];
            const double* hrow = h + (size_t)i * w;
            for (int cc = 0; cc < w; ++cc) p[cc] += hrow[cc] * ki;
        }
        /* delta = beta (v_t - alpha p);  h <- alpha h + k_t delta^T
         * (expanding exp(g)(I - beta k k^T) h + beta k v^T) */
        for (int cc = 0; cc < w; ++cc) p[cc] = b * (vt[cc] - alpha * p[cc]);
        for (int i = 0; i < K; ++i) {
            const double ki = kt[i];
            double* hrow = h + (size_t)i * w;
            for (int cc = 0; cc < w; ++cc) hrow[cc] = alpha * hrow[cc] + ki * p[cc];
        }
        /* o_t = h_t^T q_t */
        double* ot = c->out + ((size_t)t * hv + j) * V + c0;
        for (int cc = 0; cc < w; ++cc) ot[cc] = 0.0;
        for (int i = 0; i < K; ++i) {
            const double qi = qt[i];
            const double* hrow = h + (size_t)i * w;
            for (int cc = 0; cc < w; ++cc) ot[cc] += hrow[cc] * qi;
        }
    }
    if (c->h_final)
        for (int i = 0; i < K; ++i)
            for (int cc = 0; cc < w; ++cc)
                c->h_final[(((size_t)n * hv + j) * K + i) * V + c0 + cc] = h[(size_t)i * w + cc];
    free(h);
    free(p);
}

int gdn_oracle_token(const double* q, const double* k, const double* v, const double* g,
                     const double* beta, const double* h0, int64_t T, int N, const int64_t* cu,
                     int hk, int hv, int K, int V, int nthreads, double* out, double* h_final) {
    int rc = check_geometry(T, N, cu, hk, hv, K, V);
    if (rc) return rc;
    if (!q || !k || !v || !g || !beta || !out) return -1;
    token_ctx c = {q, k, v, g, beta, h0, cu, N, hk, hv, K, V, 0, 16, out, h_final};
    c.ncb = (V + c.cb - 1) / c.cb;
    run_items(token_item, &c, (int64_t)N * hv * c.ncb, nthreads);
    return 0;
}

/* --------------------------------------------- 2. one chunk's WY/UT factors */

/* Chunk factors for L <= C consecutive tokens of one value head.  Rows are contiguous:
 * kc [L, K], vc [L, V] (vc and u may be NULL when only w is wanted), gc, bc [L].
 * Outputs (each may be NULL except where a later output needs it internally):
 *   G [L], A [L, L], Tm [L, L], w [L, K], u [L, V], ktilde [L, K], gamma [1].
 * Follows [CP] "Why" with the definitions in the file header. */
int gdn_oracle_chunk_factors(int L, int K, int V, const double* kc, const double* vc,
                             const double* gc, const double* bc, double* G_out, double* A_out,
                             double* Tm_out, double* w_out, double* u_out, double* kt_out,
                             double* gamma_out) {
    if (L < 0 || K < 1 || V < 0 || (L > 0 && (!kc || !gc || !bc))) return -1;
    double* G = (double*)malloc(sizeof(double) * (size_t)(L + 1));
    double* A = (double*)calloc((size_t)L * L + 1, sizeof(double));
    double* Tm = (double*)calloc((size_t)L * L + 1, sizeof(double));
    /* G: inclusive cumulative log-decay within the chunk */
    double acc = 0.0;
    for (int t = 0; t < L; ++t) {
        acc += gc[t];
        G[t] = acc;
    }
    const double GL = L > 0 ? G[L - 1] : 0.0;
    /* A: strictly lower, beta_t exp(G_t - G_j) (k_t . k_j) */
    for (int t = 0; t < L; ++t)
        for (int j = 0; j < t; ++j) {
            double dot = 0.0;
            for (int i = 0; i < K; ++i) dot += kc[(size_t)t * K + i] * kc[(size_t)j * K + i];
            A[(size_t)t * L + j] = bc[t] * exp(G[t] - G[j]) * dot;
        }
    /* Tm = (I + A)^{-1} by forward substitution, row by row:
     * row t of (I + A) Tm = e_t gives Tm[t][:] = e_t - sum_{j<t} A[t][j] Tm[j][:]. */
    for (int t = 0; t < L; ++t) {
        for (int c = 0; c < L; ++c) Tm[(size_t)t * L + c] = (c == t) ? 1.0 : 0.0;
        for (int j = 0; j < t; ++j) {
            const double a = A[(size_t)t * L + j];
            if (a == 0.0) continue;
            for (int c = 0; c <= j; ++c) Tm[(size_t)t * L + c] -= a * Tm[(size_t)j * L + c];
        }
    }
    if (w_out)
        for (int t = 0; t < L; ++t)
            for (int i = 0; i < K; ++i) {
                double s = 0.0;
                for (int j = 0; j <= t; ++j)
                    s += Tm[(size_t)t * L + j] * bc[j] * exp(G[j]) * kc[(size_t)j * K + i];
                w_out[(size_t)t * K + i] = s;
            }
    if (u_out && vc)
        for (int t = 0; t < L; ++t)
            for (int c = 0; c < V; ++c) {
                double s = 0.0;
                for (int j = 0; j <= t; ++j) s += Tm[(size_t)t * L + j] * bc[j] * vc[(size_t)j * V + c];
                u_out[(size_t)t * V + c] = s;
            }
    if (kt_out)
        for (int j = 0; j < L; ++j)
            for (int i = 0; i < K; ++i) kt_out[(size_t)j * K + i] = exp(GL - G[j]) * kc[(size_t)j * K + i];
    if (gamma_out) *gamma_out = exp(GL);
    if (G_out) memcpy(G_out, G, sizeof(double) * (size_t)L);
    if (A_out) memcpy(A_out, A, sizeof(double) * (size_t)L * L);
    if (Tm_out) memcpy(Tm_out, Tm, sizeof(double) * (size_t)L * L);
    free(G);
    free(A);
    free(Tm);
    return 0;
}

/* Gathers the rows of chunk [t0, t0 + L) for value head j into contiguous buffers. */
static void gather_chunk(const double* q, const double* k, const double* v, const double* g,
                         const double* beta, int64_t t0, int L, int hk, int hv, int kh, int j, int K,
                         int V, double* qc, double* kc, double* vc, double* gc, double* bc) {
    for (int t = 0; t < L; ++t) {
        const size_t tt = (size_t)(t0 + t);
        if (qc) memcpy(qc + (size_t)t * K, q + (tt * hk + kh) * K, sizeof(double) * K);
        memcpy(kc + (size_t)t * K, k + (tt * hk + kh) * K, sizeof(double) * K);
        if (vc) memcpy(vc + (size_t)t * V, v + (tt * hv + j) * V, sizeof(double) * V);
        gc[t] = g[tt * hv + j];
        bc[t] = beta[tt * hv + j];
    }
}

/* All chunks of every sequence: w [T, hv, K], u [T, hv, V], gcum [T, hv] (the within-chunk
 * inclusive cumulative log-decay G).  Token-aligned; a sequence's last chunk may be short. */
typedef struct {
    const double *k, *v, *g, *beta;
    const int64_t* cu;
    int N, hk, hv, K, V, C;
    double *w, *u, *gcum;
} prep_ctx;

static void prep_item(void* vctx, int64_t item) {
    const prep_ctx* c = (const prep_ctx*)vctx;
    const int n = (int)(item / c->hv), j = (int)(item % c->hv);
    const int K = c->K, V = c->V, C = c->C, kh = j / (c->hv / c->hk);
    double* kc = (double*)malloc(sizeof(double) * (size_t)C * K);
    double* vc = (double*)malloc(sizeof(double) * (size_t)C * V);
    double* wc = (double*)malloc(sizeof(double) * (size_t)C * K);
    double* uc = (double*)malloc(sizeof(double) * (size_t)C * V);
    double gc[1024], bc[1024], G[1024];
    for (int64_t t0 = c->cu[n]; t0 < c->cu[n + 1]; t0 += C) {
        const int L = (int)((c->cu[n + 1] - t0 < C) ? c->cu[n + 1] - t0 : C);
        gather_chunk(NULL, c->k, c->v, c->g, c->beta, t0, L, c->hk, c->hv, kh, j, K, V, NULL, kc,
                     vc, gc, bc);
        gdn_oracle_chunk_factors(L, K, V, kc, vc, gc, bc, G, NULL, NULL, wc, uc, NULL, NULL);
        for (int t = 0; t < L; ++t) {
            const size_t tt = (size_t)(t0 + t);
            memcpy(c->w + (tt * c->hv + j) * K, wc + (size_t)t * K, sizeof(double) * K);
            memcpy(c->u + (tt * c->hv + j) * V, uc + (size_t)t * V, sizeof(double) * V);
            c->gcum[tt * c->hv + j] = G[t];
        }
    }
    free(kc);
    free(vc);
    free(wc);
    free(uc);
}

int gdn_oracle_prepare(const double* k, const double* v, const double* g, const double* beta,
                       int64_t T, int N, const int64_t* cu, int hk, int hv, int K, int V, int C,
                       int nthreads, double* w, double* u, double* gcum) {
    int rc = check_geometry(T, N, cu, hk, hv, K, V);
    if (rc) return rc;
    if (C < 1 || C > 1024 || !k || !v || !g || !beta || !w || !u || !gcum) return -1;
    prep_ctx c = {k, v, g, beta, cu, N, hk, hv, K, V, C, w, u, gcum};
    run_items(prep_item, &c, (int64_t)N * hv, nthreads);
    return 0;
}

/* ------------------------------- 3. the chunk map applied to the state and outputs */

/* Scratch for one chunk of one value head (sized for C rows). */
typedef struct {
    double *qc, *kc, *vc, *gc, *bc, *G, *w, *u, *kt;
    double *Mc;  /* [K, K]  gamma I - k_tilde^T w   (the chunk's transition) */
    double *Uc;  /* [K, V]  k_tilde^T u             (the chunk's zero-state write) */
    double *Oq;  /* [C, K]  q_g - attn_i w */
    double *att; /* [C, C]  attn_i */
    double *tmp; /* [K, max(K, V)] */
    double gamma;
} chunk_ws;

static void ws_alloc(chunk_ws* s, int C, int K, int V) {
    const int KV = K > V ? K : V;
    s->qc = (double*)malloc(sizeof(double) * (size_t)C * K);
    s->kc = (double*)malloc(sizeof(double) * (size_t)C * K);
    s->vc = (double*)malloc(sizeof(double) * (size_t)C * V);
    s->gc = (double*)malloc(sizeof(double) * (size_t)C);
    s->bc = (double*)malloc(sizeof(double) * (size_t)C);
    s->G = (double*)malloc(sizeof(double) * (size_t)C);
    s->w = (double*)malloc(sizeof(double) * (size_t)C * K);
    s->u = (double*)malloc(sizeof(double) * (size_t)C * V);
    s->kt = (double*)malloc(sizeof(double) * (size_t)C * K);
    s->Mc = (double*)malloc(sizeof(double) * (size_t)K * K);
    s->Uc = (double*)malloc(sizeof(double) * (size_t)K * V);
    s->Oq = (double*)malloc(sizeof(double) * (size_t)C * K);
    s->att = (double*)malloc(sizeof(double) * (size_t)C * C);
    s->tmp = (double*)malloc(sizeof(double) * (size_t)K * KV);
}

static void ws_free(chunk_ws* s) {
    free(s->qc); free(s->kc); free(s->vc); free(s->gc); free(s->bc); free(s->G);
    free(s->w); free(s->u); free(s->kt); free(s->Mc); free(s->Uc); free(s->Oq);
    free(s->att); free(s->tmp);
}

/* Builds the chunk's affine map from its WY factors ([CP] "Why"):
 *   Mc = gamma I - k_tilde^T w,  Uc = k_tilde^T u,
 *   and, when the queries are present, Oq = q_g - attn_i w and attn_i. */
static void chunk_map(chunk_ws* s, int L, int K, int V, int with_output) {
    gdn_oracle_chunk_factors(L, K, V, s->kc, s->vc, s->gc, s->bc, s->G, NULL, NULL, s->w, s->u,
                             s->kt, &s->gamma);
    for (int a = 0; a < K; ++a)
        for (int b = 0; b < K; ++b) {
            double x = 0.0;
            for (int t = 0; t < L; ++t) x += s->kt[(size_t)t * K + a] * s->w[(size_t)t * K + b];
            s->Mc[(size_t)a * K + b] = (a == b ? s->gamma : 0.0) - x;
        }
    for (int a = 0; a < K; ++a)
        for (int c = 0; c < V; ++c) {
            double x = 0.0;
            for (int t = 0; t < L; ++t) x += s->kt[(size_t)t * K + a] * s->u[(size_t)t * V + c];
            s->Uc[(size_t)a * V + c] = x;
        }
    if (!with_output) return;
    for (int t = 0; t < L; ++t)
        for (int j = 0; j < L; ++j) {
            double x = 0.0;
            if (j <= t) {
                for (int i = 0; i < K; ++i) x += s->qc[(size_t)t * K + i] * s->kc[(size_t)j * K + i];
                x *= exp(s->G[t] - s->G[j]);
            }
            s->att[(size_t)t * L + j] = x;
        }
    for (int t = 0; t < L; ++t)
        for (int i = 0; i < K; ++i) {
            double x = 0.0;
            for (int j = 0; j <= t; ++j) x += s->att[(size_t)t * L + j] * s->w[(size_t)j * K + i];
            s->Oq[(size_t)t * K + i] = exp(s->G[t]) * s->qc[(size_t)t * K + i] - x;
        }
}

/* o = Oq h + attn_i u for the L rows of the chunk starting at token t0; then
 * h <- Mc h + Uc.  h is [K, V]. */
static void chunk_apply(chunk_ws* s, int L, int K, int V, double* h, double* out, int64_t t0,
                        int hv, int j) {
    if (out)
        for (int t = 0; t < L; ++t) {
            double* ot = out + ((size_t)(t0 + t) * hv + j) * V;
            for (int c = 0; c < V; ++c) {
                double x = 0.0;
                for (int i = 0; i < K; ++i) x += s->Oq[(size_t)t * K + i] * h[(size_t)i * V + c];
                for (int jj = 0; jj <= t; ++jj) x += s->att[(size_t)t * L + jj] * s->u[(size_t)jj * V + c];
                ot[c] = x;
            }
        }
    for (int a = 0; a < K; ++a)
        for (int c = 0; c < V; ++c) {
            double x = s->Uc[(size_t)a * V + c];
            for (int b = 0; b < K; ++b) x += s->Mc[(size_t)a * K + b] * h[(size_t)b * V + c];
            s->tmp[(size_t)a * V + c] = x;
        }
    memcpy(h, s->tmp, sizeof(double) * (size_t)K * V);
}

/* Chunk range [c0, c1) of sequence n, in chunks of C tokens. */
static void segment_chunks(const int64_t* cu, int n, int C, int P, int r, int64_t* c0, int64_t* c1) {
    const int64_t Lseq = cu[n + 1] - cu[n];
    const int64_t Nc = (Lseq + C - 1) / C;
    const int64_t base = Nc / P, extra = Nc % P;
    *c0 = r * base + (r < extra ? r : extra);
    *c1 = *c0 + base + (r < extra ? 1 : 0);
}

typedef struct {
    const double *q, *k, *v, *g, *beta, *h0;
    const int64_t* cu;
    int N, hk, hv, K, V, C, P;
    const double* h_in; /* [N*P, hv, K, V] or NULL */
    double *out, *h_final, *M, *U;
} seq_ctx;

/* Runs the chunk map over chunks [c0, c1) of sequence n for value head j, starting from h. */
static void run_chunks(const seq_ctx* c, chunk_ws* s, int n, int j, int64_t c0, int64_t c1,
                       double* h, double* out) {
    const int K = c->K, V = c->V, C = c->C, kh = j / (c->hv / c->hk);
    for (int64_t ch = c0; ch < c1; ++ch) {
        const int64_t t0 = c->cu[n] + ch * C;
        const int L = (int)((c->cu[n + 1] - t0 < C) ? c->cu[n + 1] - t0 : C);
        gather_chunk(c->q, c->k, c->v, c->g, c->beta, t0, L, c->hk, c->hv, kh, j, K, V,
                     out ? s->qc : NULL, s->kc, s->vc, s->gc, s->bc);
        chunk_map(s, L, K, V, out != NULL);
        chunk_apply(s, L, K, V, h, out, t0, c->hv, j);
    }
}

/* The single-pass chunked form ([CP] "Implementation": the single-device path is the same
 * computation reassembled): h <- M_c h + U_c chunk after chunk, emitting outputs. */
static void chunked_item(void* vctx, int64_t item) {
    const seq_ctx* c = (const seq_ctx*)vctx;
    const int n = (int)(item / c->hv), j = (int)(item % c->hv);
    const int K = c->K, V = c->V;
    chunk_ws s;
    ws_alloc(&s, c->C, K, V);
    double* h = (double*)malloc(sizeof(double) * (size_t)K * V);
    for (size_t e = 0; e < (size_t)K * V; ++e)
        h[e] = c->h0 ? c->h0[((size_t)n * c->hv + j) * K * V + e] : 0.0;
    const int64_t Nc = (c->cu[n + 1] - c->cu[n] + c->C - 1) / c->C;
    run_chunks(c, &s, n, j, 0, Nc, h, c->out);
    if (c->h_final) memcpy(c->h_final + ((size_t)n * c->hv + j) * K * V, h, sizeof(double) * K * V);
    free(h);
    ws_free(&s);
}

int gdn_oracle_chunked(const double* q, const double* k, const double* v, const double* g,
                       const double* beta, const double* h0, int64_t T, int N, const int64_t* cu,
                       int hk, int hv, int K, int V, int C, int nthreads, double* out,
                       double* h_final) {
    int rc = check_geometry(T, N, cu, hk, hv, K, V);
    if (rc) return rc;
    if (C < 1 || C > 1024 || !q || !k || !v || !g || !beta || !out) return -1;
    seq_ctx c = {q, k, v, g, beta, h0, cu, N, hk, hv, K, V, C, 1, NULL, out, h_final, NULL, NULL};
    run_items(chunked_item, &c, (int64_t)N * hv, nthreads);
    return 0;
}

/* ------------------------------------------- 4. phase 1: segment summaries */

/* Zero-state pass over one segment carrying the composed transition ([CP] "Implementation",
 * phase 1): M starts at I and U (the state) at 0; per chunk
 *     U <- gamma U + k_tilde^T (u - w U)          (the chunk map applied to the state)
 *     M <- gamma M - k_tilde^T (w M)              (low-rank composition)
 * so that at the segment's end h_out = M_r h_in + U_r for any incoming h_in. */
static void summary_item(void* vctx, int64_t item) {
    const seq_ctx* c = (const seq_ctx*)vctx;
    const int P = c->P, hv = c->hv, K = c->K, V = c->V, C = c->C;
    const int r = (int)(item % P);
    const int j = (int)((item / P) % hv);
    const int n = (int)(item / ((int64_t)P * hv));
    const int kh = j / (hv / c->hk);
    int64_t c0, c1;
    segment_chunks(c->cu, n, C, P, r, &c0, &c1);
    chunk_ws s;
    ws_alloc(&s, C, K, V);
    double* M = c->M + (((size_t)n * P + r) * hv + j) * K * K;
    double* U = c->U + (((size_t)n * P + r) * hv + j) * K * V;
    double* wM = (double*)malloc(sizeof(double) * (size_t)C * (K > V ? K : V));
    for (int a = 0; a < K; ++a)
        for (int b = 0; b < K; ++b) M[(size_t)a * K + b] = (a == b) ? 1.0 : 0.0;
    memset(U, 0, sizeof(double) * (size_t)K * V);
    for (int64_t ch = c0; ch < c1; ++ch) {
        const int64_t t0 = c->cu[n] + ch * C;
        const int L = (int)((c->cu[n + 1] - t0 < C) ? c->cu[n + 1] - t0 : C);
        gather_chunk(NULL, c->k, c->v, c->g, c->beta, t0, L, c->hk, hv, kh, j, K, V, NULL, s.kc,
                     s.vc, s.gc, s.bc);
        gdn_oracle_chunk_factors(L, K, V, s.kc, s.vc, s.gc, s.bc, s.G, NULL, NULL, s.w, s.u, s.kt,
                                 &s.gamma);
        /* U <- gamma U + k_tilde^T (u - w U) */
        for (int t = 0; t < L; ++t)
            for (int cc = 0; cc < V; ++cc) {
                double x = 0.0;
                for (int i = 0; i < K; ++i) x += s.w[(size_t)t * K + i] * U[(size_t)i * V + cc];
                wM[(size_t)t * V + cc] = s.u[(size_t)t * V + cc] - x;
            }
        for (int a = 0; a < K; ++a)
            for (int cc = 0; cc < V; ++cc) {
                double x = 0.0;
                for (int t = 0; t < L; ++t) x += s.kt[(size_t)t * K + a] * wM[(size_t)t * V + cc];
                U[(size_t)a * V + cc] = s.gamma * U[(size_t)a * V + cc] + x;
            }
        /* M <- gamma M - k_tilde^T (w M) */
        for (int t = 0; t < L; ++t)
            for (int b = 0; b < K; ++b) {
                double x = 0.0;
                for (int i = 0; i < K; ++i) x += s.w[(size_t)t * K + i] * M[(size_t)i * K + b];
                wM[(size_t)t * K + b] = x;
            }
        for (int a = 0; a < K; ++a)
            for (int b = 0; b < K; ++b) {
                double x = 0.0;
                for (int t = 0; t < L; ++t) x += s.kt[(size_t)t * K + a] * wM[(size_t)t * K + b];
                M[(size_t)a * K + b] = s.gamma * M[(size_t)a * K + b] - x;
            }
    }
    free(wM);
    ws_free(&s);
}

/* M [N*P, hv, K, K], U [N*P, hv, K, V]. */
int gdn_oracle_summary(const double* k, const double* v, const double* g, const double* beta,
                       int64_t T, int N, const int64_t* cu, int hk, int hv, int K, int V, int C,
                       int P, int nthreads, double* M, double* U) {
    int rc = check_geometry(T, N, cu, hk, hv, K, V);
    if (rc) return rc;
    if (C < 1 || C > 1024 || P < 1 || !k || !v || !g || !beta || !M || !U) return -1;
    seq_ctx c = {NULL, k, v, g, beta, NULL, cu, N, hk, hv, K, V, C, P, NULL, NULL, NULL, M, U};
    run_items(summary_item, &c, (int64_t)N * hv * P, nthreads);
    return 0;
}

/* Dense transition of tokens [t0, t1) for value head j: the product of the per-token maps
 * exp(g_t) (I - beta_t k_t k_t^T), later tokens on the left, built token by token.  Used only
 * to check the low-rank M_r.  k is [T, hk, K]; out M is [K, K]. */
int gdn_oracle_dense_transition(const double* k, const double* g, const double* beta, int64_t t0,
                                int64_t t1, int hk, int hv, int K, int j, double* M) {
    if (!k || !g || !beta || !M || K < 1 || j < 0 || j >= hv || hv % hk) return -1;
    const int kh = j / (hv / hk);
    double* tmp = (double*)malloc(sizeof(double) * (size_t)K * K);
    for (int a = 0; a < K; ++a)
        for (int b = 0; b < K; ++b) M[(size_t)a * K + b] = (a == b) ? 1.0 : 0.0;
    for (int64_t t = t0; t < t1; ++t) {
        const double* kt = k + ((size_t)t * hk + kh) * K;
        const double alpha = exp(g[(size_t)t * hv + j]), b = beta[(size_t)t * hv + j];
        for (int a = 0; a < K; ++a)
            for (int c = 0; c < K; ++c) {
                double x = 0.0;
                for (int i = 0; i < K; ++i) {
                    const double Tai = alpha * ((a == i ? 1.0 : 0.0) - b * kt[a] * kt[i]);
                    x += Tai * M[(size_t)i * K + c];
                }
                tmp[(size_t)a * K + c] = x;
            }
        memcpy(M, tmp, sizeof(double) * (size_t)K * K);
    }
    free(tmp);
    return 0;
}

/* --------------------------------------------- 5. phase 2: exclusive scan */

/* h_in[n, 0] = h0[n];  h_in[n, r+1] = M[n, r] h_in[n, r] + U[n, r];
 * h_final[n] = M[n, P-1] h_in[n, P-1] + U[n, P-1]  ([CP] "Implementation", phase 2, and
 * "Why": affine maps compose, (M2, U2) o (M1, U1) = (M2 M1, M2 U1 + U2)). */
int gdn_oracle_scan(const double* M, const double* U, const double* h0, int N, int P, int hv,
                    int K, int V, double* h_in, double* h_final) {
    if (!M || !U || !h_in || N < 1 || P < 1 || hv < 1 || K < 1 || V < 1) return -1;
    const size_t KV = (size_t)K * V, KK = (size_t)K * K;
    double* h = (double*)malloc(sizeof(double) * KV);
    double* t = (double*)malloc(sizeof(double) * KV);
    for (int n = 0; n < N; ++n)
        for (int j = 0; j < hv; ++j) {
            for (size_t e = 0; e < KV; ++e) h[e] = h0 ? h0[((size_t)n * hv + j) * KV + e] : 0.0;
            for (int r = 0; r < P; ++r) {
                const size_t s = ((size_t)n * P + r) * hv + j;
                memcpy(h_in + s * KV, h, sizeof(double) * KV);
                const double* Mr = M + s * KK;
                const double* Ur = U + s * KV;
                for (int a = 0; a < K; ++a)
                    for (int c = 0; c < V; ++c) {
                        double x = Ur[(size_t)a * V + c];
                        for (int b = 0; b < K; ++b) x += Mr[(size_t)a * K + b] * h[(size_t)b * V + c];
                        t[(size_t)a * V + c] = x;
                    }
                memcpy(h, t, sizeof(double) * KV);
            }
            if (h_final) memcpy(h_final + ((size_t)n * hv + j) * KV, h, sizeof(double) * KV);
        }
    free(h);
    free(t);
    return 0;
}

/* ------------------------------------------------- 6. phase 3: re-emit */

static void emit_item(void* vctx, int64_t item) {
    const seq_ctx* c = (const seq_ctx*)vctx;
    const int P = c->P, hv = c->hv, K = c->K, V = c->V;
    const int r = (int)(item % P);
    const int j = (int)((item / P) % hv);
    const int n = (int)(item / ((int64_t)P * hv));
    int64_t c0, c1;
    segment_chunks(c->cu, n, c->C, P, r, &c0, &c1);
    chunk_ws s;
    ws_alloc(&s, c->C, K, V);
    double* h = (double*)malloc(sizeof(double) * (size_t)K * V);
    memcpy(h, c->h_in + (((size_t)n * P + r) * hv + j) * K * V, sizeof(double) * (size_t)K * V);
    run_chunks(c, &s, n, j, c0, c1, h, c->out);
    free(h);
    ws_free(&s);
}

/* Phase 3 alone: from h_in [N*P, hv, K, V] re-run every segment's chunks, emitting out. */
int gdn_oracle_emit(const double* q, const double* k, const double* v, const double* g,
                    const double* beta, const double* h_in, int64_t T, int N, const int64_t* cu,
                    int hk, int hv, int K, int V, int C, int P, int nthreads, double* out) {
    int rc = check_geometry(T, N, cu, hk, hv, K, V);
    if (rc) return rc;
    if (C < 1 || C > 1024 || P < 1 || !q || !k || !v || !g || !beta || !h_in || !out) return -1;
    seq_ctx c = {q, k, v, g, beta, NULL, cu, N, hk, hv, K, V, C, P, h_in, out, NULL, NULL, NULL};
    run_items(emit_item, &c, (int64_t)N * hv * P, nthreads);
    return 0;
}

/* The three phases end to end ([CP] "Implementation"): summaries, scan, re-emit. */
int gdn_oracle_segmented(const double* q, const double* k, const double* v, const double* g,
                         const double* beta, const double* h0, int64_t T, int N, const int64_t* cu,
                         int hk, int hv, int K, int V, int C, int P, int nthreads, double* out,
                         double* h_final) {
    int rc = check_geometry(T, N, cu, hk, hv, K, V);
    if (rc) return rc;
    if (C < 1 || C > 1024 || P < 1) return -1;
    const size_t S = (size_t)N * P * hv;
    double* M = (double*)malloc(sizeof(double) * S * K * K);
    double* U = (double*)malloc(sizeof(double) * S * K * V);
    double* h_in = (double*)malloc(sizeof(double) * S * K * V);
    if (!M || !U || !h_in) {
        free(M); free(U); free(h_in);
        return -5;
    }
    rc = gdn_oracle_summary(k, v, g, beta, T, N, cu, hk, hv, K, V, C, P, nthreads, M, U);
    if (!rc) rc = gdn_oracle_scan(M, U, h0, N, P, hv, K, V, h_in, h_final);
    if (!rc) rc = gdn_oracle_emit(q, k, v, g, beta, h_in, T, N, cu, hk, hv, K, V, C, P, nthreads, out);
    free(M);
    free(U);
    free(h_in);
    return rc;
}

/* --------------------------------------- 7. reverse mode of the per-token recurrence */

/* Gradients of L = <dout, out> + <dh_final, h_final> with respect to q, k, v, g, beta and
 * h0, by reverse mode through the token recurrence of section 1 (the plain definition; the
 * pages state no backward formulas, and this one follows from the recurrence alone).  Per
 * token, with h_prev the state before it, h its state after, F = dL/dh (the gradient from
 * later tokens plus q dout^T), alpha = exp(g), P = h_prev^T k, delta = beta (v - alpha P):
 *     dq = h dout                    dd = F^T k (dL/d delta)
 *     dv = beta dd                   dbeta = dd . (v - alpha P)
 *     dk = F delta - alpha beta h_prev dd
 *     dg = alpha (<F, h_prev> - beta dd . P)
 *     dh_prev = alpha (F - beta k dd^T)
 * States are recomputed from a checkpoint every 64 tokens.  One work item = (sequence n,
 * key head kh): its value heads run in turn, so dq and dk of a key head (summed over the
 * value heads that read it) have a single writer.
 * Layouts: dout [T, hv, V]; dh_final, dh0 [N, hv, K, V] (dh_final may be NULL = zeros);
 * dq, dk [T, hk, K]; dv [T, hv, V]; dg, dbeta [T, hv]; dh0 may be NULL. */
typedef struct {
    const double *q, *k, *v, *g, *beta, *h0, *dout, *dhf;
    const int64_t* cu;
    int N, hk, hv, K, V;
    double *dq, *dk, *dv, *dg, *dbeta, *dh0;
} bwd_ctx;

enum { kBwdBlock = 64 };

/* one token of the recurrence: h <- alpha h + k delta^T (delta, P returned) */
static void bwd_step(int K, int V, double* h, const double* kt, const double* vt, double alpha,
                     double b, double* P, double* delta) {
    for (int c = 0; c < V; ++c) P[c] = 0.0;
    for (int i = 0; i < K; ++i)
        for (int c = 0; c < V; ++c) P[c] += h[(size_t)i * V + c] * kt[i];
    for (int c = 0; c < V; ++c) delta[c] = b * (vt[c] - alpha * P[c]);
    for (int i = 0; i < K; ++i)
        for (int c = 0; c < V; ++c) h[(size_t)i * V + c] = alpha * h[(size_t)i * V + c] + kt[i] * delta[c];
}

static void bwd_item(void* vctx, int64_t item) {
    const bwd_ctx* c = (const bwd_ctx*)vctx;
    const int K = c->K, V = c->V, hk = c->hk, hv = c->hv, grp = hv / hk;
    const int kh = (int)(item % hk);
    const int n = (int)(item / hk);
    const int64_t t0 = c->cu[n], t1 = c->cu[n + 1], L = t1 - t0;
    const int64_t nblk = (L + kBwdBlock - 1) / kBwdBlock;
    const size_t KV = (size_t)K * V;
    double* ck = (double*)malloc(sizeof(double) * KV * (size_t)(nblk > 0 ? nblk : 1));
    double* hs = (double*)malloc(sizeof(double) * KV * (kBwdBlock + 1));
    double* F = (double*)malloc(sizeof(double) * KV);
    double* P = (double*)malloc(sizeof(double) * V);
    double* delta = (double*)malloc(sizeof(double) * V);
    double* dd = (double*)malloc(sizeof(double) * V);
    for (int64_t t = t0; t < t1; ++t)
        for (int i = 0; i < K; ++i) {
            c->dq[((size_t)t * hk + kh) * K + i] = 0.0;
            c->dk[((size_t)t * hk + kh) * K + i] = 0.0;
        }
    for (int jj = 0; jj < grp; ++jj) {
        const int j = kh * grp + jj;
        /* forward: the state entering every block */
        double* h = hs;
        for (size_t e = 0; e < KV; ++e) h[e] = c->h0 ? c->h0[((size_t)n * hv + j) * KV + e] : 0.0;
        for (int64_t t = t0; t < t1; ++t) {
            if ((t - t0) % kBwdBlock == 0) memcpy(ck + (size_t)((t - t0) / kBwdBlock) * KV, h, sizeof(double) * KV);
            bwd_step(K, V, h, c->k + ((size_t)t * hk + kh) * K, c->v + ((size_t)t * hv + j) * V,
                     exp(c->g[(size_t)t * hv + j]), c->beta[(size_t)t * hv + j], P, delta);
        }
        /* backward, block by block from the end */
        for (size_t e = 0; e < KV; ++e) F[e] = c->dhf ? c->dhf[((size_t)n * hv + j) * KV + e] : 0.0;
        for (int64_t bi = nblk - 1; bi >= 0; --bi) {
            const int64_t b0 = t0 + bi * kBwdBlock;
            const int64_t b1 = (b0 + kBwdBlock < t1) ? b0 + kBwdBlock : t1;
            memcpy(hs, ck + (size_t)bi * KV, sizeof(double) * KV);
            for (int64_t t = b0; t < b1; ++t) {  /* hs[i] = state before token b0 + i */
                memcpy(hs + (size_t)(t - b0 + 1) * KV, hs + (size_t)(t - b0) * KV, sizeof(double) * KV);
                bwd_step(K, V, hs + (size_t)(t - b0 + 1) * KV, c->k + ((size_t)t * hk + kh) * K,
                         c->v + ((size_t)t * hv + j) * V, exp(c->g[(size_t)t * hv + j]),
                         c->beta[(size_t)t * hv + j], P, delta);
            }
            for (int64_t t = b1 - 1; t >= b0; --t) {
                const double* hp = hs + (size_t)(t - b0) * KV;      /* before token t */
                const double* ha = hs + (size_t)(t - b0 + 1) * KV;  /* after token t */
                const double* kt = c->k + ((size_t)t * hk + kh) * K;
                const double* qt = c->q + ((size_t)t * hk + kh) * K;
                const double* vt = c->v + ((size_t)t * hv + j) * V;
                const double* ot = c->dout + ((size_t)t * hv + j) * V;
                const double alpha = exp(c->g[(size_t)t * hv + j]);
                const double b = c->beta[(size_t)t * hv + j];
                double* dqt = c->dq + ((size_t)t * hk + kh) * K;
                double* dkt = c->dk + ((size_t)t * hk + kh) * K;
                /* F = dL/dh_t: the later tokens' gradient plus this token's output */
                for (int i = 0; i < K; ++i)
                    for (int cc = 0; cc < V; ++cc) F[(size_t)i * V + cc] += qt[i] * ot[cc];
                /* dq = h_t dout */
                for (int i = 0; i < K; ++i) {
                    double s = 0.0;
                    for (int cc = 0; cc < V; ++cc) s += ha[(size_t)i * V + cc] * ot[cc];
                    dqt[i] += s;
                }
                /* P = h_prev^T k, delta, dd = F^T k */
                for (int cc = 0; cc < V; ++cc) { P[cc] = 0.0; dd[cc] = 0.0; }
                for (int i = 0; i < K; ++i)
                    for (int cc = 0; cc < V; ++cc) {
                        P[cc] += hp[(size_t)i * V + cc] * kt[i];
                        dd[cc] += F[(size_t)i * V + cc] * kt[i];
                    }
                double dbeta = 0.0, dPd = 0.0, Fh = 0.0;
                for (int cc = 0; cc < V; ++cc) {
                    const double r = vt[cc] - alpha * P[cc];
                    delta[cc] = b * r;
                    c->dv[((size_t)t * hv + j) * V + cc] = b * dd[cc];
                    dbeta += dd[cc] * r;
                    dPd += dd[cc] * P[cc];
                }
                for (size_t e = 0; e < KV; ++e) Fh += F[e] * hp[e];
                c->dbeta[(size_t)t * hv + j] = dbeta;
                c->dg[(size_t)t * hv + j] = alpha * (Fh - b * dPd);
                /* dk = F delta - alpha beta h_prev dd */
                for (int i = 0; i < K; ++i) {
                    double s = 0.0;
                    for (int cc = 0; cc < V; ++cc)
                        s += F[(size_t)i * V + cc] * delta[cc] - alpha * b * hp[(size_t)i * V + cc] * dd[cc];
                    dkt[i] += s;
                }
                /* dh_prev = alpha (F - beta k dd^T) */
                for (int i = 0; i < K; ++i)
                    for (int cc = 0; cc < V; ++cc)
                        F[(size_t)i * V + cc] = alpha * (F[(size_t)i * V + cc] - b * kt[i] * dd[cc]);
            }
        }
        if (c->dh0) memcpy(c->dh0 + ((size_t)n * hv + j) * KV, F, sizeof(double) * KV);
    }
    free(ck);
    free(hs);
    free(F);
    free(P);
    free(delta);
    free(dd);
}

int gdn_oracle_token_backward(const double* q, const double* k, const double* v, const double* g,
                              const double* beta, const double* h0, const double* dout,
                              const double* dh_final, int64_t T, int N, const int64_t* cu,
                              int hk, int hv, int K, int V, int nthreads, double* dq, double* dk,
                              double* dv, double* dg, double* dbeta, double* dh0) {
    int rc = check_geometry(T, N, cu, hk, hv, K, V);
    if (rc) return rc;
    if (!q || !k || !v || !g || !beta || !dout || !dq || !dk || !dv || !dg || !dbeta) return -1;
    bwd_ctx c = {q, k, v, g, beta, h0, dout, dh_final, cu, N, hk, hv, K, V,
                 dq, dk, dv, dg, dbeta, dh0};
    run_items(bwd_item, &c, (int64_t)N * hk, nthreads);
    return 0;
}
