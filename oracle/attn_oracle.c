/*
 * attn_oracle.c -- plain float64 CPU oracle for exact softmax attention,
 * forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load this file's library.  It shares no code,
 * header or constant with the CUDA path, and the CUDA path never calls it.
 *
 * What it computes (per head, S query rows, S key rows, head dim d):
 * the textbook attention function softmax(scale * Q K^T, mask) V and its
 * gradient with respect to Q, K and V for the scalar loss sum(dO * O).
 * The DASH pages state that the deterministic backward reaches exactly this
 * gradient and only changes the order in which the dQ partial sums are added
 * ("DASH: Deterministic Attention Scheduling for High-throughput Reproducible
 * LLM Training", technical summary section 1 (problem statement) and the
 * arXiv abstract).  So the oracle is the definition written out, step by step:
 *
 *   1. s_rc   = scale * sum_k q_rk k_ck               (unmasked pairs only)
 *   2. m_r    = max_c s_rc
 *   3. LSE_r  = m_r + ln sum_c exp(s_rc - m_r)        (natural log)
 *   4. P_rc   = exp(s_rc - LSE_r), 0 where masked
 *   5. O_r    = sum_c P_rc v_c
 *   6. D_r    = sum_k dO_rk O_rk
 *   7. dV_c   = sum_r P_rc dO_r
 *   8. dP_rc  = sum_k dO_rk v_ck
 *   9. dS_rc  = P_rc (dP_rc - D_r)
 *  10. dQ_r   = scale * sum_c dS_rc k_c
 *  11. dK_c   = scale * sum_r dS_rc q_r
 *
 * Masks: FULL (nothing masked) or CAUSAL (key c masked for query r when
 * c > r; query and key sequences have the same length, so the diagonal is
 * kept and no row is empty).  Either can be combined with a block mask: a
 * table of N x N flags over 128 x 128 tiles (row = query tile, column = key
 * tile), where a zero flag masks every key of that key tile for every query
 * of that query tile (the block-sparse masks the DASH pages name as future
 * work, technical summary section 5).  A query row with every key masked
 * has no softmax: its LSE is -infinity, its O, D and dQ are zero, and it
 * adds nothing to dK and dV.
 *
 * Organisation: steps 1-6 and 8-10 are computed per query row r (everything
 * they need lives in row r); steps 7 and 11 are sums over query rows for one
 * key row c, so they are computed per key row, recomputing s_rc, P_rc, dP_rc
 * and dS_rc from their definitions with the LSE_r and D_r of step 3 and 6.
 * Every output element is produced by exactly one thread, summing its terms in
 * ascending index order, so the result does not depend on the thread count.
 *
 * Diagnostic mode (oracle_attn_bwd_given): O and LSE are taken from the
 * caller instead of steps 1-5, to separate backward errors from forward ones.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define BLOCK_TILE 128 /* rows per tile of a block mask */

typedef struct {
    int S, d, causal;
    const unsigned char *tiles; /* block mask [N][N] (N = S / BLOCK_TILE), or NULL */
    int ntiles;
    double scale;
    const double *q, *k, *v, *dout; /* [S][d] each, this head */
    const double *o_in, *lse_in;    /* diagnostic mode: given O [S][d], LSE [S] */
    double *o, *lse, *D;            /* outputs: O [S][d], LSE [S], D [S] */
    double *dq, *dk, *dv;           /* outputs: [S][d] each */
} head_job;

typedef struct {
    head_job *job;
    int tid, nthreads;
    int phase;       /* 1: query rows, 2: key rows */
    const int *rows; /* rows to process (NULL: all S rows) */
    int nrows;
} worker_arg;

static int is_masked(const head_job *h, int r, int c)
{
    if (h->causal && c > r) return 1;
    return h->tiles != NULL && h->tiles[(size_t)(r / BLOCK_TILE) * h->ntiles + c / BLOCK_TILE] == 0;
}

static double dot(const double *a, const double *b, int d)
{
    double acc = 0.0;
    for (int x = 0; x < d; ++x) acc += a[x] * b[x];
    return acc;
}

/* Steps 1-6 and 8-10 for query row r.  s and dp are scratch rows of length S. */
static void query_row(const head_job *h, int r, double *s, double *p)
{
    const int S = h->S, d = h->d;
    const double *q_r = h->q + (size_t)r * d;
    const double *do_r = h->dout + (size_t)r * d;
    double lse, D;
    double *o_r = h->o + (size_t)r * d;

    if (h->o_in == NULL) {
        /* 1. scores of the unmasked keys */
        double m = -INFINITY;
        for (int c = 0; c < S; ++c) {
            if (is_masked(h, r, c)) continue;
            s[c] = h->scale * dot(q_r, h->k + (size_t)c * d, d);
            /* 2. running maximum */
            if (s[c] > m) m = s[c];
        }
        /* 3. log-sum-exp */
        double sum = 0.0;
        for (int c = 0; c < S; ++c)
            if (!is_masked(h, r, c)) sum += exp(s[c] - m);
        lse = (sum > 0.0) ? m + log(sum) : -INFINITY; /* no visible key: no softmax */
        /* 4. probabilities */
        for (int c = 0; c < S; ++c)
            p[c] = is_masked(h, r, c) ? 0.0 : exp(s[c] - lse);
        /* 5. output row */
        for (int x = 0; x < d; ++x) o_r[x] = 0.0;
        for (int c = 0; c < S; ++c) {
            if (p[c] == 0.0) continue;
            const double *v_c = h->v + (size_t)c * d;
            for (int x = 0; x < d; ++x) o_r[x] += p[c] * v_c[x];
        }
    } else {
        /* diagnostic mode: O and LSE given; P from the given LSE */
        lse = h->lse_in[r];
        for (int c = 0; c < S; ++c)
            p[c] = is_masked(h, r, c)
                       ? 0.0
                       : exp(h->scale * dot(q_r, h->k + (size_t)c * d, d) - lse);
        memcpy(o_r, h->o_in + (size_t)r * d, sizeof(double) * (size_t)d);
    }
    h->lse[r] = lse;

    /* 6. D_r = dO_r . O_r */
    D = dot(do_r, o_r, d);
    h->D[r] = D;

    /* 8-10. dP, dS and dQ for row r (s is reused to hold dS) */
    double *dq_r = h->dq + (size_t)r * d;
    for (int x = 0; x < d; ++x) dq_r[x] = 0.0;
    for (int c = 0; c < S; ++c) {
        if (is_masked(h, r, c)) continue;
        const double dp = dot(do_r, h->v + (size_t)c * d, d); /* 8 */
        const double ds = p[c] * (dp - D);                    /* 9 */
        const double *k_c = h->k + (size_t)c * d;
        for (int x = 0; x < d; ++x) dq_r[x] += ds * k_c[x];   /* 10 (sum) */
    }
    for (int x = 0; x < d; ++x) dq_r[x] *= h->scale;          /* 10 (scale) */
}

/* Steps 7 and 11 for key row c, using LSE_r and D_r of every query row. */
static void key_row(const head_job *h, int c)
{
    const int S = h->S, d = h->d;
    const double *k_c = h->k + (size_t)c * d;
    const double *v_c = h->v + (size_t)c * d;
    double *dk_c = h->dk + (size_t)c * d;
    double *dv_c = h->dv + (size_t)c * d;
    for (int x = 0; x < d; ++x) { dk_c[x] = 0.0; dv_c[x] = 0.0; }
    for (int r = 0; r < S; ++r) {
        if (is_masked(h, r, c)) continue;
        const double *q_r = h->q + (size_t)r * d;
        const double *do_r = h->dout + (size_t)r * d;
        const double s = h->scale * dot(q_r, k_c, d);   /* 1 */
        const double p = exp(s - h->lse[r]);            /* 4 */
        const double dp = dot(do_r, v_c, d);            /* 8 */
        const double ds = p * (dp - h->D[r]);           /* 9 */
        for (int x = 0; x < d; ++x) {
            dv_c[x] += p * do_r[x];                     /* 7 */
            dk_c[x] += ds * q_r[x];                     /* 11 (sum) */
        }
    }
    for (int x = 0; x < d; ++x) dk_c[x] *= h->scale;   /* 11 (scale) */
}

static void *worker(void *argp)
{
    worker_arg *a = (worker_arg *)argp;
    head_job *h = a->job;
    const int n = a->rows ? a->nrows : h->S;
    if (a->phase == 1) {
        double *s = (double *)malloc(sizeof(double) * (size_t)h->S);
        double *p = (double *)malloc(sizeof(double) * (size_t)h->S);
        if (s == NULL || p == NULL) { free(s); free(p); return (void *)1; }
        for (int x = a->tid; x < n; x += a->nthreads)
            query_row(h, a->rows ? a->rows[x] : x, s, p);
        free(s);
        free(p);
    } else {
        for (int x = a->tid; x < n; x += a->nthreads) key_row(h, a->rows ? a->rows[x] : x);
    }
    return NULL;
}

static int run_phase_rows(head_job *h, int phase, const int *rows, int nrows, int nthreads)
{
    pthread_t th[256];
    worker_arg args[256];
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    int failed = 0;
    for (int t = 0; t < nthreads; ++t) {
        args[t].job = h;
        args[t].tid = t;
        args[t].nthreads = nthreads;
        args[t].phase = phase;
        args[t].rows = rows;
        args[t].nrows = nrows;
        if (t > 0 && pthread_create(&th[t], NULL, worker, &args[t]) != 0) {
            /* fall back: run this share on the calling thread */
            if (worker(&args[t]) != NULL) failed = 1;
            th[t] = 0;
        }
    }
    if (worker(&args[0]) != NULL) failed = 1;
    for (int t = 1; t < nthreads; ++t) {
        void *ret = NULL;
        if (th[t] != 0) {
            pthread_join(th[t], &ret);
            if (ret != NULL) failed = 1;
        }
    }
    return failed ? -1 : 0;
}

static int run_phase(head_job *h, int phase, int nthreads)
{
    return run_phase_rows(h, phase, NULL, 0, nthreads);
}

static int run_heads(int BH, int S, int d, double scale, int causal,
                     const unsigned char *tiles,
                     const double *q, const double *k, const double *v,
                     const double *dout, const double *o_in, const double *lse_in,
                     double *o, double *lse, double *D,
                     double *dq, double *dk, double *dv, int nthreads)
{
    if (BH < 0 || S < 0 || d <= 0) return -2;
    if (tiles != NULL && (S % BLOCK_TILE) != 0) return -2;
    for (int b = 0; b < BH; ++b) {
        const size_t off = (size_t)b * (size_t)S * (size_t)d;
        head_job h;
        h.S = S; h.d = d; h.causal = causal; h.scale = scale;
        h.tiles = tiles; h.ntiles = S / BLOCK_TILE;
        h.q = q + off; h.k = k + off; h.v = v + off; h.dout = dout + off;
        h.o_in = o_in ? o_in + off : NULL;
        h.lse_in = lse_in ? lse_in + (size_t)b * S : NULL;
        h.o = o + off; h.lse = lse + (size_t)b * S; h.D = D + (size_t)b * S;
        h.dq = dq + off; h.dk = dk + off; h.dv = dv + off;
        if (run_phase(&h, 1, nthreads) != 0) return -1;
        if (run_phase(&h, 2, nthreads) != 0) return -1;
    }
    return 0;
}

/* Full forward + backward for BH independent heads, inputs [BH][S][d]. */
int oracle_attn_fwd_bwd(int BH, int S, int d, double scale, int causal,
                        const double *q, const double *k, const double *v,
                        const double *dout,
                        double *o, double *lse, double *D,
                        double *dq, double *dk, double *dv, int nthreads)
{
    return run_heads(BH, S, d, scale, causal, NULL, q, k, v, dout, NULL, NULL,
                     o, lse, D, dq, dk, dv, nthreads);
}

/* The same with a block mask: tiles [N][N], N = S / 128, row = query tile,
 * column = key tile, zero = masked (combined with `causal`).               */
int oracle_attn_fwd_bwd_block(int BH, int S, int d, double scale, int causal,
                              const unsigned char *tiles,
                              const double *q, const double *k, const double *v,
                              const double *dout,
                              double *o, double *lse, double *D,
                              double *dq, double *dk, double *dv, int nthreads)
{
    if (tiles == NULL) return -2;
    return run_heads(BH, S, d, scale, causal, tiles, q, k, v, dout, NULL, NULL,
                     o, lse, D, dq, dk, dv, nthreads);
}

/* Diagnostic backward with O [BH][S][d] and LSE [BH][S] supplied by the
 * caller (for instance the values a GPU forward produced).  o_out receives a
 * copy of o_in, lse_out a copy of lse_in. */
int oracle_attn_bwd_given(int BH, int S, int d, double scale, int causal,
                          const double *q, const double *k, const double *v,
                          const double *o_in, const double *lse_in,
                          const double *dout,
                          double *o_out, double *lse_out, double *D,
                          double *dq, double *dk, double *dv, int nthreads)
{
    if (o_in == NULL || lse_in == NULL) return -2;
    return run_heads(BH, S, d, scale, causal, NULL, q, k, v, dout, o_in, lse_in,
                     o_out, lse_out, D, dq, dk, dv, nthreads);
}

/* Selected rows of one head [S][d].  Query rows `qrows` get steps 1-6 and
 * 8-10 (O, LSE, D, dQ); key rows `krows` get steps 7 and 11 (dK, dV).  The
 * key rows need LSE_r and D_r of every query row: pass them in lse_all /
 * D_all (as a whole-head run produced them), or NULL to compute them here
 * first (a whole-head query pass).  Outputs are [nq][d], [nq], [nq], [nq][d],
 * [nk][d], [nk][d].                                                         */
int oracle_attn_rows(int S, int d, double scale, int causal,
                     const double *q, const double *k, const double *v,
                     const double *dout, const double *lse_all, const double *D_all,
                     const int *qrows, int nq, const int *krows, int nk,
                     double *o_rows, double *lse_rows, double *D_rows, double *dq_rows,
                     double *dk_rows, double *dv_rows, int nthreads)
{
    if (S <= 0 || d <= 0 || nq < 0 || nk < 0) return -2;
    for (int x = 0; x < nq; ++x) if (qrows[x] < 0 || qrows[x] >= S) return -2;
    for (int x = 0; x < nk; ++x) if (krows[x] < 0 || krows[x] >= S) return -2;
    const size_t Sd = (size_t)S * (size_t)d;
    double *o = (double *)calloc(Sd, sizeof(double));
    double *dq = (double *)calloc(Sd, sizeof(double));
    double *dk = (double *)calloc(Sd, sizeof(double));
    double *dv = (double *)calloc(Sd, sizeof(double));
    double *lse = (double *)calloc((size_t)S, sizeof(double));
    double *D = (double *)calloc((size_t)S, sizeof(double));
    int rc = 0;
    head_job h;
    if (!o || !dq || !dk || !dv || !lse || !D) { rc = -1; goto done; }
    h.S = S; h.d = d; h.causal = causal; h.scale = scale;
    h.tiles = NULL; h.ntiles = 0;
    h.q = q; h.k = k; h.v = v; h.dout = dout;
    h.o_in = NULL; h.lse_in = NULL;
    h.o = o; h.lse = lse; h.D = D; h.dq = dq; h.dk = dk; h.dv = dv;
    if (nk > 0) {
        if (lse_all != NULL && D_all != NULL) {
            memcpy(lse, lse_all, sizeof(double) * (size_t)S);
            memcpy(D, D_all, sizeof(double) * (size_t)S);
        } else if (run_phase(&h, 1, nthreads) != 0) { rc = -1; goto done; }
    }
    if (nq > 0 && run_phase_rows(&h, 1, qrows, nq, nthreads) != 0) { rc = -1; goto done; }
    if (nk > 0 && run_phase_rows(&h, 2, krows, nk, nthreads) != 0) { rc = -1; goto done; }
    for (int x = 0; x < nq; ++x) {
        const int r = qrows[x];
        memcpy(o_rows + (size_t)x * d, o + (size_t)r * d, sizeof(double) * (size_t)d);
        memcpy(dq_rows + (size_t)x * d, dq + (size_t)r * d, sizeof(double) * (size_t)d);
        lse_rows[x] = lse[r];
        D_rows[x] = D[r];
    }
    for (int x = 0; x < nk; ++x) {
        const int c = krows[x];
        memcpy(dk_rows + (size_t)x * d, dk + (size_t)c * d, sizeof(double) * (size_t)d);
        memcpy(dv_rows + (size_t)x * d, dv + (size_t)c * d, sizeof(double) * (size_t)d);
    }
done:
    free(o); free(dq); free(dk); free(dv); free(lse); free(D);
    return rc;
}
