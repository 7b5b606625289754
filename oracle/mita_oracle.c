/*
 * MiTA attention forward -- the ORACLE.
 *
 * This file is test infrastructure. Only the test suite, the smoke check and
 * the CPU-baseline leg of the benchmark load it; the product path never does.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * Plain, slow, fp64, one (batch, head) per thread. Every step follows the
 * method as it is stated in "MiTA Attention: Efficient Fast-Weight Scaling via
 * a Mixture of Top-k Activations" (gist.science technical summaries, Arabic
 * edition section 2 "Methodology / mechanism details", Dutch edition
 * "Technische samenvatting / Kernconcepten / Wiskundige Formulering", Hindi
 * edition section 2), in the order the summaries give:
 *
 *   1. landmark queries Qt = adaptive average pooling of Q      (ar s2, nl Kernconcepten 1)
 *   2. shared expert     Vt = softmax(scale * Qt K^T) V          (ar s2: Vt = Atten(Qt, K, V))
 *   3. expert index sets I_i = top-k of K^T qt_i                 (ar s2, nl Kernconcepten 3)
 *   4. routing           e_1(q)..e_s(q)                          (nl Wiskundige Formulering)
 *   5. output            softmax over K* = [Qt, K_(e1), .., K_(es)],
 *                        V* = [Vt, V_(e1), .., V_(es)]           (nl Wiskundige Formulering)
 *
 * Readings of points the summaries leave open (each is a documented
 * parameter of the build, mirrored here):
 *   - the shared expert's keys are Qt and its values Vt (nl: "Qt, Vt are the
 *     landmark keys/values");
 *   - Atten(.) is softmax attention with scale 1/sqrt(d) unless a scale is given;
 *   - top-k scores are the raw, unscaled dot products k_j . qt_i; ties go to
 *     the lower key index; I_i is returned in ascending index order;
 *   - a query is routed to the s landmarks with the largest q . qt_i (ties to
 *     the lower landmark index), listed by descending score;
 *   - overlapping expert sets are concatenated: a key chosen by two routed
 *     experts occupies two slots;
 *   - adaptive pooling bins are [floor(i*N/m), ceil((i+1)*N/m)) per axis;
 *   - one joint softmax over all m + s*k slots, non-causal.
 *
 * Causal variant (causal = 1; the summaries do not describe one, so every
 * rule below is a reading of this build, for 1-D pooling only):
 *   - the shared expert of landmark i attends to the keys of its prefix only,
 *     Vt_i = softmax over j < hi_i, where [lo_i, hi_i) is landmark i's bin;
 *   - query t has the shared slot of landmark i only once that bin is
 *     complete, hi_i <= t + 1;
 *   - expert sets and routes are selected as in the non-causal pass; of a
 *     routed expert's keys, query t attends to those with j <= t;
 *   - a query left with no slot gets a zero output row.
 *
 * Pins: see tests/test_oracle_pins.py (closed forms, brute force, library
 * special cases, a hand-derived example).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int N, d, m, k, s;
    int grid_h, grid_w; /* token grid for 2D pooling; grid_h == 1 means 1D */
    int lm_h, lm_w;     /* landmark grid; lm_h == 1 means 1D               */
    double scale;       /* <= 0 means 1/sqrt(d)                             */
    int no_shared;      /* 1: drop the m shared slots from step 5           */
    int causal;         /* 1: the causal variant (1-D pooling only)         */
} mo_params;

/* ---------------------------------------------------------------- step 1 */

/* Adaptive average pooling bin along one axis of length L into P bins. */
static void mo_bin(int i, int L, int P, int* lo, int* hi) {
    *lo = (int)(((int64_t)i * L) / P);
    *hi = (int)((((int64_t)(i + 1) * L) + P - 1) / P);
}

/* Qt[i] = mean of Q over landmark i's bin (1D, or 2D over a row-major
 * grid_h x grid_w token grid). */
static void mo_pool_head(const mo_params* p, const double* Q, double* Qt) {
    const int d = p->d;
    for (int i = 0; i < p->m; ++i) {
        int R = i / p->lm_w, C = i % p->lm_w;
        int r0, r1, c0, c1;
        mo_bin(R, p->grid_h, p->lm_h, &r0, &r1);
        mo_bin(C, p->grid_w, p->lm_w, &c0, &c1);
        double* out = Qt + (size_t)i * d;
        for (int c = 0; c < d; ++c) out[c] = 0.0;
        int64_t cnt = 0;
        for (int r = r0; r < r1; ++r)
            for (int cc = c0; cc < c1; ++cc) {
                const double* q = Q + ((size_t)r * p->grid_w + cc) * d;
                for (int c = 0; c < d; ++c) out[c] += q[c];
                ++cnt;
            }
        for (int c = 0; c < d; ++c) out[c] /= (double)cnt;
    }
}

/* ------------------------------------------------------------- helpers */

static double mo_dot(const double* a, const double* b, int d) {
    double acc = 0.0;
    for (int c = 0; c < d; ++c) acc += a[c] * b[c];
    return acc;
}

/* Sort key for "largest score first, lower index on ties". */
typedef struct {
    double v;
    int32_t j;
} mo_item;

static int mo_cmp_desc(const void* a, const void* b) {
    const mo_item* x = (const mo_item*)a;
    const mo_item* y = (const mo_item*)b;
    if (x->v > y->v) return -1;
    if (x->v < y->v) return 1;
    return (x->j < y->j) ? -1 : (x->j > y->j);
}

static int mo_cmp_i32(const void* a, const void* b) {
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

/* ------------------------------------------------------------ one head */

typedef struct {
    const mo_params* p;
    const double *Q, *K, *V;   /* [N][d] of this head            */
    int n_q;                   /* queries whose output is wanted */
    const int32_t* q_ids;      /* NULL: all N                    */
    const int32_t* I_over;     /* [m][k] or NULL                 */
    const int32_t* E_over;     /* [n_q][s] or NULL               */
    double *Qt, *Vt, *O;       /* [m][d], [m][d], [n_q][d]       */
    int32_t *I, *E;            /* [m][k], [n_q][s]               */
    uint64_t macs;
    int err;
} mo_job;

static void mo_run_head(mo_job* jb) {
    const mo_params* p = jb->p;
    const int N = p->N, d = p->d, m = p->m, k = p->k, s = p->s;
    const double tau = p->scale > 0 ? p->scale : 1.0 / sqrt((double)d);
    uint64_t macs = 0;

    /* step 1 */
    mo_pool_head(p, jb->Q, jb->Qt);

    /* steps 2 and 3, one landmark row at a time: the raw scores
     * s_ij = qt_i . k_j feed both the shared expert (scaled) and the top-k. */
    double* srow = (double*)malloc(sizeof(double) * (size_t)N);
    mo_item* items = (mo_item*)malloc(sizeof(mo_item) * (size_t)N);
    if (!srow || !items) { jb->err = 1; free(srow); free(items); return; }
    for (int i = 0; i < m; ++i) {
        const double* qt = jb->Qt + (size_t)i * d;
        double mx = -INFINITY;
        for (int j = 0; j < N; ++j) {
            srow[j] = mo_dot(qt, jb->K + (size_t)j * d, d);
            if (tau * srow[j] > mx) mx = tau * srow[j];
        }
        macs += (uint64_t)N * d;
        /* Vt_i = sum_j softmax_j(tau s_ij) v_j, max-subtracted; the causal
         * variant keeps the keys of landmark i's prefix, j < hi_i */
        int jend = N;
        if (p->causal) {
            int lo, hi;
            mo_bin(i, N, m, &lo, &hi);
            jend = hi;
            mx = -INFINITY;
            for (int j = 0; j < jend; ++j)
                if (tau * srow[j] > mx) mx = tau * srow[j];
        }
        double* vt = jb->Vt + (size_t)i * d;
        for (int c = 0; c < d; ++c) vt[c] = 0.0;
        double den = 0.0;
        for (int j = 0; j < jend; ++j) {
            double w = exp(tau * srow[j] - mx);
            den += w;
            const double* v = jb->V + (size_t)j * d;
            for (int c = 0; c < d; ++c) vt[c] += w * v[c];
        }
        for (int c = 0; c < d; ++c) vt[c] /= den;
        macs += (uint64_t)jend * d;
        /* I_i: first k of (score desc, index asc), then ascending index */
        int32_t* Ii = jb->I + (size_t)i * k;
        if (jb->I_over) {
            memcpy(Ii, jb->I_over + (size_t)i * k, sizeof(int32_t) * (size_t)k);
        } else {
            for (int j = 0; j < N; ++j) { items[j].v = srow[j]; items[j].j = j; }
            qsort(items, (size_t)N, sizeof(mo_item), mo_cmp_desc);
            for (int t = 0; t < k; ++t) Ii[t] = items[t].j;
            qsort(Ii, (size_t)k, sizeof(int32_t), mo_cmp_i32);
        }
    }
    free(items);
    free(srow);

    /* steps 4 and 5 per query */
    const int nslot = (p->no_shared ? 0 : m) + s * k;
    double* logit = (double*)malloc(sizeof(double) * (size_t)nslot);
    const double** vals = (const double**)malloc(sizeof(double*) * (size_t)nslot);
    mo_item* r = (mo_item*)malloc(sizeof(mo_item) * (size_t)m);
    if (!logit || !vals || !r) { jb->err = 1; free(logit); free(vals); free(r); return; }
    for (int t = 0; t < jb->n_q; ++t) {
        const int qi = jb->q_ids ? jb->q_ids[t] : t;
        const double* q = jb->Q + (size_t)qi * d;
        int32_t* Et = jb->E + (size_t)t * s;
        /* step 4: route to the s landmarks with the largest q . qt_i */
        for (int i = 0; i < m; ++i) { r[i].v = mo_dot(q, jb->Qt + (size_t)i * d, d); r[i].j = i; }
        macs += (uint64_t)m * d;
        if (jb->E_over) {
            memcpy(Et, jb->E_over + (size_t)t * s, sizeof(int32_t) * (size_t)s);
        } else {
            qsort(r, (size_t)m, sizeof(mo_item), mo_cmp_desc);
            for (int e = 0; e < s; ++e) Et[e] = r[e].j;
        }
        /* step 5: K* = [Qt, K_(e1), ..., K_(es)], V* = [Vt, V_(e1), ...];
         * the causal variant drops the landmarks whose bin is not complete at
         * qi and the routed keys after qi */
        int n = 0;
        if (!p->no_shared)
            for (int i = 0; i < m; ++i) {
                if (p->causal) {
                    int lo, hi;
                    mo_bin(i, N, m, &lo, &hi);
                    if (hi > qi + 1) continue;
                }
                logit[n] = tau * mo_dot(q, jb->Qt + (size_t)i * d, d);
                vals[n++] = jb->Vt + (size_t)i * d;
            }
        for (int e = 0; e < s; ++e) {
            const int32_t* Ie = jb->I + (size_t)Et[e] * k;
            for (int t2 = 0; t2 < k; ++t2) {
                if (p->causal && Ie[t2] > qi) continue;
                logit[n] = tau * mo_dot(q, jb->K + (size_t)Ie[t2] * d, d);
                vals[n++] = jb->V + (size_t)Ie[t2] * d;
            }
        }
        if (n == 0) {  /* causal only: no slot at all */
            double* o = jb->O + (size_t)t * d;
            for (int c = 0; c < d; ++c) o[c] = 0.0;
            continue;
        }
        double mx = -INFINITY;
        for (int u = 0; u < n; ++u) if (logit[u] > mx) mx = logit[u];
        double den = 0.0;
        double* o = jb->O + (size_t)t * d;
        for (int c = 0; c < d; ++c) o[c] = 0.0;
        for (int u = 0; u < n; ++u) {
            double w = exp(logit[u] - mx);
            den += w;
            for (int c = 0; c < d; ++c) o[c] += w * vals[u][c];
        }
        for (int c = 0; c < d; ++c) o[c] /= den;
        macs += 2ull * (uint64_t)n * d;
    }
    free(r);
    free(vals);
    free(logit);
    jb->macs = macs;
}

static void* mo_worker(void* arg) {
    mo_job** q = (mo_job**)arg;
    /* arg points at {jobs, counter}; see mo_forward */
    mo_job* jobs = q[0];
    int* next = (int*)q[1];
    int njobs = *(int*)q[2];
    pthread_mutex_t* mu = (pthread_mutex_t*)q[3];
    for (;;) {
        pthread_mutex_lock(mu);
        int h = (*next)++;
        pthread_mutex_unlock(mu);
        if (h >= njobs) break;
        mo_run_head(&jobs[h]);
    }
    return NULL;
}

/* ------------------------------------------------------------ C API */

static int mo_check(const mo_params* p) {
    if (p->N < 1 || p->d < 1 || p->m < 1 || p->m > p->N) return -1;
    if (p->k < 1 || p->k > p->N || p->s < 1 || p->s > p->m) return -1;
    if (p->grid_h < 1 || p->grid_w < 1 || p->grid_h * p->grid_w != p->N) return -1;
    if (p->lm_h < 1 || p->lm_w < 1 || p->lm_h * p->lm_w != p->m) return -1;
    if (p->lm_h > p->grid_h || p->lm_w > p->grid_w) return -1;
    if (p->causal && p->grid_h != 1) return -1; /* causal: 1-D token order only */
    return 0;
}

/* Landmark queries only (step 1), for n_heads heads laid out [n_heads][N][d]. */
int mo_pool(const mo_params* p, int n_heads, const double* Q, double* Qt) {
    if (mo_check(p)) return -1;
    for (int h = 0; h < n_heads; ++h)
        mo_pool_head(p, Q + (size_t)h * p->N * p->d, Qt + (size_t)h * p->m * p->d);
    return 0;
}

/* Raw scores S[i][j] = A_i . B_j (used by tests for the gap rule). */
int mo_scores(const double* A, int na, const double* B, int nb, int d, double* S) {
    for (int i = 0; i < na; ++i)
        for (int j = 0; j < nb; ++j) S[(size_t)i * nb + j] = mo_dot(A + (size_t)i * d, B + (size_t)j * d, d);
    return 0;
}

/*
 * Full forward for n_heads independent heads, inputs [n_heads][N][d].
 * q_ids (length n_q, shared by all heads) selects the queries whose routes
 * and outputs are computed; NULL with n_q == N means every query.
 * I_over [n_heads][m][k] / E_over [n_heads][n_q][s] replace steps 3 / 4 by
 * given index sets (used to recompute outputs on another implementation's
 * sets). Outputs: Qt, Vt [n_heads][m][d]; I [n_heads][m][k];
 * E [n_heads][n_q][s]; O [n_heads][n_q][d]. macs (may be NULL) receives the
 * multiply-add count of steps 2, 4 and 5.
 */
int mo_forward(const mo_params* p, int n_heads, const double* Q, const double* K, const double* V,
               int n_q, const int32_t* q_ids, const int32_t* I_over, const int32_t* E_over,
               double* Qt, double* Vt, int32_t* I, int32_t* E, double* O, int nthreads,
               uint64_t* macs) {
    if (mo_check(p) || n_heads < 0 || n_q < 0) return -1;
    if (!q_ids && n_q != p->N) return -1;
    for (int t = 0; q_ids && t < n_q; ++t)
        if (q_ids[t] < 0 || q_ids[t] >= p->N) return -1;
    const size_t Nd = (size_t)p->N * p->d, md = (size_t)p->m * p->d;
    mo_job* jobs = (mo_job*)calloc((size_t)(n_heads > 0 ? n_heads : 1), sizeof(mo_job));
    if (!jobs) return -2;
    for (int h = 0; h < n_heads; ++h) {
        mo_job* jb = &jobs[h];
        jb->p = p;
        jb->Q = Q + h * Nd; jb->K = K + h * Nd; jb->V = V + h * Nd;
        jb->n_q = n_q; jb->q_ids = q_ids;
        jb->I_over = I_over ? I_over + (size_t)h * p->m * p->k : NULL;
        jb->E_over = E_over ? E_over + (size_t)h * n_q * p->s : NULL;
        jb->Qt = Qt + h * md; jb->Vt = Vt + h * md;
        jb->I = I + (size_t)h * p->m * p->k;
        jb->E = E + (size_t)h * n_q * p->s;
        jb->O = O + (size_t)h * n_q * p->d;
    }
    if (nthreads < 1) nthreads = 1;
    if (nthreads > n_heads) nthreads = n_heads > 0 ? n_heads : 1;
    int next = 0;
    pthread_mutex_t mu = PTHREAD_MUTEX_INITIALIZER;
    void* ctx[4] = {jobs, &next, &n_heads, &mu};
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!th) { free(jobs); return -2; }
    int started = 0;
    for (int t = 1; t < nthreads; ++t)
        if (pthread_create(&th[t], NULL, mo_worker, ctx) == 0) ++started; else break;
    mo_worker(ctx);
    for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
    free(th);
    int err = 0;
    uint64_t total = 0;
    for (int h = 0; h < n_heads; ++h) { err |= jobs[h].err; total += jobs[h].macs; }
    free(jobs);
    if (macs) *macs = total;
    return err ? -2 : 0;
}
