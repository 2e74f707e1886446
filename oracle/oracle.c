/*
 * CPU oracle -- TEST INFRASTRUCTURE, not part of the product path.
 *
 * Plain, slow, obviously correct restatement of the two operations in fp64.
 * The only structure beyond the defining sums is that independent output rows
 * (addmm) or (image, channel) planes (conv2d) are handed to worker threads;
 * every output element is still one sequential sum in the defining order.
 * See oracle.h for the definitions and their sources.
 */
#define _GNU_SOURCE
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <sched.h>
#include <stdlib.h>
#include <unistd.h>

/* ORACLE_PLANT selects one deliberate mistake for the tests that check the
 * pins catch it (0, the default, builds the correct oracle):
 *   1 addmm subtracts products      2 addmm drops beta*self
 *   3 addmm ignores self_2d         4 conv uses dH on the width axis
 *   5 conv drops the bias           6 conv shifts ih by one
 *   7 conv output size misses -1    8 S sums signed products
 *   9 the fp32 loop accumulates in fp64 */
#ifndef ORACLE_PLANT
#define ORACLE_PLANT 0
#endif

int oracle_default_threads(void) {
#ifdef CPU_COUNT
    cpu_set_t set;
    if (sched_getaffinity(0, sizeof(set), &set) == 0) {
        int n = CPU_COUNT(&set);
        if (n > 0) return n;
    }
#endif
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/* ---------------------------------------------------------------- threads */

typedef void (*work_fn)(void* ctx, int64_t item);

typedef struct {
    work_fn fn;
    void* ctx;
    int64_t nitems;
    int64_t first, step;
} worker_arg;

static void* worker_main(void* p) {
    worker_arg* a = (worker_arg*)p;
    for (int64_t i = a->first; i < a->nitems; i += a->step) a->fn(a->ctx, i);
    return NULL;
}

/* Runs fn(ctx, i) for i in [0, nitems) on up to nthreads threads. */
static void run_items(work_fn fn, void* ctx, int64_t nitems, int nthreads) {
    if (nthreads <= 0) nthreads = oracle_default_threads();
    if (nthreads > nitems) nthreads = (int)(nitems > 0 ? nitems : 1);
    if (nthreads <= 1) {
        for (int64_t i = 0; i < nitems; ++i) fn(ctx, i);
        return;
    }
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    worker_arg* args = (worker_arg*)malloc(sizeof(worker_arg) * (size_t)nthreads);
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        args[t].fn = fn;
        args[t].ctx = ctx;
        args[t].nitems = nitems;
        args[t].first = t;
        args[t].step = nthreads;
        if (pthread_create(&th[t], NULL, worker_main, &args[t]) == 0) {
            ++started;
        } else {
            /* could not start a thread: do its share on this one */
            worker_main(&args[t]);
            th[t] = 0;
        }
    }
    for (int t = 0; t < nthreads; ++t)
        if (th[t]) pthread_join(th[t], NULL);
    (void)started;
    free(args);
    free(th);
}

/* ------------------------------------------------------------------ addmm */

typedef struct {
    const float *self, *mat1, *mat2;
    int self_2d;
    int64_t M, N, K;
    double beta, alpha;
    const int64_t* rows;
    double *ref, *sabs;
} addmm_ctx;

/* One output row: out[i, j] = beta * self(i, j) + alpha * sum_k mat1[i,k] mat2[k,j]. */
static void addmm_row(void* p, int64_t r) {
    const addmm_ctx* c = (const addmm_ctx*)p;
    const int64_t i = c->rows ? c->rows[r] : r;
    for (int64_t j = 0; j < c->N; ++j) {
        double acc = 0.0, s = 0.0;
        if (c->alpha != 0.0) {
            for (int64_t k = 0; k < c->K; ++k) {
                double prod = (double)c->mat1[i * c->K + k] * (double)c->mat2[k * c->N + j];
                acc += (ORACLE_PLANT == 1) ? -prod : prod;
                s += (ORACLE_PLANT == 8) ? prod : fabs(prod);
            }
        }
        double self_val = 0.0;
        if (c->beta != 0.0)
            self_val = (c->self_2d && ORACLE_PLANT != 3) ? (double)c->self[i * c->N + j]
                                                         : (double)c->self[j];
        double v = 0.0;
        if (c->beta != 0.0 && ORACLE_PLANT != 2) v += c->beta * self_val;
        if (c->alpha != 0.0) v += c->alpha * acc;
        c->ref[r * c->N + j] = v;
        if (c->sabs) c->sabs[r * c->N + j] = s;
    }
}

int oracle_addmm(const float* self, int self_2d, const float* mat1, const float* mat2,
                 int64_t M, int64_t N, int64_t K, double beta, double alpha,
                 const int64_t* rows, int64_t nrows, int nthreads,
                 double* ref, double* sabs) {
    if (M < 0 || N < 0 || K < 0 || nrows < 0 || !ref) return ORACLE_EARG;
    if (self_2d != 0 && self_2d != 1) return ORACLE_EARG;
    if (beta != 0.0 && !self) return ORACLE_EARG;
    if (alpha != 0.0 && K > 0 && (!mat1 || !mat2)) return ORACLE_EARG;
    if (!rows && nrows != M) return ORACLE_EARG;
    if (rows)
        for (int64_t r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= M) return ORACLE_EARG;
    addmm_ctx c = {self, mat1, mat2, self_2d, M, N, K, beta, alpha, rows, ref, sabs};
    run_items(addmm_row, &c, nrows, nthreads);
    return ORACLE_OK;
}

int oracle_addmm_fp32_naive(const float* self, int self_2d, const float* mat1,
                            const float* mat2, int64_t M, int64_t N, int64_t K,
                            float beta, float alpha, float* out) {
    if (M < 0 || N < 0 || K < 0 || !self || !mat1 || !mat2 || !out) return ORACLE_EARG;
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
#if ORACLE_PLANT == 9
            double acc = 0.0;
#else
            float acc = 0.0f;
#endif
            for (int64_t k = 0; k < K; ++k) acc += mat1[i * K + k] * mat2[k * N + j];
            float sv = self_2d ? self[i * N + j] : self[j];
            out[i * N + j] = beta * sv + alpha * acc;
        }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------ conv2d */

int64_t oracle_conv_out_size(int64_t in, int64_t k, int64_t stride, int64_t pad, int64_t dil) {
    if (in < 1 || k < 1 || stride < 1 || pad < 0 || dil < 1) return -1;
    int64_t span = in + 2 * pad - dil * (k - 1) - ((ORACLE_PLANT == 7) ? 0 : 1);
    if (span < 0) return -1;
    return span / stride + 1;
}

typedef struct {
    const float *x, *w, *bias;
    int64_t B, IC, H, W, OC, KH, KW, sH, sW, pH, pW, dH, dW, OH, OW;
    const int64_t* ocs;
    int64_t nocs;
    double *ref, *sabs;
} conv_ctx;

/* One (image b, selected channel c) output plane, seven nested loops in
 * total: b, oc, oh, ow, then ic, kh, kw over the receptive field. */
static void conv_plane(void* p, int64_t item) {
    const conv_ctx* c = (const conv_ctx*)p;
    const int64_t b = item / c->nocs, ci = item % c->nocs;
    const int64_t oc = c->ocs ? c->ocs[ci] : ci;
    double* out = c->ref + (b * c->nocs + ci) * c->OH * c->OW;
    double* sab = c->sabs ? c->sabs + (b * c->nocs + ci) * c->OH * c->OW : NULL;
    for (int64_t oh = 0; oh < c->OH; ++oh)
        for (int64_t ow = 0; ow < c->OW; ++ow) {
            double acc = (c->bias && ORACLE_PLANT != 5) ? (double)c->bias[oc] : 0.0;
            double s = 0.0;
            for (int64_t ic = 0; ic < c->IC; ++ic)
                for (int64_t kh = 0; kh < c->KH; ++kh)
                    for (int64_t kw = 0; kw < c->KW; ++kw) {
                        const int64_t ih = oh * c->sH - c->pH + kh * c->dH +
                                           ((ORACLE_PLANT == 6) ? 1 : 0);
                        const int64_t iw = ow * c->sW - c->pW +
                                           kw * ((ORACLE_PLANT == 4) ? c->dH : c->dW);
                        if (ih < 0 || ih >= c->H || iw < 0 || iw >= c->W) continue;
                        const double wv = c->w[((oc * c->IC + ic) * c->KH + kh) * c->KW + kw];
                        const double xv = c->x[((b * c->IC + ic) * c->H + ih) * c->W + iw];
                        acc += wv * xv;
                        s += fabs(wv * xv);
                    }
            out[oh * c->OW + ow] = acc;
            if (sab) sab[oh * c->OW + ow] = s;
        }
}

int oracle_conv2d(const float* x, const float* w, const float* bias,
                  int64_t B, int64_t IC, int64_t H, int64_t W, int64_t OC,
                  int64_t KH, int64_t KW, int64_t sH, int64_t sW, int64_t pH, int64_t pW,
                  int64_t dH, int64_t dW, const int64_t* ocs, int64_t nocs, int nthreads,
                  double* ref, double* sabs) {
    if (B < 0 || IC < 0 || OC < 0 || nocs < 0 || !ref) return ORACLE_EARG;
    const int64_t OH = oracle_conv_out_size(H, KH, sH, pH, dH);
    const int64_t OW = oracle_conv_out_size(W, KW, sW, pW, dW);
    if (OH < 1 || OW < 1) return ORACLE_EARG;
    if (!ocs && nocs != OC) return ORACLE_EARG;
    if (ocs)
        for (int64_t c = 0; c < nocs; ++c)
            if (ocs[c] < 0 || ocs[c] >= OC) return ORACLE_EARG;
    if (B > 0 && IC > 0 && (!x || !w)) return ORACLE_EARG;
    conv_ctx c = {x, w, bias, B, IC, H, W, OC, KH, KW, sH, sW, pH, pW, dH, dW, OH, OW,
                  ocs, nocs, ref, sabs};
    run_items(conv_plane, &c, B * nocs, nthreads);
    return ORACLE_OK;
}
