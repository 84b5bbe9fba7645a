/*
 * Scaled dot-product attention forward: the CPU oracle.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the bench's CPU
 * baseline may load this library.  It shares no code, header, table or helper
 * with the CUDA path; it is slow on purpose and meant to be checked by eye.
 *
 * What it computes (the naive reference of the VeriTile page
 * "VeriTile.Examples.FlashAttention1.NaiveRefinement", definitions
 * fa1NaiveReference4D / fa1NaiveCausalReference4D, and the CPU routine
 * `expectedOutput` of the accy page "tiny.accy.kernel.library.attention"):
 * for every batch b, head h and query row i
 *
 *   A_i   = { j < S_k }                 (non-causal)
 *         = { j < S_k : j <= i }        (causal, key j <= query i, top-left)
 *   s_j   = scale * sum_{d < D_qk} Q[b,h,i,d] * K[b,h,j,d]      j in A_i
 *   m     = max_{j in A_i} s_j
 *   l     = sum_{j in A_i} exp(s_j - m)
 *   O[b,h,i,e] = sum_{j in A_i} (exp(s_j - m) / l) * V[b,h,j,e]   e < D_v
 *
 * in fp64 with the host libm's natural-base exp.  The inputs are the exact
 * values of the stored fp32 or bf16 elements, widened to double; `scale` is
 * the fp32 value the caller passes, widened.  Tensors are contiguous
 * [B,H,S,D] with D innermost.
 *
 * oracle_attn_fwd_ld is an independent brute force in long double for tiny
 * inputs: it forms the softmax weights as exp(s_j) / sum_k exp(s_k) without
 * the max shift, so it shares the definition but not the algorithm.
 *
 * Build (done by the repository's build step): gcc -O2 -shared -fPIC
 *   -o liboracle.so attn_oracle.c -lm -lpthread
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_BF16 = 1 };

/* The stored element idx of a tensor, widened exactly to double. */
static double elem(const void *base, int dtype, int64_t idx) {
    if (dtype == ORC_F32) {
        return (double)((const float *)base)[idx];
    } else {
        uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
}

typedef struct {
    const void *Q, *K, *V;
    double *O;                  /* output rows, D_v doubles each */
    int64_t B, H, S_q, S_k, D_qk, D_v;
    double scale;
    int causal, dtype;
    const int64_t *rows;        /* NULL: all rows in order; else (b, h, i) triples */
    int64_t nrows;
    int64_t next;               /* work counter, guarded by mu */
    pthread_mutex_t mu;
} job_t;

/* One output row O[b,h,i,:] following the five steps above. */
static void one_row(const job_t *J, int64_t b, int64_t h, int64_t i, double *s, double *out) {
    const int64_t bh = b * J->H + h;
    const int64_t q0 = (bh * J->S_q + i) * J->D_qk;
    /* step 1: the allowed keys are j < n_keys */
    int64_t n_keys = J->S_k;
    if (J->causal && i + 1 < n_keys) n_keys = i + 1;
    /* step 2: scores */
    for (int64_t j = 0; j < n_keys; ++j) {
        const int64_t k0 = (bh * J->S_k + j) * J->D_qk;
        double dot = 0.0;
        for (int64_t d = 0; d < J->D_qk; ++d)
            dot += elem(J->Q, J->dtype, q0 + d) * elem(J->K, J->dtype, k0 + d);
        s[j] = J->scale * dot;
    }
    /* step 3: row max */
    double m = -INFINITY;
    for (int64_t j = 0; j < n_keys; ++j)
        if (s[j] > m) m = s[j];
    /* step 4: shifted exponential sum */
    double l = 0.0;
    for (int64_t j = 0; j < n_keys; ++j) l += exp(s[j] - m);
    /* step 5: value-weighted sum */
    for (int64_t e = 0; e < J->D_v; ++e) out[e] = 0.0;
    for (int64_t j = 0; j < n_keys; ++j) {
        const double w = exp(s[j] - m) / l;
        const int64_t v0 = (bh * J->S_k + j) * J->D_v;
        for (int64_t e = 0; e < J->D_v; ++e) out[e] += w * elem(J->V, J->dtype, v0 + e);
    }
}

static void *worker(void *arg) {
    job_t *J = (job_t *)arg;
    double *s = (double *)malloc(sizeof(double) * (size_t)(J->S_k > 0 ? J->S_k : 1));
    if (!s) return (void *)1;
    const int64_t total = J->rows ? J->nrows : J->B * J->H * J->S_q;
    for (;;) {
        pthread_mutex_lock(&J->mu);
        int64_t r = J->next;
        J->next += 16;
        pthread_mutex_unlock(&J->mu);
        if (r >= total) break;
        int64_t r_end = r + 16 < total ? r + 16 : total;
        for (; r < r_end; ++r) {
            int64_t b, h, i;
            if (J->rows) {
                b = J->rows[3 * r]; h = J->rows[3 * r + 1]; i = J->rows[3 * r + 2];
            } else {
                i = r % J->S_q; h = (r / J->S_q) % J->H; b = r / (J->S_q * J->H);
            }
            one_row(J, b, h, i, s, J->O + r * J->D_v);
        }
    }
    free(s);
    return NULL;
}

static int run(job_t *J, int nthreads) {
    if (J->B < 0 || J->H < 0 || J->S_q < 0 || J->S_k < 1 || J->D_qk < 1 || J->D_v < 1) return 1;
    if (J->dtype != ORC_F32 && J->dtype != ORC_BF16) return 1;
    if (J->rows) {
        for (int64_t r = 0; r < J->nrows; ++r) {
            const int64_t *t = J->rows + 3 * r;
            if (t[0] < 0 || t[0] >= J->B || t[1] < 0 || t[1] >= J->H || t[2] < 0 || t[2] >= J->S_q) return 2;
        }
    }
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t th[256];
    pthread_mutex_init(&J->mu, NULL);
    J->next = 0;
    int started = 0, rc = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, worker, J) != 0) break;
        ++started;
    }
    if (started == 0) rc = 3, worker(J);
    for (int t = 0; t < started; ++t) {
        void *ret = NULL;
        pthread_join(th[t], &ret);
        if (ret) rc = 4;
    }
    pthread_mutex_destroy(&J->mu);
    return rc == 3 ? 0 : rc;
}

/* Full output O[B,H,S_q,D_v] in fp64.  Returns 0 on success. */
int oracle_attn_fwd(const void *Q, const void *K, const void *V, double *O,
                    int64_t B, int64_t H, int64_t S_q, int64_t S_k, int64_t D_qk, int64_t D_v,
                    double scale, int causal, int dtype, int nthreads) {
    job_t J = {Q, K, V, O, B, H, S_q, S_k, D_qk, D_v, scale, causal, dtype, NULL, 0};
    return run(&J, nthreads);
}

/* Selected output rows: rows holds nrows (b, h, i) triples; O receives nrows x D_v. */
int oracle_attn_rows(const void *Q, const void *K, const void *V, double *O,
                     int64_t B, int64_t H, int64_t S_q, int64_t S_k, int64_t D_qk, int64_t D_v,
                     double scale, int causal, int dtype, const int64_t *rows, int64_t nrows,
                     int nthreads) {
    job_t J = {Q, K, V, O, B, H, S_q, S_k, D_qk, D_v, scale, causal, dtype, rows, nrows};
    return run(&J, nthreads);
}

/* Long-double brute force (single thread, tiny inputs): weights exp(s_j)/sum exp(s_k). */
int oracle_attn_fwd_ld(const void *Q, const void *K, const void *V, long double *O,
                       int64_t B, int64_t H, int64_t S_q, int64_t S_k, int64_t D_qk, int64_t D_v,
                       double scale, int causal, int dtype) {
    if (B < 0 || H < 0 || S_q < 0 || S_k < 1 || D_qk < 1 || D_v < 1) return 1;
    if (dtype != ORC_F32 && dtype != ORC_BF16) return 1;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t h = 0; h < H; ++h)
            for (int64_t i = 0; i < S_q; ++i) {
                long double den = 0.0L;
                long double *o = O + ((b * H + h) * S_q + i) * D_v;
                for (int64_t e = 0; e < D_v; ++e) o[e] = 0.0L;
                for (int64_t j = 0; j < S_k; ++j) {
                    if (causal && j > i) continue;
                    long double dot = 0.0L;
                    for (int64_t d = 0; d < D_qk; ++d)
                        dot += (long double)elem(Q, dtype, ((b * H + h) * S_q + i) * D_qk + d) *
                               (long double)elem(K, dtype, ((b * H + h) * S_k + j) * D_qk + d);
                    long double w = expl((long double)scale * dot);
                    den += w;
                    for (int64_t e = 0; e < D_v; ++e)
                        o[e] += w * (long double)elem(V, dtype, ((b * H + h) * S_k + j) * D_v + e);
                }
                for (int64_t e = 0; e < D_v; ++e) o[e] /= den;
            }
    return 0;
}
