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
 *   A_i   = the allowed keys of row i (below)
 *   s_j   = scale * sum_{d < D_qk} Q[b,h,i,d] * K[b,g,j,d]      j in A_i
 *   m     = max_{j in A_i} s_j
 *   l     = sum_{j in A_i} exp(s_j - m)
 *   O[b,h,i,e] = sum_{j in A_i} (exp(s_j - m) / l) * V[b,g,j,e]   e < D_v
 *   LSE[b,h,i] = m + log(l)            (natural log of sum_{j in A_i} exp(s_j))
 *
 * in fp64 with the host libm's natural-base exp and log.  g is the key/value
 * head of query head h: g = h / (H / H_kv) (grouped heads, the num_kv_heads
 * indexing of the VeriTile coverage table's block-sparse attention row; H_kv = H
 * is plain multi-head attention).  The allowed keys, with o = offset >= 0 and
 * w = window >= 1:
 *
 *   ORC_MASK_NONE       A_i = { j < S_k }
 *   ORC_MASK_CAUSAL     A_i = { j < S_k : j <= i + o }
 *                       (o = 0: key j <= query i, top-left; o > 0: query i sits
 *                       at key position i + o, the start_position of the coverage
 *                       table's attention_llama causal row)
 *   ORC_MASK_WINDOW     A_i = { j < S_k : i + o - w < j <= i + o }
 *                       (the w most recent keys: the sliding window of the
 *                       attention_fwd_triton3 row, case 1)
 *   ORC_MASK_WINDOW_COMPLEMENT
 *                       A_i = { j < S_k : j <= i + o - w }
 *                       (the causal keys the window leaves out: case 2)
 *
 * A row whose A_i is empty (possible only with the window kinds) has O = 0 and
 * LSE = -inf: the empty weighted sum, and the log of an empty sum of exponentials.
 * The inputs are the exact values of the stored fp32 or bf16 elements, widened
 * to double; `scale` is the fp32 value the caller passes, widened.  Tensors are
 * contiguous: Q [B,H,S_q,D_qk], K [B,H_kv,S_k,D_qk], V [B,H_kv,S_k,D_v],
 * O [B,H,S_q,D_v], LSE [B,H,S_q].
 *
 * oracle_attn_general_ld is an independent brute force in long double for
 * tiny inputs: it forms the softmax weights as exp(s_j) / sum_k exp(s_k)
 * without the max shift, so it shares the definition but not the algorithm.
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
enum { ORC_MASK_NONE = 0, ORC_MASK_CAUSAL = 1, ORC_MASK_WINDOW = 2, ORC_MASK_WINDOW_COMPLEMENT = 3 };

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
    double *LSE;                /* NULL, or one double per output row */
    int64_t B, H, H_kv, S_q, S_k, D_qk, D_v;
    double scale;
    int mask, dtype;
    int64_t offset, window;
    const int64_t *rows;        /* NULL: all rows in order; else (b, h, i) triples */
    int64_t nrows;
    int64_t next;               /* work counter, guarded by mu */
    pthread_mutex_t mu;
} job_t;

/* Is key j in the allowed set A_i of query row i?  (The table in the header.) */
static int allowed(const job_t *J, int64_t i, int64_t j) {
    switch (J->mask) {
    case ORC_MASK_NONE: return 1;
    case ORC_MASK_CAUSAL: return j <= i + J->offset;
    case ORC_MASK_WINDOW: return i + J->offset - J->window < j && j <= i + J->offset;
    case ORC_MASK_WINDOW_COMPLEMENT: return j <= i + J->offset - J->window;
    }
    return 0;
}

/* One output row O[b,h,i,:] (and LSE[b,h,i]) following the steps above.  keys and s hold S_k entries. */
static void one_row(const job_t *J, int64_t b, int64_t h, int64_t i, int64_t *keys, double *s,
                    double *out, double *lse) {
    const int64_t g = h / (J->H / J->H_kv);               /* key/value head of query head h */
    const int64_t q0 = ((b * J->H + h) * J->S_q + i) * J->D_qk;
    const int64_t kv = b * J->H_kv + g;
    /* step 1: the allowed keys, in increasing order */
    int64_t n_keys = 0;
    for (int64_t j = 0; j < J->S_k; ++j)
        if (allowed(J, i, j)) keys[n_keys++] = j;
    /* step 2: scores */
    for (int64_t n = 0; n < n_keys; ++n) {
        const int64_t j = keys[n];
        const int64_t k0 = (kv * J->S_k + j) * J->D_qk;
        double dot = 0.0;
        for (int64_t d = 0; d < J->D_qk; ++d)
            dot += elem(J->Q, J->dtype, q0 + d) * elem(J->K, J->dtype, k0 + d);
        s[n] = J->scale * dot;
    }
    /* step 3: row max */
    double m = -INFINITY;
    for (int64_t n = 0; n < n_keys; ++n)
        if (s[n] > m) m = s[n];
    /* step 4: shifted exponential sum */
    double l = 0.0;
    for (int64_t n = 0; n < n_keys; ++n) l += exp(s[n] - m);
    /* step 5: value-weighted sum (empty for a row with no allowed key) */
    for (int64_t e = 0; e < J->D_v; ++e) out[e] = 0.0;
    for (int64_t n = 0; n < n_keys; ++n) {
        const double w = exp(s[n] - m) / l;
        const int64_t v0 = (kv * J->S_k + keys[n]) * J->D_v;
        for (int64_t e = 0; e < J->D_v; ++e) out[e] += w * elem(J->V, J->dtype, v0 + e);
    }
    if (lse) *lse = n_keys > 0 ? m + log(l) : -INFINITY;
}

static void *worker(void *arg) {
    job_t *J = (job_t *)arg;
    const size_t n = (size_t)(J->S_k > 0 ? J->S_k : 1);
    double *s = (double *)malloc(sizeof(double) * n);
    int64_t *keys = (int64_t *)malloc(sizeof(int64_t) * n);
    if (!s || !keys) {
        free(s);
        free(keys);
        return (void *)1;
    }
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
            one_row(J, b, h, i, keys, s, J->O + r * J->D_v, J->LSE ? J->LSE + r : NULL);
        }
    }
    free(s);
    free(keys);
    return NULL;
}

/* Argument checks shared by the fp64 and long-double entry points. */
static int bad_args(int64_t B, int64_t H, int64_t H_kv, int64_t S_q, int64_t S_k, int64_t D_qk, int64_t D_v,
                    int mask, int64_t offset, int64_t window, int dtype) {
    if (B < 0 || H < 0 || S_q < 0 || S_k < 1 || D_qk < 1 || D_v < 1) return 1;
    if (H_kv < 1 || (H > 0 && H % H_kv != 0)) return 1;
    if (dtype != ORC_F32 && dtype != ORC_BF16) return 1;
    if (mask < ORC_MASK_NONE || mask > ORC_MASK_WINDOW_COMPLEMENT || offset < 0) return 1;
    if ((mask == ORC_MASK_WINDOW || mask == ORC_MASK_WINDOW_COMPLEMENT) && window < 1) return 1;
    return 0;
}

static int run(job_t *J, int nthreads) {
    if (bad_args(J->B, J->H, J->H_kv, J->S_q, J->S_k, J->D_qk, J->D_v, J->mask, J->offset, J->window, J->dtype))
        return 1;
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

/* General form: O (and LSE if not NULL) for all rows (rows == NULL) or for nrows (b, h, i)
 * triples.  mask, offset, window and H_kv as in the header.  Returns 0 on success. */
int oracle_attn_general(const void *Q, const void *K, const void *V, double *O, double *LSE,
                        int64_t B, int64_t H, int64_t H_kv, int64_t S_q, int64_t S_k, int64_t D_qk,
                        int64_t D_v, double scale, int mask, int64_t offset, int64_t window, int dtype,
                        const int64_t *rows, int64_t nrows, int nthreads) {
    job_t J;
    memset(&J, 0, sizeof J);
    J.Q = Q; J.K = K; J.V = V; J.O = O; J.LSE = LSE;
    J.B = B; J.H = H; J.H_kv = H_kv; J.S_q = S_q; J.S_k = S_k; J.D_qk = D_qk; J.D_v = D_v;
    J.scale = scale; J.mask = mask; J.dtype = dtype; J.offset = offset; J.window = window;
    J.rows = rows; J.nrows = nrows;
    return run(&J, nthreads);
}

/* Full output O[B,H,S_q,D_v] in fp64, H_kv = H, non-causal or causal with offset 0. */
int oracle_attn_fwd(const void *Q, const void *K, const void *V, double *O,
                    int64_t B, int64_t H, int64_t S_q, int64_t S_k, int64_t D_qk, int64_t D_v,
                    double scale, int causal, int dtype, int nthreads) {
    return oracle_attn_general(Q, K, V, O, NULL, B, H, H > 0 ? H : 1, S_q, S_k, D_qk, D_v, scale,
                               causal ? ORC_MASK_CAUSAL : ORC_MASK_NONE, 0, 0, dtype, NULL, 0, nthreads);
}

/* Selected output rows: rows holds nrows (b, h, i) triples; O receives nrows x D_v. */
int oracle_attn_rows(const void *Q, const void *K, const void *V, double *O,
                     int64_t B, int64_t H, int64_t S_q, int64_t S_k, int64_t D_qk, int64_t D_v,
                     double scale, int causal, int dtype, const int64_t *rows, int64_t nrows,
                     int nthreads) {
    return oracle_attn_general(Q, K, V, O, NULL, B, H, H > 0 ? H : 1, S_q, S_k, D_qk, D_v, scale,
                               causal ? ORC_MASK_CAUSAL : ORC_MASK_NONE, 0, 0, dtype, rows, nrows, nthreads);
}

/* Long-double brute force (single thread, tiny inputs): weights exp(s_j)/sum exp(s_k) over the
 * keys the mask keeps, written out again for each kind; LSE = log of that sum.  An empty row
 * gives O = 0 and LSE = -inf. */
int oracle_attn_general_ld(const void *Q, const void *K, const void *V, long double *O, long double *LSE,
                           int64_t B, int64_t H, int64_t H_kv, int64_t S_q, int64_t S_k, int64_t D_qk,
                           int64_t D_v, double scale, int mask, int64_t offset, int64_t window, int dtype) {
    if (bad_args(B, H, H_kv, S_q, S_k, D_qk, D_v, mask, offset, window, dtype)) return 1;
    const int64_t group = H / H_kv;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t h = 0; h < H; ++h)
            for (int64_t i = 0; i < S_q; ++i) {
                long double den = 0.0L;
                long double *o = O + ((b * H + h) * S_q + i) * D_v;
                for (int64_t e = 0; e < D_v; ++e) o[e] = 0.0L;
                for (int64_t j = 0; j < S_k; ++j) {
                    int keep = 1;
                    if (mask == ORC_MASK_CAUSAL) keep = !(j > i + offset);
                    if (mask == ORC_MASK_WINDOW) keep = !(j > i + offset) && !(j + window <= i + offset);
                    if (mask == ORC_MASK_WINDOW_COMPLEMENT) keep = !(j + window > i + offset);
                    if (!keep) continue;
                    const int64_t kvrow = (b * H_kv + h / group) * S_k + j;
                    long double dot = 0.0L;
                    for (int64_t d = 0; d < D_qk; ++d)
                        dot += (long double)elem(Q, dtype, ((b * H + h) * S_q + i) * D_qk + d) *
                               (long double)elem(K, dtype, kvrow * D_qk + d);
                    long double w = expl((long double)scale * dot);
                    den += w;
                    for (int64_t e = 0; e < D_v; ++e)
                        o[e] += w * (long double)elem(V, dtype, kvrow * D_v + e);
                }
                if (den > 0.0L)
                    for (int64_t e = 0; e < D_v; ++e) o[e] /= den;
                if (LSE) LSE[(b * H + h) * S_q + i] = den > 0.0L ? logl(den) : -INFINITY;
            }
    return 0;
}

/* The long-double brute force for H_kv = H, non-causal or causal with offset 0. */
int oracle_attn_fwd_ld(const void *Q, const void *K, const void *V, long double *O,
                       int64_t B, int64_t H, int64_t S_q, int64_t S_k, int64_t D_qk, int64_t D_v,
                       double scale, int causal, int dtype) {
    return oracle_attn_general_ld(Q, K, V, O, NULL, B, H, H > 0 ? H : 1, S_q, S_k, D_qk, D_v, scale,
                                  causal ? ORC_MASK_CAUSAL : ORC_MASK_NONE, 0, 0, dtype);
}
