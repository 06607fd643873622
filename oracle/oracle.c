/*
 * oracle.c - exact softmax attention, plain fp64 CPU reference ("the oracle").
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or load
 * this file or the library built from it; only the tests, the smoke check and
 * the CPU-baseline leg of the benchmark do.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * What it computes (the plain definition, no blocking, no online rescaling):
 *
 *   "Ring Attention explained" (guijiagi.com), section "朴素 Attention 的显存墙":
 *       Attn(Q,K,V) = softmax(Q K^T / sqrt(d)) V
 *   "第12章 FlashAttention原理与实现", the `standard_attention` function of the
 *   benchmark section: scores = Q K^T * scale, softmax over the key axis, times V.
 *
 * For one query row i of batch b and query head h, with KV head hk = h / (Hq/Hkv)
 * (consecutive query heads share a KV head: the plainest reading of the GQA remark
 * in "序列并行与 Ring Attention" section "1. Ulysses"):
 *
 *   visible keys      j in [kv_lo, kv_hi), and j <= i when causal
 *                     ("Ring Attention explained", section "因果掩码处理": the
 *                      diagonal block is lower-triangular, i.e. key i is seen)
 *   s_j   = scale * sum_t q[b,h,i,t] * k[b,hk,j,t]
 *   M     = max_j s_j                    (first pass)
 *   Z     = sum_j exp(s_j - M)           (second pass)
 *   O[t]  = sum_j exp(s_j - M) v[b,hk,j,t] / Z
 *   LSE   = M + ln Z                     (natural log of the scaled scores'
 *                                         exp-sum, the quantity that the
 *                                         `update_out_and_lse` merge of the
 *                                         Twinkle page combines)
 *
 * A row with no visible key gets O = 0 and LSE = -inf: the identity of the merge.
 *
 * Inputs are contiguous [B, H, N, D] arrays of float32, float64 or bfloat16 bits
 * (uint16); every element is converted to double exactly before use.
 *
 * ORACLE_PLANT (compile-time, default 0) selects a deliberately wrong variant.
 * The pin tests build each variant and check that at least one pin rejects it.
 * The default build contains none of them.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_PLANT
#define ORACLE_PLANT 0
#endif

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F64 = 2 };

static double elem(const void *base, int dtype, int64_t idx) {
    if (dtype == ORACLE_F32) return (double)((const float *)base)[idx];
    if (dtype == ORACLE_BF16) {
        uint32_t bits = ((uint32_t)((const uint16_t *)base)[idx]) << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return ((const double *)base)[idx];
}

typedef struct {
    const void *q, *k, *v;
    int dtype;
    int64_t B, Hq, Hkv, N, D;
    int causal;
    double scale;
    int64_t kv_lo, kv_hi;
    const int64_t *rows; /* NULL: every row, in (b, h, i) order */
    int64_t nrows;
    double *o_out, *lse_out;
    int64_t next; /* shared work counter, guarded by mu */
    pthread_mutex_t mu;
} job_t;

/* One query row, two passes over its visible keys. */
static void attend_row(const job_t *J, int64_t b, int64_t h, int64_t i, double *qrow,
                       double *s, double *o, double *lse) {
    const int64_t D = J->D;
    const int64_t G = J->Hq / J->Hkv;
#if ORACLE_PLANT == 3
    const int64_t hk = h % J->Hkv; /* planted: wrong GQA head map */
#else
    const int64_t hk = h / G;
#endif
    const int64_t qbase = ((b * J->Hq + h) * J->N + i) * D;
    const int64_t kvhead = (b * J->Hkv + hk) * J->N;

    int64_t lo = J->kv_lo, hi = J->kv_hi;
#if ORACLE_PLANT == 2
    if (J->causal && i < hi) hi = i; /* planted: causal diagonal excluded */
#else
    if (J->causal && i + 1 < hi) hi = i + 1;
#endif
    for (int64_t t = 0; t < D; ++t) o[t] = 0.0;
    if (hi <= lo) {
        *lse = -INFINITY;
        return;
    }
    for (int64_t t = 0; t < D; ++t) qrow[t] = elem(J->q, J->dtype, qbase + t);

    /* pass 1: scaled scores and their maximum */
    double M = -INFINITY;
    for (int64_t j = lo; j < hi; ++j) {
        double acc = 0.0;
        for (int64_t t = 0; t < D; ++t) {
#if ORACLE_PLANT == 4
            /* planted: operands transposed (query row j against key row i) */
            acc += elem(J->q, J->dtype, ((b * J->Hq + h) * J->N + j) * D + t) *
                   elem(J->k, J->dtype, (kvhead + i) * D + t);
#else
            acc += qrow[t] * elem(J->k, J->dtype, (kvhead + j) * D + t);
#endif
        }
#if ORACLE_PLANT == 1
        s[j - lo] = acc; /* planted: scale dropped */
#else
        s[j - lo] = J->scale * acc;
#endif
        if (s[j - lo] > M) M = s[j - lo];
    }

    /* pass 2: exp-sum and weighted sum of value rows */
    double Z = 0.0;
    for (int64_t j = lo; j < hi; ++j) {
#if ORACLE_PLANT == 6
        const double w = exp(M - s[j - lo]); /* planted: sign of the shift flipped */
#else
        const double w = exp(s[j - lo] - M);
#endif
        Z += w;
        for (int64_t t = 0; t < D; ++t) o[t] += w * elem(J->v, J->dtype, (kvhead + j) * D + t);
    }
    for (int64_t t = 0; t < D; ++t) o[t] /= Z;
#if ORACLE_PLANT == 5
    *lse = log(Z); /* planted: maximum left out of the LSE */
#else
    *lse = M + log(Z);
#endif
}

static void *worker(void *arg) {
    job_t *J = (job_t *)arg;
    const int64_t span = J->kv_hi - J->kv_lo > 0 ? J->kv_hi - J->kv_lo : 1;
    double *qrow = (double *)malloc(sizeof(double) * (size_t)J->D);
    double *s = (double *)malloc(sizeof(double) * (size_t)span);
    for (;;) {
        pthread_mutex_lock(&J->mu);
        const int64_t r = J->next++;
        pthread_mutex_unlock(&J->mu);
        if (r >= J->nrows) break;
        int64_t b, h, i;
        if (J->rows) {
            b = J->rows[3 * r + 0];
            h = J->rows[3 * r + 1];
            i = J->rows[3 * r + 2];
        } else {
            i = r % J->N;
            h = (r / J->N) % J->Hq;
            b = r / (J->N * J->Hq);
        }
        attend_row(J, b, h, i, qrow, s, J->o_out + r * J->D, J->lse_out + r);
    }
    free(qrow);
    free(s);
    return NULL;
}

/*
 * Attention for a list of query rows (or for every row when rows == NULL).
 *   q:    [B, Hq, N, D] contiguous; k, v: [B, Hkv, N, D] contiguous
 *   dtype: 0 float32, 1 bfloat16 bits, 2 float64
 *   kv_lo, kv_hi: the window of key positions a row may see (before causality)
 *   rows: nrows triples (b, h, i), or NULL for all B*Hq*N rows in (b, h, i) order
 *   o_out: nrows x D doubles; lse_out: nrows doubles
 * Returns 0, or -1 on bad arguments.
 */
int oracle_attention_rows(const void *q, const void *k, const void *v, int dtype, int64_t B,
                          int64_t Hq, int64_t Hkv, int64_t N, int64_t D, int causal,
                          double scale, int64_t kv_lo, int64_t kv_hi, const int64_t *rows,
                          int64_t nrows, double *o_out, double *lse_out, int nthreads) {
    if (!q || !k || !v || !o_out || !lse_out) return -1;
    if (B < 0 || Hq < 1 || Hkv < 1 || N < 0 || D < 1 || Hq % Hkv != 0) return -1;
    if (dtype != ORACLE_F32 && dtype != ORACLE_BF16 && dtype != ORACLE_F64) return -1;
    if (kv_lo < 0) kv_lo = 0;
    if (kv_hi > N) kv_hi = N;
    if (!rows) nrows = B * Hq * N;
    for (int64_t r = 0; rows && r < nrows; ++r) {
        if (rows[3 * r] < 0 || rows[3 * r] >= B || rows[3 * r + 1] < 0 ||
            rows[3 * r + 1] >= Hq || rows[3 * r + 2] < 0 || rows[3 * r + 2] >= N)
            return -1;
    }
    if (nrows == 0) return 0;

    job_t J;
    memset(&J, 0, sizeof J);
    J.q = q;
    J.k = k;
    J.v = v;
    J.dtype = dtype;
    J.B = B;
    J.Hq = Hq;
    J.Hkv = Hkv;
    J.N = N;
    J.D = D;
    J.causal = causal;
    J.scale = scale;
    J.kv_lo = kv_lo;
    J.kv_hi = kv_hi;
    J.rows = rows;
    J.nrows = nrows;
    J.o_out = o_out;
    J.lse_out = lse_out;
    pthread_mutex_init(&J.mu, NULL);

    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > nrows) nthreads = (int)nrows;
    pthread_t tid[256];
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tid[started], NULL, worker, &J) == 0) ++started;
    }
    worker(&J);
    for (int t = 0; t < started; ++t) pthread_join(tid[t], NULL);
    pthread_mutex_destroy(&J.mu);
    return 0;
}

/* Which planted variant this compiled library is (0 = the real oracle). */
int oracle_plant(void) { return ORACLE_PLANT; }
