/*
 * oracle.c -- plain, slow, double-precision CPU reference for attention over a
 * paged KV cache.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg call it; the library never does.  It shares no
 * code, header or table with the CUDA path.
 *
 * What it computes (page titles of the subject's web pages):
 *  - "为什么Attention是O(n²)" (answer.freetools.me), section on the mathematics:
 *    Attention(Q,K,V) = softmax(Q K^T / sqrt(d_k)) V, evaluated here literally
 *    row by row: every score, then the row maximum, the exponentials, their
 *    sum, the weighted sum of V, and the division (two passes, no tiling).
 *  - "Flash Attention与Paged Attention如何共同优化大模型推理？" (ipipp.com):
 *    section 2, the causal flag of the library call (`is_causal=True`);
 *    section 3, the cache layout [num_blocks, 2, num_heads, block_size,
 *    head_dim] with K at index 0 and V at index 1 of the second axis.
 *  - "企业官网建设流程全解析" (cf-1.com), section 2.1: token i of a sequence lives
 *    in physical block block_table[i / block_size] at offset i % block_size.
 *  - The same page and the answer.freetools.me page (prefill / decode): a decode
 *    step appends the new token's K and V to the cache.
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - element address: row-major over [NB, 2, Hkv, bs, D];
 *  - under grouped-query attention the cache's head axis counts KV heads and
 *    query head h reads KV head h / (Hq / Hkv);
 *  - causal alignment: a chunk of q_len queries over a context of L tokens
 *    (the chunk's own tokens included) puts query r at absolute position
 *    L - q_len + r, which sees keys 0 .. L - q_len + r;
 *  - an empty context gives output 0 and lse = -inf.
 *
 * All fp16 / bf16 inputs are converted exactly to double.  The log-sum-exp of
 * the scaled scores (lse = M + ln sum exp(s_i - M)) is returned beside the
 * output; the split-KV merge is checked against it.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_F16 = 0, ORACLE_BF16 = 1 };

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
static double half_bits_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^-14 / 2^10 */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(f | 0x400), e - 25);    /* (1.f) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double to_double(int dtype, uint16_t h) {
    return dtype == ORACLE_BF16 ? bf16_bits_to_double(h) : half_bits_to_double(h);
}

/* Element offset of cache[pb][kv][h][off][0]. */
static size_t cache_row(int pb, int kv, int h, int off, int hkv, int bs, int d) {
    return ((((size_t)pb * 2 + kv) * hkv + h) * bs + off) * (size_t)d;
}

/* ------------------------------------------------------------------------- */
/* Append: for token t of sequence b (t-th of its new tokens), position
 * pos = ctx_before[b] + t, page = table[b][pos / bs], offset pos % bs;
 * copy the 16-bit patterns of K and V.  Returns 0, or -1 on an out-of-range
 * page id / table slot (nothing is written for that token). */
int oracle_kv_cache_append(uint16_t *cache, int nb, int hkv, int bs, int d,
                           const uint16_t *k_new, const uint16_t *v_new,
                           const int *cu_new_lens, const int *ctx_before,
                           const int *block_tables, int batch, int mb) {
    int rc = 0;
    for (int b = 0; b < batch; ++b) {
        for (int t = cu_new_lens[b]; t < cu_new_lens[b + 1]; ++t) {
            long pos = (long)ctx_before[b] + (t - cu_new_lens[b]);
            long logical = pos / bs;
            if (logical < 0 || logical >= mb) { rc = -1; continue; }
            int pb = block_tables[(size_t)b * mb + logical];
            if (pb < 0 || pb >= nb) { rc = -1; continue; }
            int off = (int)(pos % bs);
            for (int h = 0; h < hkv; ++h) {
                const uint16_t *ks = k_new + ((size_t)t * hkv + h) * d;
                const uint16_t *vs = v_new + ((size_t)t * hkv + h) * d;
                uint16_t *kd = cache + cache_row(pb, 0, h, off, hkv, bs, d);
                uint16_t *vd = cache + cache_row(pb, 1, h, off, hkv, bs, d);
                for (int e = 0; e < d; ++e) { kd[e] = ks[e]; vd[e] = vs[e]; }
            }
        }
    }
    return rc;
}

/* ------------------------------------------------------------------------- */
typedef struct {
    int dtype;
    const uint16_t *cache; int nb, hkv, bs, d;
    const uint16_t *q; int hq;
    const int *cu_q_lens, *context_lens, *block_tables; int batch, mb;
    double scale; int causal;
    const long *rows; long n_rows;        /* selected global query rows */
    double *out, *lse;                    /* [n_rows, hq, d], [n_rows, hq] */
    long next; pthread_mutex_t lock;      /* work counter over (row, head) */
    int status;
} attn_job;

/* One (query row, query head): the definition written out. */
static int attend_one(attn_job *J, long sel, int h, double *s, double *acc) {
    long row = J->rows ? J->rows[sel] : sel;
    int b = 0;
    while (b < J->batch && !(J->cu_q_lens[b] <= row && row < J->cu_q_lens[b + 1])) ++b;
    double *o = J->out + ((size_t)sel * J->hq + h) * J->d;
    double *lse = J->lse ? J->lse + (size_t)sel * J->hq + h : NULL;
    if (b == J->batch) return -1;
    int L = J->context_lens[b];
    int q_len = J->cu_q_lens[b + 1] - J->cu_q_lens[b];
    long r = row - J->cu_q_lens[b];
    long kmax = J->causal ? (long)L - q_len + r + 1 : L;
    if (kmax > L) kmax = L;
    int group = J->hq / J->hkv;
    int g = h / group;
    const uint16_t *qv = J->q + ((size_t)row * J->hq + h) * J->d;

    for (int e = 0; e < J->d; ++e) o[e] = 0.0;
    if (kmax <= 0) { if (lse) *lse = -INFINITY; return 0; }

    /* pass 1: scores */
    for (long i = 0; i < kmax; ++i) {
        long logical = i / J->bs;
        if (logical >= J->mb) return -1;
        int pb = J->block_tables[(size_t)b * J->mb + logical];
        if (pb < 0 || pb >= J->nb) return -1;
        const uint16_t *kr = J->cache + cache_row(pb, 0, g, (int)(i % J->bs), J->hkv, J->bs, J->d);
        double dot = 0.0;
        for (int e = 0; e < J->d; ++e) dot += to_double(J->dtype, qv[e]) * to_double(J->dtype, kr[e]);
        s[i] = J->scale * dot;
    }
    /* pass 2: max, exponentials, sum, weighted sum of V */
    double M = -INFINITY;
    for (long i = 0; i < kmax; ++i) if (s[i] > M) M = s[i];
    double sum = 0.0;
    for (int e = 0; e < J->d; ++e) acc[e] = 0.0;
    for (long i = 0; i < kmax; ++i) {
        double w = exp(s[i] - M);
        sum += w;
        int pb = J->block_tables[(size_t)b * J->mb + i / J->bs];
        const uint16_t *vr = J->cache + cache_row(pb, 1, g, (int)(i % J->bs), J->hkv, J->bs, J->d);
        for (int e = 0; e < J->d; ++e) acc[e] += w * to_double(J->dtype, vr[e]);
    }
    for (int e = 0; e < J->d; ++e) o[e] = acc[e] / sum;
    if (lse) *lse = M + log(sum);
    return 0;
}

static void *attn_worker(void *arg) {
    attn_job *J = (attn_job *)arg;
    long max_keys = 0;
    for (int b = 0; b < J->batch; ++b) if (J->context_lens[b] > max_keys) max_keys = J->context_lens[b];
    double *s = (double *)malloc(sizeof(double) * (size_t)(max_keys > 0 ? max_keys : 1));
    double *acc = (double *)malloc(sizeof(double) * (size_t)J->d);
    long total = J->n_rows * J->hq;
    for (;;) {
        long w;
        pthread_mutex_lock(&J->lock);
        w = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (w >= total) break;
        if (attend_one(J, w / J->hq, (int)(w % J->hq), s, acc) != 0) {
            pthread_mutex_lock(&J->lock);
            J->status = -1;
            pthread_mutex_unlock(&J->lock);
        }
    }
    free(s);
    free(acc);
    return NULL;
}

/* Paged attention for every selected query row and every query head.
 * Decode is the case q_len = 1 per sequence (causal or not: the one query
 * sees the whole context).  rows == NULL selects all rows 0..n_rows-1.
 * Returns 0, -1 on an out-of-range page id / table slot / row, -2 on bad
 * arguments. */
int oracle_paged_attention(int dtype, const uint16_t *cache, int nb, int hkv, int bs, int d,
                           const uint16_t *q, int hq, const int *cu_q_lens, const int *context_lens,
                           const int *block_tables, int batch, int mb, double scale, int causal,
                           const long *rows, long n_rows, double *out, double *lse, int nthreads) {
    if (hkv <= 0 || hq <= 0 || hq % hkv != 0 || d <= 0 || bs <= 0 || batch < 0) return -2;
    attn_job J;
    J.dtype = dtype; J.cache = cache; J.nb = nb; J.hkv = hkv; J.bs = bs; J.d = d;
    J.q = q; J.hq = hq; J.cu_q_lens = cu_q_lens; J.context_lens = context_lens;
    J.block_tables = block_tables; J.batch = batch; J.mb = mb; J.scale = scale; J.causal = causal;
    J.rows = rows; J.n_rows = n_rows; J.out = out; J.lse = lse; J.next = 0; J.status = 0;
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads == 1) {
        attn_worker(&J);
    } else {
        pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
        for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, attn_worker, &J);
        for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
        free(th);
    }
    pthread_mutex_destroy(&J.lock);
    return J.status;
}

/* ------------------------------------------------------------------------- */
/* Split-KV merge.  Each of n_rows rows has S partial results: O_s (already
 * divided by its own sum) and lse_s = log of that sum of exp(scores).  The
 * merged result is the softmax over the union of the splits' keys:
 *   M = max_s lse_s,  w_s = exp(lse_s - M),  O = sum_s w_s O_s / sum_s w_s,
 *   lse = M + log sum_s w_s.
 * A split with lse_s = -inf (no keys) has weight 0; if every split is empty
 * the output is 0 and lse = -inf.  Inputs are double here. */
int oracle_attn_combine(const double *partial_o, const double *partial_lse, long n_rows,
                        int num_splits, int d, double *out, double *lse) {
    for (long r = 0; r < n_rows; ++r) {
        const double *ls = partial_lse + (size_t)r * num_splits;
        double M = -INFINITY;
        for (int s = 0; s < num_splits; ++s) if (ls[s] > M) M = ls[s];
        double *o = out + (size_t)r * d;
        for (int e = 0; e < d; ++e) o[e] = 0.0;
        if (M == -INFINITY) { if (lse) lse[r] = -INFINITY; continue; }
        double wsum = 0.0;
        for (int s = 0; s < num_splits; ++s) {
            if (ls[s] == -INFINITY) continue;
            double w = exp(ls[s] - M);
            wsum += w;
            const double *os = partial_o + ((size_t)r * num_splits + s) * d;
            for (int e = 0; e < d; ++e) o[e] += w * os[e];
        }
        for (int e = 0; e < d; ++e) o[e] /= wsum;
        if (lse) lse[r] = M + log(wsum);
    }
    return 0;
}
