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
 *
 * FP8 cache (the "KV cache compression" the answer.freetools.me page names,
 * with no scheme given; reading listed in the design notes): every cached row
 * (one token's K or V of one KV head, head_dim values) is stored as OCP FP8
 * E4M3 codes with one FP32 scale, scale = amax / 448 and code = round-to-
 * nearest-even, saturating, of x * (448 / amax), all in binary32 arithmetic;
 * an all-zero row stores scale 0 and zero codes.  The attention reads each
 * element as decode(code) * scale, exactly, in double.
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

/* OCP FP8 E4M3 ("FN" variant): 1 sign, 4 exponent (bias 7), 3 fraction bits;
 * no infinities, S.1111.111 is NaN, largest finite (1 + 6/8) * 2^8 = 448;
 * exponent field 0 holds the subnormals m * 2^-9. */
static double e4m3_to_double(uint8_t c) {
    int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) v = NAN;
    else if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp((double)(8 + m), e - 10);   /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* Nearest E4M3 value, ties to the even fraction, magnitudes beyond 448
 * saturated to 448 (a finite input never gives NaN). */
static uint8_t double_to_e4m3(double x) {
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a >= 448.0) return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {                   /* subnormal spacing 2^-9 */
        double q = rint(a * 512.0);             /* exact scaling; rint rounds ties to even */
        return sign | (uint8_t)q;               /* q = 8 is the smallest normal, code 0x08 */
    }
    int e2;
    frexp(a, &e2);                              /* a in [2^(e2-1), 2^e2) */
    int e = e2 - 1;
    double r = rint(ldexp(a, 3 - e)) - 8.0;     /* fraction in eighths, rounded */
    if (r == 8.0) { r = 0.0; e += 1; }
    if (e > 8 || (e == 8 && r > 6.0)) return sign | 0x7E;
    return sign | (uint8_t)(((e + 7) << 3) | (int)r);
}

void oracle_e4m3_encode(const float *x, uint8_t *codes, long n) {
    for (long i = 0; i < n; ++i) codes[i] = double_to_e4m3((double)x[i]);
}

void oracle_e4m3_decode(const uint8_t *codes, double *x, long n) {
    for (long i = 0; i < n; ++i) x[i] = e4m3_to_double(codes[i]);
}

/* Quantise one row of d values (binary32 arithmetic throughout). */
static float quantise_row(int dtype, const uint16_t *src, uint8_t *dst, int d) {
    float amax = 0.0f;
    for (int e = 0; e < d; ++e) {
        float a = fabsf((float)to_double(dtype, src[e]));
        if (a > amax) amax = a;
    }
    if (amax == 0.0f) {
        for (int e = 0; e < d; ++e) dst[e] = 0;
        return 0.0f;
    }
    float scale = amax / 448.0f;
    float inv = 448.0f / amax;
    for (int e = 0; e < d; ++e) {
        float y = (float)to_double(dtype, src[e]) * inv;
        dst[e] = double_to_e4m3((double)y);
    }
    return scale;
}

/* Element offset of cache[pb][kv][h][off][0]. */
static size_t cache_row(int pb, int kv, int h, int off, int hkv, int bs, int d) {
    return ((((size_t)pb * 2 + kv) * hkv + h) * bs + off) * (size_t)d;
}

/* ------------------------------------------------------------------------- */
/* Append: for token t of sequence b (t-th of its new tokens), position
 * pos = ctx_before[b] + t, page = table[b][pos / bs], offset pos % bs; `row`
 * writes token t's K and V rows of every head there.  Returns 0, or -1 on an
 * out-of-range page id / table slot (nothing is written for that token). */
typedef void (*append_row_fn)(void *ctx, int t, int pb, int off);

static int append_walk(int nb, int bs, const int *cu_new_lens, const int *ctx_before, const int *block_tables,
                       int batch, int mb, append_row_fn row, void *ctx) {
    int rc = 0;
    for (int b = 0; b < batch; ++b) {
        for (int t = cu_new_lens[b]; t < cu_new_lens[b + 1]; ++t) {
            long pos = (long)ctx_before[b] + (t - cu_new_lens[b]);
            long logical = pos / bs;
            if (logical < 0 || logical >= mb) { rc = -1; continue; }
            int pb = block_tables[(size_t)b * mb + logical];
            if (pb < 0 || pb >= nb) { rc = -1; continue; }
            row(ctx, t, pb, (int)(pos % bs));
        }
    }
    return rc;
}

typedef struct {
    int hkv, bs, d, dtype;
    const uint16_t *k_new, *v_new;
    uint16_t *cache;                  /* native: 16-bit patterns copied */
    uint8_t *codes; float *scales;    /* FP8: quantised */
} append_job;

/* Native cache: copy the 16-bit patterns of K and V. */
static void copy_rows(void *ctx, int t, int pb, int off) {
    append_job *A = (append_job *)ctx;
    for (int h = 0; h < A->hkv; ++h) {
        const uint16_t *ks = A->k_new + ((size_t)t * A->hkv + h) * A->d;
        const uint16_t *vs = A->v_new + ((size_t)t * A->hkv + h) * A->d;
        uint16_t *kd = A->cache + cache_row(pb, 0, h, off, A->hkv, A->bs, A->d);
        uint16_t *vd = A->cache + cache_row(pb, 1, h, off, A->hkv, A->bs, A->d);
        for (int e = 0; e < A->d; ++e) { kd[e] = ks[e]; vd[e] = vs[e]; }
    }
}

/* FP8 cache: quantise each K and V row, store its codes and scale. */
static void quantise_rows(void *ctx, int t, int pb, int off) {
    append_job *A = (append_job *)ctx;
    for (int h = 0; h < A->hkv; ++h) {
        for (int kv = 0; kv < 2; ++kv) {
            const uint16_t *src = (kv == 0 ? A->k_new : A->v_new) + ((size_t)t * A->hkv + h) * A->d;
            size_t row = cache_row(pb, kv, h, off, A->hkv, A->bs, A->d);
            A->scales[row / (size_t)A->d] = quantise_row(A->dtype, src, A->codes + row, A->d);
        }
    }
}

int oracle_kv_cache_append(uint16_t *cache, int nb, int hkv, int bs, int d,
                           const uint16_t *k_new, const uint16_t *v_new,
                           const int *cu_new_lens, const int *ctx_before,
                           const int *block_tables, int batch, int mb) {
    append_job A = {hkv, bs, d, 0, k_new, v_new, cache, NULL, NULL};
    return append_walk(nb, bs, cu_new_lens, ctx_before, block_tables, batch, mb, copy_rows, &A);
}

/* The same walk into an FP8 cache: codes [NB, 2, Hkv, bs, D] bytes, scales
 * [NB, 2, Hkv, bs] FP32; each new row is quantised as described above. */
int oracle_kv_cache_append_fp8(uint8_t *codes, float *scales, int nb, int hkv, int bs, int d, int dtype,
                               const uint16_t *k_new, const uint16_t *v_new,
                               const int *cu_new_lens, const int *ctx_before,
                               const int *block_tables, int batch, int mb) {
    append_job A = {hkv, bs, d, dtype, k_new, v_new, NULL, codes, scales};
    return append_walk(nb, bs, cu_new_lens, ctx_before, block_tables, batch, mb, quantise_rows, &A);
}

/* ------------------------------------------------------------------------- */
typedef struct {
    int dtype;
    const uint16_t *cache; int nb, hkv, bs, d;
    const uint8_t *codes; const float *scales;   /* FP8 cache (cache == NULL) */
    const uint16_t *q; int hq;
    const int *cu_q_lens, *context_lens, *block_tables; int batch, mb;
    double scale; int causal;
    const long *rows; long n_rows;        /* selected global query rows */
    double *out, *lse;                    /* [n_rows, hq, d], [n_rows, hq] */
    long next; pthread_mutex_t lock;      /* work counter over (row, head) */
    int status;
} attn_job;

/* Element e of the cached row starting at element offset `row`. */
static double kv_elem(const attn_job *J, size_t row, int e) {
    if (J->codes) return e4m3_to_double(J->codes[row + e]) * (double)J->scales[row / (size_t)J->d];
    return to_double(J->dtype, J->cache[row + e]);
}

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
        size_t kr = cache_row(pb, 0, g, (int)(i % J->bs), J->hkv, J->bs, J->d);
        double dot = 0.0;
        for (int e = 0; e < J->d; ++e) dot += to_double(J->dtype, qv[e]) * kv_elem(J, kr, e);
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
        size_t vr = cache_row(pb, 1, g, (int)(i % J->bs), J->hkv, J->bs, J->d);
        for (int e = 0; e < J->d; ++e) acc[e] += w * kv_elem(J, vr, e);
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
static int run_attention(attn_job *J, int nthreads);

int oracle_paged_attention(int dtype, const uint16_t *cache, int nb, int hkv, int bs, int d,
                           const uint16_t *q, int hq, const int *cu_q_lens, const int *context_lens,
                           const int *block_tables, int batch, int mb, double scale, int causal,
                           const long *rows, long n_rows, double *out, double *lse, int nthreads) {
    if (hkv <= 0 || hq <= 0 || hq % hkv != 0 || d <= 0 || bs <= 0 || batch < 0) return -2;
    attn_job J;
    J.dtype = dtype; J.cache = cache; J.codes = NULL; J.scales = NULL;
    J.nb = nb; J.hkv = hkv; J.bs = bs; J.d = d;
    J.q = q; J.hq = hq; J.cu_q_lens = cu_q_lens; J.context_lens = context_lens;
    J.block_tables = block_tables; J.batch = batch; J.mb = mb; J.scale = scale; J.causal = causal;
    J.rows = rows; J.n_rows = n_rows; J.out = out; J.lse = lse;
    return run_attention(&J, nthreads);
}

/* The same attention over an FP8 cache (q in dtype). */
int oracle_paged_attention_fp8(int dtype, const uint8_t *codes, const float *scales, int nb, int hkv, int bs,
                               int d, const uint16_t *q, int hq, const int *cu_q_lens, const int *context_lens,
                               const int *block_tables, int batch, int mb, double scale, int causal,
                               const long *rows, long n_rows, double *out, double *lse, int nthreads) {
    if (hkv <= 0 || hq <= 0 || hq % hkv != 0 || d <= 0 || bs <= 0 || batch < 0) return -2;
    attn_job J;
    J.dtype = dtype; J.cache = NULL; J.codes = codes; J.scales = scales;
    J.nb = nb; J.hkv = hkv; J.bs = bs; J.d = d;
    J.q = q; J.hq = hq; J.cu_q_lens = cu_q_lens; J.context_lens = context_lens;
    J.block_tables = block_tables; J.batch = batch; J.mb = mb; J.scale = scale; J.causal = causal;
    J.rows = rows; J.n_rows = n_rows; J.out = out; J.lse = lse;
    return run_attention(&J, nthreads);
}

static int run_attention(attn_job *J0, int nthreads) {
    attn_job J = *J0;
    J.next = 0; J.status = 0;
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
