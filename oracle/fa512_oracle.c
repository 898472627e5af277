/*
 * fp64 reference for head-dim-512 attention: TEST INFRASTRUCTURE ONLY.
 *
 * This file is the oracle that the CUDA path is checked against.  Only the
 * tests, the smoke check and the benchmark's CPU-baseline leg may load it; the
 * library itself never calls it and shares no code with it.
 *
 * What it computes is the plain definition of softmax attention, written out
 * with no blocking, no online rescaling and no split of the key range:
 *
 *   s_j   = scale * sum_d q[d] * k_j[d]           for every visible key j
 *   m     = max_j s_j
 *   lse   = m + ln( sum_j exp(s_j - m) )
 *   o[d]  = sum_j exp(s_j - lse) * v_j[d]
 *   no visible key:  o = 0, lse = -inf
 *
 * Sources (page title, then the part of the page):
 *   - "Writing a FlashAttention Prefill Kernel for Gemma 4" (mila.toddt.me),
 *     opening section and "The starting point": a classical attention
 *     materialises the [chunk x attended_len] score matrix; flash attention
 *     reaches the same result without writing it.  The oracle materialises it.
 *   - "Flash-Decoding for MQA in CUDA" (mila.toddt.me), section "The test
 *     that catches what parity misses": an FP64 host reference over the same
 *     bf16-rounded inputs.  Inputs here are bf16 bit patterns, widened
 *     exactly to double.
 *   - Same page, section "One KV head breaks the textbook": a decode query
 *     reads the live band [max(0, len - window), len) of its sequence, with
 *     keys walked by absolute position.
 *   - vllm-project/flash-attention PR #199, review item F4: a row with no
 *     visible key returns LSE = -inf (and O = 0).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - query head h reads KV head h / G with G = n_q_heads / n_kv_heads
 *     (consecutive grouping);
 *   - query row i of a prefill sits at absolute position q_offset + i; with
 *     causal set, key j is visible iff j <= q_offset + i;
 *   - window > 0 keeps keys j > position - window (window keys including the
 *     query's own position); window <= 0 means no window;
 *   - lse is the natural log of sum_j exp(s_j), in units of the scaled logits;
 *   - a decode query sits at position kv_len - 1 of its sequence.
 *
 * Threads split the (row, head) pairs; every pair is computed independently
 * in fp64, so the result does not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bf16 -> double, exact: a bf16 value is the upper half of an IEEE binary32. */
static double bf16_to_double(uint16_t b)
{
    uint32_t bits = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/*
 * Attention of one query vector against an explicit list of key rows.
 * q: head_dim bf16 values.  key_rows/val_rows: pointers to the n_keys visible
 * key and value rows (head_dim bf16 values each).  Writes o[head_dim], *lse.
 * work: caller-provided scratch of n_keys doubles (the materialised scores).
 */
static void attend_one(const uint16_t *q, const uint16_t *const *key_rows,
                       const uint16_t *const *val_rows, int n_keys, int head_dim,
                       double scale, double *o, double *lse, double *s)
{
    int d, j;
    if (n_keys == 0) {
        for (d = 0; d < head_dim; ++d) o[d] = 0.0;
        *lse = -INFINITY;
        return;
    }
    /* scores */
    double m = -INFINITY;
    for (j = 0; j < n_keys; ++j) {
        double acc = 0.0;
        for (d = 0; d < head_dim; ++d)
            acc += bf16_to_double(q[d]) * bf16_to_double(key_rows[j][d]);
        s[j] = scale * acc;
        if (s[j] > m) m = s[j];
    }
    /* log-sum-exp */
    double sum = 0.0;
    for (j = 0; j < n_keys; ++j) sum += exp(s[j] - m);
    double l = m + log(sum);
    *lse = l;
    /* probabilities times values */
    for (d = 0; d < head_dim; ++d) o[d] = 0.0;
    for (j = 0; j < n_keys; ++j) {
        double p = exp(s[j] - l);
        const uint16_t *vr = val_rows[j];
        for (d = 0; d < head_dim; ++d) o[d] += p * bf16_to_double(vr[d]);
    }
}

/*
 * One OCP FP8 E4M3 value (the "e4m3fn" encoding): 1 sign bit, 4 exponent
 * bits with bias 7, 3 mantissa bits; exponent field 0 holds the subnormals
 * m/8 * 2^-6; there are no infinities and S.1111.111 is NaN, so the largest
 * finite value is 1.75 * 2^8 = 448.
 */
static double e4m3_to_double(uint8_t x)
{
    const int sign = x >> 7, e = (x >> 3) & 15, m = x & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/*
 * attend_one over an FP8 cache: key and value element d of a row are
 * k_scale * e4m3(k[d]) and v_scale * e4m3(v[d]) (per-tensor scales), widened
 * to double before use; everything else is attend_one, term for term.
 */
static void attend_one_fp8(const uint16_t *q, const uint8_t *const *key_rows,
                           const uint8_t *const *val_rows, int n_keys, int head_dim,
                           double scale, double k_scale, double v_scale, double *o,
                           double *lse, double *s)
{
    int d, j;
    if (n_keys == 0) {
        for (d = 0; d < head_dim; ++d) o[d] = 0.0;
        *lse = -INFINITY;
        return;
    }
    double m = -INFINITY;
    for (j = 0; j < n_keys; ++j) {
        double acc = 0.0;
        for (d = 0; d < head_dim; ++d)
            acc += bf16_to_double(q[d]) * (k_scale * e4m3_to_double(key_rows[j][d]));
        s[j] = scale * acc;
        if (s[j] > m) m = s[j];
    }
    double sum = 0.0;
    for (j = 0; j < n_keys; ++j) sum += exp(s[j] - m);
    double l = m + log(sum);
    *lse = l;
    for (d = 0; d < head_dim; ++d) o[d] = 0.0;
    for (j = 0; j < n_keys; ++j) {
        double p = exp(s[j] - l);
        const uint8_t *vr = val_rows[j];
        for (d = 0; d < head_dim; ++d) o[d] += p * (v_scale * e4m3_to_double(vr[d]));
    }
}

/* All 256 E4M3 codes decoded, for the tests that pin the decoding itself. */
void oracle_e4m3_table(double *out)
{
    for (int i = 0; i < 256; ++i) out[i] = e4m3_to_double((uint8_t)i);
}

/* ------------------------------------------------------------------ prefill */

typedef struct {
    const uint16_t *q, *k, *v;
    double *out, *lse;
    int seqlen_q, seqlen_k, q_offset, n_q_heads, n_kv_heads, head_dim;
    double scale;
    int causal, window;
    const int *rows;
    int n_rows;
    int n_threads, tid;
} prefill_job;

/* Visible key interval [lo, hi) of the query at absolute position p. */
static void visible_range(long p, int seqlen_k, int causal, int window, long *lo, long *hi)
{
    long a = 0, b = seqlen_k;
    if (causal && p + 1 < b) b = p + 1;
    if (window > 0 && p - window + 1 > a) a = p - window + 1;
    if (b < a) b = a;
    *lo = a;
    *hi = b;
}

static void *prefill_worker(void *arg)
{
    prefill_job *J = (prefill_job *)arg;
    const int D = J->head_dim;
    const int G = J->n_q_heads / J->n_kv_heads;
    const uint16_t **krows = (const uint16_t **)malloc(sizeof(void *) * (size_t)(J->seqlen_k + 1));
    const uint16_t **vrows = (const uint16_t **)malloc(sizeof(void *) * (size_t)(J->seqlen_k + 1));
    double *s = (double *)malloc(sizeof(double) * (size_t)(J->seqlen_k + 1));
    long total = (long)J->n_rows * J->n_q_heads;
    for (long w = J->tid; w < total; w += J->n_threads) {
        int r = (int)(w / J->n_q_heads);
        int h = (int)(w % J->n_q_heads);
        int i = J->rows ? J->rows[r] : r;
        int hk = h / G;
        long p = (long)J->q_offset + i;
        long lo, hi;
        visible_range(p, J->seqlen_k, J->causal, J->window, &lo, &hi);
        int n = 0;
        for (long j = lo; j < hi; ++j, ++n) {
            krows[n] = J->k + ((size_t)j * J->n_kv_heads + hk) * D;
            vrows[n] = J->v + ((size_t)j * J->n_kv_heads + hk) * D;
        }
        const uint16_t *qr = J->q + ((size_t)i * J->n_q_heads + h) * D;
        double *o = J->out + ((size_t)r * J->n_q_heads + h) * D;
        double *l = J->lse + (size_t)h * J->n_rows + r;
        attend_one(qr, krows, vrows, n, D, J->scale, o, l, s);
    }
    free(krows);
    free(vrows);
    free(s);
    return NULL;
}

/*
 * q   [seqlen_q, n_q_heads, head_dim]   bf16 bits
 * k,v [seqlen_k, n_kv_heads, head_dim]  bf16 bits
 * rows: NULL for every query row, else n_rows row indices into q.
 * out [n_rows, n_q_heads, head_dim] fp64;  lse [n_q_heads, n_rows] fp64.
 * Returns 0, or -1 on invalid arguments.
 */
int oracle_prefill(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                   double *out, double *lse, int seqlen_q, int seqlen_k, int q_offset,
                   int n_q_heads, int n_kv_heads, int head_dim, double scale, int causal,
                   int window, const int *rows, int n_rows, int n_threads)
{
    if (seqlen_q < 0 || seqlen_k < 0 || n_q_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0)
        return -1;
    if (n_q_heads % n_kv_heads != 0) return -1;
    if (!rows) n_rows = seqlen_q;
    if (rows)
        for (int r = 0; r < n_rows; ++r)
            if (rows[r] < 0 || rows[r] >= seqlen_q) return -1;
    if (n_threads < 1) n_threads = 1;
    prefill_job *jobs = (prefill_job *)calloc((size_t)n_threads, sizeof(prefill_job));
    pthread_t *th = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    for (int t = 0; t < n_threads; ++t) {
        prefill_job J = {q, k, v, out, lse, seqlen_q, seqlen_k, q_offset, n_q_heads,
                         n_kv_heads, head_dim, scale, causal, window, rows, n_rows,
                         n_threads, t};
        jobs[t] = J;
        pthread_create(&th[t], NULL, prefill_worker, &jobs[t]);
    }
    for (int t = 0; t < n_threads; ++t) pthread_join(th[t], NULL);
    free(jobs);
    free(th);
    return 0;
}

/* ------------------------------------------------------------- paged decode */

typedef struct {
    const uint16_t *q, *kp, *vp;
    const int *page_table, *kv_lens;
    double *out, *lse;
    int batch, n_q_heads, n_kv_heads, head_dim, page_size, max_pages;
    double scale;
    int window;
    int n_threads, tid;
    int max_len;
    int q_len;
    /* FP8 cache (kp, vp unused): e4m3 bytes and their per-tensor scales */
    const uint8_t *kp8, *vp8;
    double k_scale, v_scale;
} decode_job;

static void *decode_worker(void *arg)
{
    decode_job *J = (decode_job *)arg;
    const int D = J->head_dim;
    const int G = J->n_q_heads / J->n_kv_heads;
    const uint16_t **krows = (const uint16_t **)malloc(sizeof(void *) * (size_t)(J->max_len + 1));
    const uint16_t **vrows = (const uint16_t **)malloc(sizeof(void *) * (size_t)(J->max_len + 1));
    const uint8_t **krows8 = (const uint8_t **)malloc(sizeof(void *) * (size_t)(J->max_len + 1));
    const uint8_t **vrows8 = (const uint8_t **)malloc(sizeof(void *) * (size_t)(J->max_len + 1));
    double *s = (double *)malloc(sizeof(double) * (size_t)(J->max_len + 1));
    long total = (long)J->batch * J->q_len * J->n_q_heads;
    for (long w = J->tid; w < total; w += J->n_threads) {
        int bt = (int)(w / J->n_q_heads);      /* b * q_len + t */
        int h = (int)(w % J->n_q_heads);
        int b = bt / J->q_len;
        int t = bt % J->q_len;
        int hk = h / G;
        int len = J->kv_lens[b];
        /* the q_len queries are the sequence's last q_len positions:
           query t sits at len - q_len + t (negative: no key is visible) */
        long p = (long)len - J->q_len + t;
        long lo, hi;
        visible_range(p, len, 1, J->window, &lo, &hi);
        if (p < 0) hi = lo = 0;
        int n = 0;
        for (long j = lo; j < hi; ++j, ++n) {
            /* logical position j lives in page page_table[b][j / page_size],
               slot j % page_size */
            int page = J->page_table[(size_t)b * J->max_pages + j / J->page_size];
            int slot = (int)(j % J->page_size);
            size_t row = ((size_t)page * J->page_size + slot) * J->n_kv_heads + hk;
            if (J->kp8) {
                krows8[n] = J->kp8 + row * D;
                vrows8[n] = J->vp8 + row * D;
            } else {
                krows[n] = J->kp + row * D;
                vrows[n] = J->vp + row * D;
            }
        }
        const uint16_t *qr = J->q + ((size_t)bt * J->n_q_heads + h) * D;
        double *o = J->out + ((size_t)bt * J->n_q_heads + h) * D;
        double *l = J->lse + (size_t)bt * J->n_q_heads + h;
        if (J->kp8)
            attend_one_fp8(qr, krows8, vrows8, n, D, J->scale, J->k_scale, J->v_scale, o, l, s);
        else
            attend_one(qr, krows, vrows, n, D, J->scale, o, l, s);
    }
    free(krows);
    free(vrows);
    free(krows8);
    free(vrows8);
    free(s);
    return NULL;
}

/*
 * q        [batch, n_q_heads, head_dim]                      bf16 bits
 * k_pages  [num_pages, page_size, n_kv_heads, head_dim]      bf16 bits
 * v_pages  same layout as k_pages
 * page_table [batch, max_pages_per_seq] int32 page indices
 * kv_lens  [batch] int32 live lengths
 * out [batch, n_q_heads, head_dim] fp64;  lse [batch, n_q_heads] fp64.
 * Returns 0, or -1 on invalid arguments (including a page index or length
 * outside the table; num_pages bounds the page indices).
 */
int oracle_decode_paged_q(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                          const int *page_table, const int *kv_lens, double *out, double *lse,
                          int batch, int q_len, int n_q_heads, int n_kv_heads, int head_dim,
                          int page_size, int max_pages_per_seq, int num_pages, double scale,
                          int window, int n_threads);

int oracle_decode_paged(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                        const int *page_table, const int *kv_lens, double *out, double *lse,
                        int batch, int n_q_heads, int n_kv_heads, int head_dim, int page_size,
                        int max_pages_per_seq, int num_pages, double scale, int window,
                        int n_threads)
{
    return oracle_decode_paged_q(q, k_pages, v_pages, page_table, kv_lens, out, lse, batch, 1,
                                 n_q_heads, n_kv_heads, head_dim, page_size, max_pages_per_seq,
                                 num_pages, scale, window, n_threads);
}

/*
 * Several query tokens per sequence (draft tokens being verified, a short
 * chunk appended to a paged cache): the q_len queries of sequence b are its
 * last q_len positions, query t at position kv_lens[b] - q_len + t, each
 * causal over the cache (and windowed like any query).
 * q   [batch, q_len, n_q_heads, head_dim]   bf16 bits
 * out [batch, q_len, n_q_heads, head_dim] fp64;  lse [batch, q_len, n_q_heads] fp64.
 * Other arguments as oracle_decode_paged; q_len = 1 is that function.
 */
static int run_decode(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                      const uint8_t *k_pages8, const uint8_t *v_pages8, double k_scale,
                      double v_scale, const int *page_table, const int *kv_lens, double *out,
                      double *lse, int batch, int q_len, int n_q_heads, int n_kv_heads,
                      int head_dim, int page_size, int max_pages_per_seq, int num_pages,
                      double scale, int window, int n_threads);

int oracle_decode_paged_q(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                          const int *page_table, const int *kv_lens, double *out, double *lse,
                          int batch, int q_len, int n_q_heads, int n_kv_heads, int head_dim,
                          int page_size, int max_pages_per_seq, int num_pages, double scale,
                          int window, int n_threads)
{
    return run_decode(q, k_pages, v_pages, NULL, NULL, 1.0, 1.0, page_table, kv_lens, out, lse,
                      batch, q_len, n_q_heads, n_kv_heads, head_dim, page_size,
                      max_pages_per_seq, num_pages, scale, window, n_threads);
}

/*
 * Decode of q_len query tokens per sequence over an FP8 E4M3 paged cache
 * (vllm-project/flash-attention PR #199, "Summary": the paged KV cache in
 * FP8).  k_pages / v_pages hold one e4m3 byte per element in the layout of
 * oracle_decode_paged; a key element is k_scale * e4m3(byte), a value
 * element v_scale * e4m3(byte).  Other arguments as oracle_decode_paged_q.
 */
int oracle_decode_paged_fp8(const uint16_t *q, const uint8_t *k_pages, const uint8_t *v_pages,
                            const int *page_table, const int *kv_lens, double *out, double *lse,
                            int batch, int q_len, int n_q_heads, int n_kv_heads, int head_dim,
                            int page_size, int max_pages_per_seq, int num_pages, double scale,
                            double k_scale, double v_scale, int window, int n_threads)
{
    if (!k_pages || !v_pages) return -1;
    return run_decode(q, NULL, NULL, k_pages, v_pages, k_scale, v_scale, page_table, kv_lens,
                      out, lse, batch, q_len, n_q_heads, n_kv_heads, head_dim, page_size,
                      max_pages_per_seq, num_pages, scale, window, n_threads);
}

static int run_decode(const uint16_t *q, const uint16_t *k_pages, const uint16_t *v_pages,
                      const uint8_t *k_pages8, const uint8_t *v_pages8, double k_scale,
                      double v_scale, const int *page_table, const int *kv_lens, double *out,
                      double *lse, int batch, int q_len, int n_q_heads, int n_kv_heads,
                      int head_dim, int page_size, int max_pages_per_seq, int num_pages,
                      double scale, int window, int n_threads)
{
    if (batch < 0 || q_len < 1 || n_q_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 ||
        page_size <= 0)
        return -1;
    if (n_q_heads % n_kv_heads != 0) return -1;
    int max_len = 0;
    for (int b = 0; b < batch; ++b) {
        int len = kv_lens[b];
        if (len < 0 || len > max_pages_per_seq * page_size) return -1;
        if (len > max_len) max_len = len;
        int np = (len + page_size - 1) / page_size;
        for (int p = 0; p < np; ++p) {
            int pg = page_table[(size_t)b * max_pages_per_seq + p];
            if (pg < 0 || pg >= num_pages) return -1;
        }
    }
    if (n_threads < 1) n_threads = 1;
    decode_job *jobs = (decode_job *)calloc((size_t)n_threads, sizeof(decode_job));
    pthread_t *th = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    for (int t = 0; t < n_threads; ++t) {
        decode_job J = {q, k_pages, v_pages, page_table, kv_lens, out, lse, batch,
                        n_q_heads, n_kv_heads, head_dim, page_size, max_pages_per_seq,
                        scale, window, n_threads, t, max_len, q_len,
                        k_pages8, v_pages8, k_scale, v_scale};
        jobs[t] = J;
        pthread_create(&th[t], NULL, decode_worker, &jobs[t]);
    }
    for (int t = 0; t < n_threads; ++t) pthread_join(th[t], NULL);
    free(jobs);
    free(th);
    return 0;
}
