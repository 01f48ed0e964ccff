/*
 * oracle.c — plain, slow, fp64 CPU oracle for paged-KV attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  It shares no code, header,
 * table or helper with the CUDA library, and the CUDA library never calls it.
 *
 * What it computes (all in double precision, from inputs widened exactly from
 * their stored fp32 / fp16 / bf16 encodings):
 *
 *   oracle_paged_decode — single-query attention of sequence s, head h over the
 *     keys j in [start_s, ctx_s), each key gathered through the sequence's
 *     block table:
 *         x_j  = scale * (q . K_j + A[s,h,j])           (A absent -> 0)
 *         out  = sum_j softmax(x)_j V_j
 *     This is the formula of "PagedAttention: Support custom attention bias
 *     for T5 model (1/2)", opening section: softmax((QK^T + A)/sqrt(d_k)) V,
 *     with 1/sqrt(d_k) generalised to a caller-given scale that multiplies
 *     the bias too.  A is the fully materialised bias padded to a row stride
 *     (same page, first comment); a NULL A means no bias (same page, the
 *     review answer on the optional pointer).  The block table is whichever
 *     one the caller passes: decoder self-attention and encoder
 *     cross-attention each have their own ("Add Encoder-decoder model support
 *     and T5 Model support", the comments settling on two block tables).
 *     start_s = max(0, ctx_s - W) for a window W > 0, else 0: the query is the
 *     last token (position ctx_s - 1) and keeps the W most recent keys,
 *     itself included ("[V1] Add sliding window support to Flex Attention
 *     backend", causal sliding window).  ctx_s = 0 gives a zero row.
 *
 *   oracle_paged_decode_t5 — the same with A[s,h,j] taken from a T5 relative-
 *     position table, bias_table[h, min(ctx_s - 1 - j, num_buckets - 1)], in
 *     place of a materialised A (the in-kernel T5 bias the same page proposes).
 *
 *   oracle_prefill — for every query row i of a packed variable-length batch
 *     (cu_seqlens), softmax attention over the keys j of the same sequence
 *     that the mask keeps, with r, c the positions inside the sequence:
 *         window <= 0, causal = 0 : all j
 *         window <= 0, causal = 1 : c <= r
 *         window  > 0, causal = 0 : |r - c| < window   (bidirectional band)
 *         window  > 0, causal = 1 : 0 <= r - c < window
 *     ("[V1] Add sliding window support to Flex Attention backend":
 *     bidirectional attention with a sliding window for encoder-only models.)
 *
 *   oracle_prefill_chunked — the same with keys restricted to the query's
 *     own chunk of `chunk` positions (chunked local attention, same page).
 *
 *   oracle_prefill_biased — oracle_prefill with an additive relative-position
 *     bias inside the softmax, x = scale * (q . k + A) as in the formula above,
 *     where A depends only on the signed distance d = r - c between the query
 *     and key positions and saturates at num_buckets - 1 in either direction:
 *         A[h, r, c] = rel_bias[h, (num_buckets - 1) + clamp(d, -(num_buckets - 1), num_buckets - 1)]
 *     rel_bias is [H, 2 * num_buckets - 1].  This is the T5 bias of an
 *     encoder's bidirectional self-attention ("Add Encoder-decoder model
 *     support and T5 Model support": T5 adds a custom bias in its attention;
 *     "PagedAttention: Support custom attention bias for T5 model (1/2)": the
 *     distance is capped and larger distances reuse the last value).  A causal
 *     layer only reads the non-negative half, which is the decode table.
 *
 *   oracle_paged_prefill — prefill of the newest tokens of each sequence
 *     against keys held in the paged cache ("Add Encoder-decoder model
 *     support and T5 Model support": prompt and generated tokens keep their KV
 *     blocks apart, and prefill as well as decode kernels read cross-attention
 *     keys through their block table).  Sequence s has Lq_s query rows
 *     (cu_seqlens_q) and ctx_s keys (context_lens) behind block-table row s;
 *     query row r sits at key position p = ctx_s - Lq_s + r (the queries are
 *     the last Lq_s tokens, already written to the cache).  The mask is
 *     oracle_prefill's with r replaced by p and keys c in [0, ctx_s); the
 *     optional bias is oracle_prefill_biased's with d = p - c.  With
 *     causal = 0 and no window or bias, p plays no part: every query attends
 *     to all ctx_s keys (a decoder prompt's cross-attention to the encoder).
 *
 *   oracle_reshape_and_cache — the plain scatter of token rows into cache
 *     blocks, cache[slot / bs, h, slot % bs, :] = key[t, h, :]; slot < 0 skips
 *     the token.  Byte copies, so the result is exact.
 *
 * Cache layout (both oracle and library): [num_blocks, H, block_size, D].
 *
 * Work is spread over plain pthreads by (sequence, head) or (row, head); every
 * output element is computed by exactly one thread in a fixed order, so the
 * result does not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2 };

/* ---- exact widening of the storage encodings ---------------------------- */

static double half_bits_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int mant = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)mant, -24);                 /* zero / subnormal */
    else if (expo == 31)
        v = mant ? NAN : INFINITY;
    else
        v = ldexp((double)(mant | 0x400), expo - 25);  /* (1.m) * 2^(e-15) */
    return sign ? -v : v;
}

static double bf16_bits_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double load_elem(const void *base, size_t idx, int dtype)
{
    switch (dtype) {
    case ORC_F32: return (double)((const float *)base)[idx];
    case ORC_F16: return half_bits_to_double(((const uint16_t *)base)[idx]);
    default:      return bf16_bits_to_double(((const uint16_t *)base)[idx]);
    }
}

/* exported for the tests that pin the widening against numpy */
double oracle_widen(const void *base, long long idx, int dtype)
{
    return load_elem(base, (size_t)idx, dtype);
}

/* ---- a tiny thread pool: run fn(i, ctx) for i in [0, n) ----------------- */

typedef void (*item_fn)(long long i, void *ctx);

struct pool_arg {
    item_fn fn;
    void *ctx;
    long long n;
    int tid, nthreads;
};

static void *pool_worker(void *p)
{
    struct pool_arg *a = (struct pool_arg *)p;
    for (long long i = a->tid; i < a->n; i += a->nthreads)
        a->fn(i, a->ctx);
    return NULL;
}

static void run_items(item_fn fn, void *ctx, long long n, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (n < nthreads) nthreads = (int)(n > 0 ? n : 1);
    pthread_t th[256];
    struct pool_arg args[256];
    for (int t = 0; t < nthreads; ++t) {
        args[t].fn = fn; args[t].ctx = ctx; args[t].n = n;
        args[t].tid = t; args[t].nthreads = nthreads;
    }
    for (int t = 1; t < nthreads; ++t)
        pthread_create(&th[t], NULL, pool_worker, &args[t]);
    pool_worker(&args[0]);
    for (int t = 1; t < nthreads; ++t)
        pthread_join(th[t], NULL);
}

/* ---- softmax-weighted sum over an explicit list of logits --------------- */

/* out[d] = sum_j exp(x_j - max x) V_j[d] / sum_j exp(x_j - max x).
 * vrow(j) gives the element index of row j's first value.  n == 0 -> zeros. */
static void softmax_combine(double *out, const double *x, const size_t *vrow, int n,
                            const void *v, int dtype, int D)
{
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (n == 0) return;
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) if (x[j] > m) m = x[j];
    double l = 0.0;
    for (int j = 0; j < n; ++j) {
        double p = exp(x[j] - m);
        l += p;
        for (int d = 0; d < D; ++d) out[d] += p * load_elem(v, vrow[j] + d, dtype);
    }
    for (int d = 0; d < D; ++d) out[d] /= l;
}

/* ---- paged decode -------------------------------------------------------- */

struct decode_ctx {
    double *out;
    const void *q, *k_cache, *v_cache;
    const int32_t *block_tables, *context_lens;
    const float *bias;
    const float *bias_table;    /* [H, num_buckets] relative-position table, or NULL */
    int num_buckets;
    const int32_t *pairs;       /* optional list of (s, h) pairs */
    int window;
    double scale;
    int block_size, num_seqs, num_heads, head_dim, max_blocks_per_seq, bias_row_stride, dtype;
};

static void decode_item(long long item, void *p)
{
    const struct decode_ctx *c = (const struct decode_ctx *)p;
    const int H = c->num_heads, D = c->head_dim, bs = c->block_size;
    int s, h;
    if (c->pairs) { s = c->pairs[2 * item]; h = c->pairs[2 * item + 1]; }
    else          { s = (int)(item / H); h = (int)(item % H); }
    double *o = c->out + (size_t)item * D;
    const int ctx = c->context_lens[s];
    int start = 0;
    if (c->window > 0 && ctx > c->window) start = ctx - c->window;
    const int n = ctx > start ? ctx - start : 0;
    double *x = (double *)malloc(sizeof(double) * (n > 0 ? n : 1));
    size_t *vrow = (size_t *)malloc(sizeof(size_t) * (n > 0 ? n : 1));
    const size_t qoff = ((size_t)s * H + h) * D;
    for (int t = 0; t < n; ++t) {
        const int j = start + t;
        const int32_t blk = c->block_tables[(size_t)s * c->max_blocks_per_seq + j / bs];
        const size_t row = (((size_t)blk * H + h) * bs + (j % bs)) * D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += load_elem(c->q, qoff + d, c->dtype) * load_elem(c->k_cache, row + d, c->dtype);
        double a = 0.0;
        if (c->bias) {
            a = (double)c->bias[((size_t)s * H + h) * c->bias_row_stride + j];
        } else if (c->bias_table) {
            /* key j lies (ctx - 1 - j) positions behind the query; distances past
               the table's last column reuse that column */
            int d = (ctx - 1) - j;
            if (d > c->num_buckets - 1) d = c->num_buckets - 1;
            a = (double)c->bias_table[(size_t)h * c->num_buckets + d];
        }
        x[t] = c->scale * (dot + a);
        vrow[t] = row;
    }
    softmax_combine(o, x, vrow, n, c->v_cache, c->dtype, D);
    free(x);
    free(vrow);
}

/* out: double [num_items, D] where items are all (s, h) in s-major order when
 * pairs == NULL, else the num_pairs listed (s, h) pairs in order. */
void oracle_paged_decode(double *out, const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *block_tables, const int32_t *context_lens,
                         const float *bias, int window, double scale, int block_size,
                         int num_seqs, int num_heads, int head_dim, int max_blocks_per_seq,
                         int bias_row_stride, int dtype, const int32_t *pairs, int num_pairs,
                         int nthreads)
{
    struct decode_ctx c = {out, q, k_cache, v_cache, block_tables, context_lens, bias, NULL, 0, pairs,
                           window, scale, block_size, num_seqs, num_heads, head_dim,
                           max_blocks_per_seq, bias_row_stride, dtype};
    long long n = pairs ? num_pairs : (long long)num_seqs * num_heads;
    run_items(decode_item, &c, n, nthreads);
}

/* Paged decode with the T5 relative-position bias read from its table instead
 * of a materialised A: A[s,h,j] = bias_table[h, min(ctx_s - 1 - j, num_buckets - 1)]
 * ("PagedAttention: Support custom attention bias for T5 model (1/2)": the
 * relative distance is capped, larger distances reuse the last value, and the
 * page proposes computing the T5 bias in the kernel instead of materialising
 * it).  Otherwise identical to oracle_paged_decode. */
void oracle_paged_decode_t5(double *out, const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, const int32_t *context_lens,
                            const float *bias_table, int num_buckets, int window, double scale,
                            int block_size, int num_seqs, int num_heads, int head_dim,
                            int max_blocks_per_seq, int dtype, const int32_t *pairs, int num_pairs,
                            int nthreads)
{
    struct decode_ctx c = {out, q, k_cache, v_cache, block_tables, context_lens, NULL, bias_table,
                           num_buckets, pairs, window, scale, block_size, num_seqs, num_heads,
                           head_dim, max_blocks_per_seq, 0, dtype};
    long long n = pairs ? num_pairs : (long long)num_seqs * num_heads;
    run_items(decode_item, &c, n, nthreads);
}

/* ---- packed varlen prefill ---------------------------------------------- */

struct prefill_ctx {
    double *out;
    const void *q, *k, *v;
    const int32_t *cu_seqlens;
    const int64_t *rows;        /* optional list of token rows */
    int num_seqs, num_heads, head_dim, window, causal, dtype;
    double scale;
    int chunk;                  /* > 0: keys only from the query's own chunk of this many positions */
    const float *rel_bias;      /* optional [H, 2 * num_buckets - 1] relative-position bias */
    int num_buckets;
};

/* The relative-position bias for a query d positions after its key (d < 0:
 * before it); distances beyond num_buckets - 1 either way reuse the end
 * columns. */
static double rel_term(const float *rel_bias, int num_buckets, int h, int d)
{
    const int cap = num_buckets - 1;
    if (d > cap) d = cap;
    if (d < -cap) d = -cap;
    return (double)rel_bias[(size_t)h * (2 * num_buckets - 1) + cap + d];
}

static int mask_keeps(int r, int c, int window, int causal, int chunk)
{
    if (causal && c > r) return 0;
    if (chunk > 0 && r / chunk != c / chunk) return 0;
    if (window > 0) {
        int d = r - c;
        if (d < 0) d = -d;
        if (d >= window) return 0;
    }
    return 1;
}

static void prefill_item(long long item, void *p)
{
    const struct prefill_ctx *c = (const struct prefill_ctx *)p;
    const int H = c->num_heads, D = c->head_dim;
    const long long row_i = item / H;
    const int h = (int)(item % H);
    const long long i = c->rows ? c->rows[row_i] : row_i;
    int b = 0;
    while (b + 1 <= c->num_seqs && c->cu_seqlens[b + 1] <= i) ++b;
    const long long s0 = c->cu_seqlens[b];
    const int L = c->cu_seqlens[b + 1] - c->cu_seqlens[b];
    const int r = (int)(i - s0);
    double *o = c->out + (size_t)item * D;
    double *x = (double *)malloc(sizeof(double) * (L > 0 ? L : 1));
    size_t *vrow = (size_t *)malloc(sizeof(size_t) * (L > 0 ? L : 1));
    int n = 0;
    const size_t qoff = ((size_t)i * H + h) * D;
    for (int col = 0; col < L; ++col) {
        if (!mask_keeps(r, col, c->window, c->causal, c->chunk)) continue;
        const size_t row = ((size_t)(s0 + col) * H + h) * D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += load_elem(c->q, qoff + d, c->dtype) * load_elem(c->k, row + d, c->dtype);
        const double bias = c->rel_bias ? rel_term(c->rel_bias, c->num_buckets, h, r - col) : 0.0;
        x[n] = c->scale * (dot + bias);
        vrow[n] = row;
        ++n;
    }
    softmax_combine(o, x, vrow, n, c->v, c->dtype, D);
    free(x);
    free(vrow);
}

/* out: double [num_rows, H, D] for the listed token rows (rows == NULL: all
 * cu_seqlens[num_seqs] rows in order). */
void oracle_prefill(double *out, const void *q, const void *k, const void *v,
                    const int32_t *cu_seqlens, int num_seqs, int num_heads, int head_dim,
                    int window, int causal, double scale, int dtype,
                    const int64_t *rows, long long num_rows, int nthreads)
{
    struct prefill_ctx c = {out, q, k, v, cu_seqlens, rows, num_seqs, num_heads, head_dim,
                            window, causal, dtype, scale, 0, NULL, 0};
    long long nr = rows ? num_rows : (long long)cu_seqlens[num_seqs];
    run_items(prefill_item, &c, nr * num_heads, nthreads);
}

/* Chunked local attention: a query at position r of its sequence sees only
 * the keys of its own chunk, positions [r / chunk * chunk, r / chunk * chunk
 * + chunk) (causal: and c <= r) — the block-diagonal "chunked local
 * attention" layers that "[V1] Add sliding window support to Flex Attention
 * backend" discusses beside the sliding window. */
void oracle_prefill_chunked(double *out, const void *q, const void *k, const void *v,
                            const int32_t *cu_seqlens, int num_seqs, int num_heads, int head_dim,
                            int chunk, int causal, double scale, int dtype,
                            const int64_t *rows, long long num_rows, int nthreads)
{
    struct prefill_ctx c = {out, q, k, v, cu_seqlens, rows, num_seqs, num_heads, head_dim,
                            -1, causal, dtype, scale, chunk, NULL, 0};
    long long nr = rows ? num_rows : (long long)cu_seqlens[num_seqs];
    run_items(prefill_item, &c, nr * num_heads, nthreads);
}

/* Prefill with the relative-position bias A[h, r, c] = rel_bias[h, cap +
 * clamp(r - c, -cap, cap)], cap = num_buckets - 1, added to q . k before the
 * scale (the T5 bias of an encoder's self-attention). */
void oracle_prefill_biased(double *out, const void *q, const void *k, const void *v,
                           const int32_t *cu_seqlens, int num_seqs, int num_heads, int head_dim,
                           int window, int causal, double scale, int dtype, const float *rel_bias,
                           int num_buckets, const int64_t *rows, long long num_rows, int nthreads)
{
    struct prefill_ctx c = {out, q, k, v, cu_seqlens, rows, num_seqs, num_heads, head_dim,
                            window, causal, dtype, scale, 0, rel_bias, num_buckets};
    long long nr = rows ? num_rows : (long long)cu_seqlens[num_seqs];
    run_items(prefill_item, &c, nr * num_heads, nthreads);
}

/* ---- prefill against the paged cache -------------------------------------- */

struct paged_prefill_ctx {
    double *out;
    const void *q, *k_cache, *v_cache;
    const int32_t *cu_seqlens_q, *context_lens, *block_tables;
    const float *rel_bias;
    const int64_t *rows;
    int num_seqs, num_heads, head_dim, block_size, max_blocks_per_seq, window, causal, num_buckets, dtype;
    double scale;
};

static void paged_prefill_item(long long item, void *p)
{
    const struct paged_prefill_ctx *c = (const struct paged_prefill_ctx *)p;
    const int H = c->num_heads, D = c->head_dim, bs = c->block_size;
    const long long row_i = item / H;
    const int h = (int)(item % H);
    const long long i = c->rows ? c->rows[row_i] : row_i;
    int b = 0;
    while (b + 1 <= c->num_seqs && c->cu_seqlens_q[b + 1] <= i) ++b;
    const int Lq = c->cu_seqlens_q[b + 1] - c->cu_seqlens_q[b];
    const int ctx = c->context_lens[b];
    const int pos = ctx - Lq + (int)(i - c->cu_seqlens_q[b]);   /* the query's own key position */
    double *o = c->out + (size_t)item * D;
    double *x = (double *)malloc(sizeof(double) * (ctx > 0 ? ctx : 1));
    size_t *vrow = (size_t *)malloc(sizeof(size_t) * (ctx > 0 ? ctx : 1));
    int n = 0;
    const size_t qoff = ((size_t)i * H + h) * D;
    for (int col = 0; col < ctx; ++col) {
        if (!mask_keeps(pos, col, c->window, c->causal, 0)) continue;
        const int32_t blk = c->block_tables[(size_t)b * c->max_blocks_per_seq + col / bs];
        const size_t row = (((size_t)blk * H + h) * bs + (col % bs)) * D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += load_elem(c->q, qoff + d, c->dtype) * load_elem(c->k_cache, row + d, c->dtype);
        const double bias = c->rel_bias ? rel_term(c->rel_bias, c->num_buckets, h, pos - col) : 0.0;
        x[n] = c->scale * (dot + bias);
        vrow[n] = row;
        ++n;
    }
    softmax_combine(o, x, vrow, n, c->v_cache, c->dtype, D);
    free(x);
    free(vrow);
}

/* out: double [num_rows, H, D] for the listed query rows (rows == NULL: all
 * cu_seqlens_q[num_seqs] rows in order). */
void oracle_paged_prefill(double *out, const void *q, const void *k_cache, const void *v_cache,
                          const int32_t *block_tables, const int32_t *cu_seqlens_q, const int32_t *context_lens,
                          int num_seqs, int num_heads, int head_dim, int block_size, int max_blocks_per_seq,
                          int window, int causal, double scale, const float *rel_bias, int num_buckets, int dtype,
                          const int64_t *rows, long long num_rows, int nthreads)
{
    struct paged_prefill_ctx c = {out, q, k_cache, v_cache, cu_seqlens_q, context_lens, block_tables,
                                  rel_bias, rows, num_seqs, num_heads, head_dim, block_size,
                                  max_blocks_per_seq, window, causal, num_buckets, dtype, scale};
    long long nr = rows ? num_rows : (long long)cu_seqlens_q[num_seqs];
    run_items(paged_prefill_item, &c, nr * num_heads, nthreads);
}

/* ---- reshape_and_cache --------------------------------------------------- */

void oracle_reshape_and_cache(void *k_cache, void *v_cache, const void *key, const void *value,
                              const int64_t *slot_mapping, long long num_tokens, int num_heads,
                              int head_dim, int block_size, int elt_bytes)
{
    const size_t rowb = (size_t)head_dim * elt_bytes;
    for (long long t = 0; t < num_tokens; ++t) {
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        const int64_t blk = slot / block_size, off = slot % block_size;
        for (int h = 0; h < num_heads; ++h) {
            const size_t src = ((size_t)t * num_heads + h) * rowb;
            const size_t dst = (((size_t)blk * num_heads + h) * block_size + off) * rowb;
            memcpy((char *)k_cache + dst, (const char *)key + src, rowb);
            memcpy((char *)v_cache + dst, (const char *)value + src, rowb);
        }
    }
}
