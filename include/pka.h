/*
 * pka.h — C ABI of libpka.so: paged-KV attention kernels for GB300 (sm_103a).
 *
 * The operation is softmax((Q K^T + A) / sqrt(d_k)) V as written in
 * "PagedAttention: Support custom attention bias for T5 model (1/2)" (opening
 * section), with 1/sqrt(d_k) passed in as `scale`, which multiplies the bias
 * as well.  K and V live in a paged cache and are reached through per-sequence
 * block tables; decoder self-attention and encoder cross-attention each use
 * their own table and are two calls ("Add Encoder-decoder model support and
 * T5 Model support", the comments that settle on two block tables).  The
 * optional sliding window follows "[V1] Add sliding window support to Flex
 * Attention backend": causal for decode, bidirectional for encoder prefill.
 *
 * Conventions shared by every entry point
 *  - Every pointer argument is a DEVICE pointer owned by the caller; the
 *    library never allocates, frees or keeps a pointer after the call.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default
 *    stream) and runs asynchronously.  Outputs are valid once that work has
 *    completed.
 *  - The decode kernels are launched with programmatic stream serialization:
 *    they may start while the previous kernel in the stream finishes, and
 *    read nothing before it has completed.  They also let the NEXT kernel in
 *    the stream start early if that kernel was itself launched with
 *    programmatic stream serialization; such a kernel must wait for its
 *    dependencies (cudaGridDependencySynchronize / griddepcontrol.wait)
 *    before reading a decode's outputs, as the CUDA programming model
 *    requires of any kernel launched that way.  Kernels launched without
 *    that attribute see plain stream order.
 *  - Arguments are checked on the host before anything is launched; a bad
 *    argument returns PKA_ERR_INVALID_ARG (or PKA_ERR_UNSUPPORTED for a legal
 *    but unimplemented shape / dtype) and launches nothing.  A failed launch
 *    returns PKA_ERR_CUDA.
 *  - Data-dependent checks (a block id outside [0, num_blocks), a context
 *    length outside [0, max_context_len]) happen on the device: the kernel
 *    never reads or writes outside the buffers described by the size
 *    arguments, ORs a PKA_DEVCHK_* bit into *status (when status != NULL) and
 *    produces unspecified values for the affected rows.  The caller reads
 *    *status after synchronising; the library never synchronises.
 *  - Alignment: q, out, key, value, k, v, k_cache and v_cache must be 16-byte
 *    aligned; attn_bias 4-byte aligned; integer arrays naturally aligned.
 *  - Cache layout: [num_blocks, num_heads, block_size, head_dim], row-major;
 *    one (block, head) is one contiguous block_size * head_dim run.
 *  - Supported now: head_dim in {64, 128}; block_size 16; num_kv_heads ==
 *    num_heads.  Decode: f32, f16, bf16 (q, caches and out share one dtype;
 *    the bias is always f32).  Prefill: bf16 or f16; head_dim 64, or 128 for
 *    pka_swa_prefill and pka_chunked_prefill (the biased and paged prefills
 *    answer PKA_ERR_UNSUPPORTED at 128).
 */
#ifndef PKA_H
#define PKA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKA_API __attribute__((visibility("default")))
#else
#define PKA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PKA_OK = 0,
    PKA_ERR_INVALID_ARG = 1,
    PKA_ERR_UNSUPPORTED = 2,
    PKA_ERR_CUDA = 3,
    PKA_ERR_WORKSPACE = 4   /* workspace NULL, misaligned or smaller than required */
} pka_status;

typedef enum { PKA_F32 = 0, PKA_F16 = 1, PKA_BF16 = 2 } pka_dtype;

/* Bits the kernels OR into the optional device status word. */
#define PKA_DEVCHK_BLOCK_ID     0x1  /* a block-table entry outside [0, num_blocks) */
#define PKA_DEVCHK_CONTEXT_LEN  0x2  /* a context length < 0, > max_context_len or
                                        > max_blocks_per_seq * block_size */
#define PKA_DEVCHK_SLOT         0x4  /* a slot >= num_blocks * block_size */
#define PKA_DEVCHK_TIMEOUT      0x8  /* a pipeline wait gave up (a copy never landed) */
#define PKA_DEVCHK_CU_SEQLENS   0x10 /* cu_seqlens not non-decreasing within [0, num_tokens] */

/* Human-readable name of a status code (static string, never NULL). */
PKA_API const char *pka_status_string(pka_status s);

/* Library version, major * 10000 + minor * 100 + patch. */
PKA_API int pka_version(void);

/*
 * pka_reshape_and_cache — scatter new K/V token rows into the paged caches:
 *   k_cache[slot / block_size, h, slot % block_size, :] = key[t, h, :]
 *   v_cache[...same...]                                  = value[t, h, :]
 * with slot = slot_mapping[t]; slot < 0 skips token t (padding).  This is the
 * KV-caching step that "Add Encoder-decoder model support and T5 Model
 * support" lists for cross-attention (its split-out "Cross-attention KV
 * caching and memory-management" item), for the blocks that the block tables
 * of either attention type point at.
 *
 *   key, value    [num_tokens, num_heads, head_dim] of dtype, contiguous
 *   k_cache, v_cache [num_blocks, num_heads, block_size, head_dim] of dtype
 *   slot_mapping  int64 [num_tokens]
 *   status        int32 device word or NULL (PKA_DEVCHK_SLOT on a slot past
 *                 the cache; that token is skipped)
 * Exact: the cache receives the bytes of key/value unchanged.  Two tokens that
 * map to the same slot leave one of them (unspecified which).
 * num_tokens == 0 is a no-op.
 */
PKA_API pka_status pka_reshape_and_cache(const void *key, const void *value, void *k_cache, void *v_cache,
                                 const int64_t *slot_mapping, int num_tokens, int num_heads,
                                 int head_dim, int block_size, int num_blocks, pka_dtype dtype,
                                 int32_t *status, void *stream);

/*
 * pka_paged_attn_decode — one query token per sequence against its paged
 * K/V ("PagedAttention: Support custom attention bias for T5 model (1/2)":
 * the paged kernel with the optional bias pointer).  For sequence s, head h:
 *   ctx   = context_lens[s]  (keys 0 .. ctx-1; the query is token ctx-1)
 *   start = sliding_window > 0 ? max(0, ctx - sliding_window) : 0
 *   x_j   = scale * (q[s,h,:] . K_j + A[s,h,j])      for j in [start, ctx)
 *   out[s,h,:] = sum_j softmax(x)_j V_j                (ctx == 0: zeros)
 * with K_j = k_cache[block_tables[s, j / bs], h, j % bs, :] and V_j likewise.
 * A is read only inside [start, ctx): padding (any value, NaN included) and
 * block-table entries outside the window are never read — blocks before the
 * window may be evicted ("[V1] Add sliding window support to Flex Attention
 * backend": the direct build skips blocks outside the window when the page
 * table evicts them).  Cache rows outside [start, ctx) inside the blocks
 * that are read -- the rows past ctx in the sequence's last block (not yet
 * written), the rows before start in the window's first block -- may hold any
 * bits, NaN and Inf included: they contribute exactly nothing.
 *
 *   out           [num_seqs, num_heads, head_dim] of dtype
 *   q             [num_seqs, num_heads, head_dim] of dtype
 *   k_cache, v_cache [num_blocks, num_heads, block_size, head_dim] of dtype
 *   block_tables  int32 [num_seqs, max_blocks_per_seq]
 *   context_lens  int32 [num_seqs], each in [0, max_context_len]
 *   attn_bias     f32 [num_seqs, num_heads, bias_row_stride] or NULL (no bias,
 *                 no extra work; the review answer that a null bias pointer is
 *                 a no-op); bias_row_stride >= max_context_len (the bias is
 *                 padded to the maximum sequence length).
 *   sliding_window -1 (none) or >= 1
 *   scale         multiplies q.k AND the bias (1/sqrt(head_dim) gives the
 *                 formula as printed)
 *   workspace     device scratch of at least
 *                 pka_paged_attn_decode_workspace_size(...) bytes, 256-byte
 *                 aligned, ZERO-FILLED before its first use.  Every call that
 *                 completes leaves the whole workspace zero again, so it is
 *                 reused without clearing by later calls of any shape (after a
 *                 PKA_DEVCHK_TIMEOUT, zero it again).  Calls that share a
 *                 workspace must not overlap in time (same stream, or ordered
 *                 by events).
 *   status        int32 device word or NULL (PKA_DEVCHK_* bits)
 * Accumulation is f32 whatever the I/O dtype; f16 outputs stay finite for
 * finite inputs (the f16 overflow report in "Add Encoder-decoder model support
 * and T5 Model support").
 */
PKA_API size_t pka_paged_attn_decode_workspace_size(int num_seqs, int num_heads, int head_dim,
                                            int max_context_len, int sliding_window);

PKA_API pka_status pka_paged_attn_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
                                 const int32_t *block_tables, const int32_t *context_lens,
                                 const float *attn_bias, int sliding_window, float scale,
                                 int block_size, int num_seqs, int num_heads, int head_dim,
                                 int max_blocks_per_seq, int bias_row_stride, int num_blocks,
                                 int max_context_len, pka_dtype dtype, void *workspace,
                                 size_t workspace_bytes, int32_t *status, void *stream);

/*
 * pka_paged_attn_decode_t5bias — pka_paged_attn_decode with the T5 relative-
 * position bias computed in the kernel from its table instead of a
 * materialised A ("PagedAttention: Support custom attention bias for T5 model
 * (1/2)": the page proposes computing the T5 relative-position bias in the
 * kernel, and its first review comment caps the relative distance — T5-large
 * uses 128 — with larger distances reusing the last value):
 *   A[s,h,j] = bias_table[h, min(ctx_s - 1 - j, num_buckets - 1)]
 * (key j lies ctx_s - 1 - j positions behind the query).  No bias rows are
 * read and nothing is padded to max_seq_len.
 *   bias_table  f32 [num_heads, num_buckets], 4-byte aligned;
 *               num_heads * num_buckets <= PKA_MAX_BIAS_TABLE
 *               (PKA_ERR_UNSUPPORTED beyond; it is cached in shared memory)
 * Every other argument, the workspace and the errors are as for
 * pka_paged_attn_decode (no attn_bias / bias_row_stride).
 */
#define PKA_MAX_BIAS_TABLE 3072

PKA_API pka_status pka_paged_attn_decode_t5bias(void *out, const void *q, const void *k_cache, const void *v_cache,
                                                const int32_t *block_tables, const int32_t *context_lens,
                                                const float *bias_table, int num_buckets, int sliding_window,
                                                float scale, int block_size, int num_seqs, int num_heads,
                                                int head_dim, int max_blocks_per_seq, int num_blocks,
                                                int max_context_len, pka_dtype dtype, void *workspace,
                                                size_t workspace_bytes, int32_t *status, void *stream);

/*
 * pka_paged_attn_decode_multi — several decode problems in one launch.  An
 * encoder-decoder decode step attends twice per layer: decoder self-attention
 * over the generated tokens' cache blocks and cross-attention over the
 * prompt's ("Add Encoder-decoder model support and T5 Model support": the two
 * attention types keep separate block tables, and cross-attention's context
 * is the encoder length, fixed for the request).  Both go into one grid here:
 * each problem keeps its own q/out, caches, block table, context lengths,
 * bias, window, scale and workspace, and every problem computes exactly what
 * pka_paged_attn_decode (or, with bias_table, pka_paged_attn_decode_t5bias)
 * computes for it alone.  The problems only share one launch (a single
 * launch latency and one tail instead of two).
 *
 *   problems      host array of num_problems descriptors (read during the
 *                 call only); each field means what the argument of the same
 *                 name means for pka_paged_attn_decode.  bias_table /
 *                 num_buckets select the in-kernel T5 bias as for
 *                 pka_paged_attn_decode_t5bias; a problem has attn_bias or
 *                 bias_table, not both.  When two problems both use a table
 *                 it must be the same table (same pointer and num_buckets:
 *                 it is cached once in shared memory).
 *   num_problems  1 or 2 (PKA_ERR_UNSUPPORTED beyond)
 *   block_size, num_heads, head_dim, dtype   shared by all problems
 *   workspace     each problem's own workspace field: sized by
 *                 pka_paged_attn_decode_workspace_size for that problem,
 *                 zero-filled before first use and left zero, as for
 *                 pka_paged_attn_decode; the problems' workspaces must not
 *                 overlap.  PKA_ERR_WORKSPACE if any is missing or short.
 *   status        one int32 device word or NULL for all problems
 *   key_new, value_new  optional, 16-byte aligned: the K and V rows of each
 *                 sequence's newest token, position ctx_s - 1, fused append.
 *                 The launch first writes them to the cache at
 *                   k_cache[block_tables[s, (ctx_s-1) / 16], h, (ctx_s-1) % 16, :]
 *                 (v_cache likewise) — what pka_reshape_and_cache does with
 *                 that slot — and attends with them, so one launch does the
 *                 scatter and the decode of a step ("Add Encoder-decoder model
 *                 support and T5 Model support": KV caching of the new token
 *                 precedes its attention).  Results and cache contents are
 *                 bit-identical to pka_reshape_and_cache followed by the
 *                 decode.  The caches of such a problem are written (the
 *                 const qualifier notwithstanding); the block holding
 *                 position ctx_s - 1 must belong to sequence s alone, and no
 *                 other problem of the launch may read it.  ctx_s == 0
 *                 appends nothing.  A block id out of range sets
 *                 PKA_DEVCHK_BLOCK_ID and skips the write.
 * Problems with num_seqs == 0 are skipped.  The problems' out arrays must
 * not overlap (PKA_ERR_INVALID_ARG).  Errors are those of the single-problem calls, checked per
 * problem before anything is enqueued.
 */
typedef struct {
    void *out;
    const void *q;
    const void *k_cache;
    const void *v_cache;
    const int32_t *block_tables;
    const int32_t *context_lens;
    const float *attn_bias;      /* or NULL */
    const float *bias_table;     /* or NULL: T5 table [num_heads, num_buckets] */
    int num_buckets;
    int sliding_window;
    float scale;
    int num_seqs;
    int max_blocks_per_seq;
    int bias_row_stride;
    int num_blocks;
    int max_context_len;
    void *workspace;
    size_t workspace_bytes;
    const void *key_new;         /* or NULL: [num_seqs, num_heads, head_dim] of dtype */
    const void *value_new;       /* NULL exactly when key_new is */
} pka_decode_problem;

PKA_API pka_status pka_paged_attn_decode_multi(const pka_decode_problem *problems, int num_problems,
                                               int block_size, int num_heads, int head_dim, pka_dtype dtype,
                                               int32_t *status, void *stream);

/*
 * pka_paged_attn_decode_noalloc — pka_paged_attn_decode for callers that
 * cannot allocate device memory.  The pages have no counterpart: this is an
 * interface convenience, not part of the method.
 *
 * Some callers have no way to hand over a scratch workspace: code embedded in
 * a host framework that owns all device memory through its own pool and
 * forbids allocations outside it, or a latency-critical loop where a
 * cudaMalloc could stall the device.  This entry point takes the same
 * arguments as pka_paged_attn_decode minus the workspace, computes the same
 * result with the same kernel, and allocates nothing: its scratch is one
 * fixed device array of PKA_NOALLOC_SCRATCH_BYTES inside libpka, which every
 * GPU that loads the library holds until the process exits.
 *  - Returns PKA_ERR_WORKSPACE, with nothing enqueued, when the call needs more
 *    scratch than that (compare pka_paged_attn_decode_workspace_size with
 *    PKA_NOALLOC_SCRATCH_BYTES).  Other argument errors are as for
 *    pka_paged_attn_decode.
 *  - All calls on a device share the array and it keeps the last call's
 *    contents; each call clears, on its own stream, the part that must start at
 *    zero.  Calls whose work overlaps on the GPU (different streams not ordered
 *    by events) race on the array and produce wrong results.
 *  - The array's device address is looked up on the first call made with a
 *    device current; make that first call before any stream capture begins.
 */
#define PKA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

PKA_API pka_status pka_paged_attn_decode_noalloc(void *out, const void *q, const void *k_cache,
                                                 const void *v_cache, const int32_t *block_tables,
                                                 const int32_t *context_lens, const float *attn_bias,
                                                 int sliding_window, float scale, int block_size, int num_seqs,
                                                 int num_heads, int head_dim, int max_blocks_per_seq,
                                                 int bias_row_stride, int num_blocks, int max_context_len,
                                                 pka_dtype dtype, int32_t *status, void *stream);

/*
 * pka_swa_prefill — attention for every token of a packed variable-length
 * batch ("[V1] Add sliding window support to Flex Attention backend":
 * bidirectional attention with a sliding window for encoder-only models; the
 * alternating full / window layers).  For a token at position r of sequence
 * b (rows cu_seqlens[b] .. cu_seqlens[b+1]-1), the keys are the positions c of
 * the same sequence with
 *   window <= 0 (-1), causal = 0 : every c
 *   window <= 0 (-1), causal = 1 : c <= r
 *   window  > 0,      causal = 0 : |r - c| < window
 *   window  > 0,      causal = 1 : 0 <= r - c < window
 *   out[i,h,:] = sum_c softmax(scale * q[i,h,:] . k[c,h,:])_c v[c,h,:]
 * Only key tiles that intersect the mask are visited.
 *
 *   out, q, k, v  [num_tokens, num_heads, head_dim] of dtype (PKA_BF16 or
 *                 PKA_F16; head_dim 64 or 128), contiguous
 *   cu_seqlens    int32 [num_seqs + 1], non-decreasing, cu_seqlens[0] = 0,
 *                 cu_seqlens[num_seqs] = num_tokens
 *   max_seqlen    upper bound on every sequence length (a longer sequence
 *                 sets PKA_DEVCHK_CU_SEQLENS; its rows past max_seqlen are
 *                 not written)
 *   window        -1 (full) or >= 1
 *   causal        0 or 1
 *   status        int32 device word or NULL (PKA_DEVCHK_CU_SEQLENS,
 *                 PKA_DEVCHK_TIMEOUT)
 * Accumulation is f32; P is rounded to the operand type (bf16 or f16) before
 * the P.V product, whose operands must share one type.
 * Work items are handed to the CTAs through a pair of device counters that
 * the library owns (no workspace argument); a launch leaves its pair at zero
 * when it ends (also after a PKA_DEVCHK_TIMEOUT).
 *  - An eager launch takes the next of 1024 pairs in turn, shared by this and
 *    the other prefill entry points: at most 1024 eager launches may be in
 *    flight on the GPU at once.
 *  - A launch made while `stream` is being captured into a CUDA graph takes a
 *    pair that no other launch is ever given (8192 such pairs per device per
 *    process), which the graph keeps for every replay; replays of one
 *    instantiated graph are ordered, so they never share it at once.  Do not
 *    run two instances of one captured graph at the same time.  Captures past
 *    the 8192th deal items statically (no counter; correct, somewhat slower).
 */
PKA_API pka_status pka_swa_prefill(void *out, const void *q, const void *k, const void *v,
                           const int32_t *cu_seqlens, int num_seqs, int num_tokens, int max_seqlen,
                           int num_heads, int head_dim, int window, int causal, float scale,
                           pka_dtype dtype, int32_t *status, void *stream);

/*
 * pka_chunked_prefill — chunked local attention over a packed variable-length
 * batch: the block-diagonal "chunked local attention" layers that "[V1] Add
 * sliding window support to Flex Attention backend" discusses beside the
 * sliding window (Llama4: full and chunked-local layers).  A token at
 * position r of its sequence attends to the keys of its own chunk,
 *   c in [r / chunk * chunk, min(L, r / chunk * chunk + chunk))   (causal: and c <= r),
 * with the same softmax, layout, tensor-core kernel, key-tile skipping and
 * errors as pka_swa_prefill (no window).  chunk >= 1.
 */
PKA_API pka_status pka_chunked_prefill(void *out, const void *q, const void *k, const void *v,
                                       const int32_t *cu_seqlens, int num_seqs, int num_tokens, int max_seqlen,
                                       int num_heads, int head_dim, int chunk, int causal, float scale,
                                       pka_dtype dtype, int32_t *status, void *stream);

/*
 * pka_prefill_biased — pka_swa_prefill with an additive relative-position
 * bias in the scores: the T5 bias of an encoder's bidirectional
 * self-attention ("Add Encoder-decoder model support and T5 Model support":
 * T5 carries a custom bias in its attention; "PagedAttention: Support custom
 * attention bias for T5 model (1/2)": softmax((QK^T + A)/sqrt(d_k)) V, the
 * relative distance capped, larger distances reusing the last value).  With
 * cap = num_buckets - 1 and d = r - c (query position minus key position):
 *   A[h, r, c] = rel_bias[h, cap + clamp(d, -cap, cap)]
 *   out[i,h,:] = sum_c softmax(scale * (q[i,h,:] . k[c,h,:] + A[h,r,c]))_c v[c,h,:]
 * over the keys pka_swa_prefill's mask keeps.  A causal layer only reads the
 * table's non-negative half, columns cap .. 2 cap, which is the decode-side
 * table of pka_paged_attn_decode_t5bias.
 *   rel_bias   f32 [num_heads, 2 * num_buckets - 1], 4-byte aligned, not NULL
 *   num_buckets >= 1
 * Every other argument and error as for pka_swa_prefill.
 */
PKA_API pka_status pka_prefill_biased(void *out, const void *q, const void *k, const void *v,
                                      const int32_t *cu_seqlens, int num_seqs, int num_tokens, int max_seqlen,
                                      int num_heads, int head_dim, int window, int causal, const float *rel_bias,
                                      int num_buckets, float scale, pka_dtype dtype, int32_t *status, void *stream);

/*
 * pka_paged_prefill — prefill of each sequence's newest tokens against its
 * keys in the paged cache ("Add Encoder-decoder model support and T5 Model
 * support": prompt and generated tokens keep separate KV blocks, and the
 * prefill kernels as well as the decode kernels read cross-attention keys
 * through their own block table).  Sequence s has Lq_s = cu_seqlens_q[s+1] -
 * cu_seqlens_q[s] query rows and ctx_s = context_lens[s] keys, key j at
 *   k_cache[block_tables[s, j / 16], h, j % 16, :]   (v_cache likewise).
 * Query row r of s sits at key position p = ctx_s - Lq_s + r (the queries are
 * the last Lq_s positions, whose K/V reshape_and_cache has already written).
 * The keys c in [0, ctx_s) kept are pka_swa_prefill's with r replaced by p
 * (causal: c <= p; window: |p - c| < window, causal 0 <= p - c < window); the
 * optional bias is pka_prefill_biased's with d = p - c.  A row that keeps no
 * key (ctx_s == 0, or rows at p < 0 when Lq_s > ctx_s) is written as zeros.
 * With causal = 0, window -1 and no bias every query attends to all ctx_s
 * keys: a decoder prompt's cross-attention to the encoder.
 *
 *   out, q        [num_tokens, num_heads, 64] of dtype (PKA_BF16 or PKA_F16),
 *                 rows packed by cu_seqlens_q
 *   k_cache, v_cache [num_blocks, num_heads, 16, 64] of dtype, 16-byte aligned
 *   block_tables  int32 [num_seqs, max_blocks_per_seq]; entries of blocks
 *                 with no kept key (before every row's window, past ctx_s)
 *                 are never read
 *   context_lens  int32 [num_seqs], each in [0, max_blocks_per_seq * 16]
 *                 (PKA_DEVCHK_CONTEXT_LEN and clamped otherwise)
 *   max_query_len upper bound on every Lq_s
 *   rel_bias      NULL or f32 [num_heads, 2 * num_buckets - 1]
 *   block_size    16
 *   status        int32 device word or NULL (PKA_DEVCHK_CU_SEQLENS,
 *                 PKA_DEVCHK_CONTEXT_LEN, PKA_DEVCHK_BLOCK_ID — the entry is
 *                 replaced by block 0 — and PKA_DEVCHK_TIMEOUT)
 * Cache rows past ctx_s in the last block may hold any bits (NaN included).
 * Accumulation is f32; P is rounded to the operand type before the P.V product.
 */
PKA_API pka_status pka_paged_prefill(void *out, const void *q, const void *k_cache, const void *v_cache,
                                     const int32_t *block_tables, const int32_t *cu_seqlens_q,
                                     const int32_t *context_lens, int num_seqs, int num_tokens, int max_query_len,
                                     int num_heads, int head_dim, int block_size, int max_blocks_per_seq,
                                     int num_blocks, int window, int causal, const float *rel_bias, int num_buckets,
                                     float scale, pka_dtype dtype, int32_t *status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PKA_H */
