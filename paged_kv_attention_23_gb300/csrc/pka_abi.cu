// pka_abi.cu — the extern "C" entry points of libpka.so: argument checks on
// the host, then one launch on the caller's stream.  Nothing here allocates.
#include <cuda.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "pka_launch.h"

namespace pka {

void *current_context()
{
    using GetCurrentFn = CUresult (*)(CUcontext *);
    static GetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<GetCurrentFn>(p);
    });
    CUcontext c = nullptr;
    if (fn == nullptr || fn(&c) != CUDA_SUCCESS) return nullptr;
    return c;
}

}  // namespace pka

namespace {

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool dtype_ok(pka_dtype d) { return d == PKA_F32 || d == PKA_F16 || d == PKA_BF16; }

int elt_bytes(pka_dtype d) { return d == PKA_F32 ? 4 : 2; }

pka_status from_cuda(cudaError_t e) { return e == cudaSuccess ? PKA_OK : PKA_ERR_CUDA; }

// Every check of one decode problem, in the order the single-problem entry
// points apply them; on PKA_OK fills the launch arguments (a.num_seqs == 0:
// nothing to launch).
pka_status prepare_decode(const pka_decode_problem &p, int block_size, int num_heads, int head_dim,
                          pka_dtype dtype, int32_t *status, pka::DecodeArgs &a, pka::DecodePlan &plan)
{
    if (p.bias_table) {
        if (p.attn_bias || p.num_buckets < 1 || num_heads < 1) return PKA_ERR_INVALID_ARG;
        if ((long long)num_heads * p.num_buckets > PKA_MAX_BIAS_TABLE) return PKA_ERR_UNSUPPORTED;
        if (!aligned(p.bias_table, 4)) return PKA_ERR_INVALID_ARG;
    }
    if (p.num_seqs < 0 || num_heads < 1 || p.max_blocks_per_seq < 1 || p.num_blocks < 1 || p.max_context_len < 0 ||
        !dtype_ok(dtype) || !std::isfinite(p.scale))
        return PKA_ERR_INVALID_ARG;
    if (p.sliding_window != -1 && p.sliding_window < 1) return PKA_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return PKA_ERR_UNSUPPORTED;
    if (block_size != 16) return PKA_ERR_UNSUPPORTED;
    if ((long long)p.max_context_len > (long long)p.max_blocks_per_seq * block_size) return PKA_ERR_INVALID_ARG;
    if (p.attn_bias && (p.bias_row_stride < p.max_context_len || p.bias_row_stride < 1)) return PKA_ERR_INVALID_ARG;
    if ((p.key_new == nullptr) != (p.value_new == nullptr) || !aligned(p.key_new, 16) || !aligned(p.value_new, 16))
        return PKA_ERR_INVALID_ARG;
    a.num_seqs = 0;
    if (p.num_seqs == 0) return PKA_OK;
    if (!p.out || !p.q || !p.k_cache || !p.v_cache || !p.block_tables || !p.context_lens) return PKA_ERR_INVALID_ARG;
    if (!aligned(p.out, 16) || !aligned(p.q, 16) || !aligned(p.k_cache, 16) || !aligned(p.v_cache, 16) ||
        !aligned(p.block_tables, 4) || !aligned(p.context_lens, 4) || !aligned(p.attn_bias, 4) ||
        !aligned(status, 4))
        return PKA_ERR_INVALID_ARG;
    plan = pka::decode_plan(p.max_context_len, p.sliding_window, block_size);
    const size_t need = pka::decode_workspace_bytes(p.num_seqs, num_heads, head_dim, plan);
    if (!p.workspace || !aligned(p.workspace, 256) || p.workspace_bytes < need) return PKA_ERR_WORKSPACE;
    a.out = p.out;
    a.q = p.q;
    a.k_cache = p.k_cache;
    a.v_cache = p.v_cache;
    a.block_tables = p.block_tables;
    a.context_lens = p.context_lens;
    a.bias = p.attn_bias;
    a.bias_table = p.bias_table;
    a.num_buckets = p.bias_table ? p.num_buckets : 0;
    a.k_new = p.key_new;
    a.v_new = p.value_new;
    a.status = status;
    a.scale = p.scale;
    a.window = p.sliding_window;
    a.num_seqs = p.num_seqs;
    a.num_heads = num_heads;
    a.head_dim = head_dim;
    a.max_blocks_per_seq = p.max_blocks_per_seq;
    a.num_blocks = p.num_blocks;
    a.max_context_len = p.max_context_len;
    a.bias_row_stride = p.attn_bias ? p.bias_row_stride : 0;
    a.dtype = dtype;
    a.workspace = p.workspace;
    return PKA_OK;
}

// Checks shared by every prefill entry point; on PKA_OK fills the packed-key
// launch arguments (a.num_tokens == 0: nothing to launch).
pka_status prepare_prefill(void *out, const void *q, const void *k, const void *v, const int32_t *cu_seqlens,
                           int num_seqs, int num_tokens, int max_seqlen, int num_heads, int head_dim, int window,
                           int causal, float scale, pka_dtype dtype, int32_t *status, pka::PrefillArgs &a,
                           bool head_dim_128 = false)
{
    if (num_seqs < 0 || num_tokens < 0 || max_seqlen < 0 || num_heads < 1 || !std::isfinite(scale) ||
        (causal != 0 && causal != 1) || !dtype_ok(dtype))
        return PKA_ERR_INVALID_ARG;
    if (window != -1 && window < 1) return PKA_ERR_INVALID_ARG;
    if (dtype != PKA_BF16 && dtype != PKA_F16) return PKA_ERR_UNSUPPORTED;
    if (head_dim != 64 && !(head_dim == 128 && head_dim_128)) return PKA_ERR_UNSUPPORTED;
    a.num_tokens = 0;
    a.dtype = dtype;
    if (num_seqs == 0 || num_tokens == 0) return PKA_OK;
    if (!out || !q || !k || !v || !cu_seqlens) return PKA_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(cu_seqlens, 4) ||
        !aligned(status, 4))
        return PKA_ERR_INVALID_ARG;
    a.out = out;
    a.q = q;
    a.k = k;
    a.v = v;
    a.cu_seqlens = cu_seqlens;
    a.context_lens = nullptr;
    a.block_tables = nullptr;
    a.rel_bias = nullptr;
    a.num_buckets = 0;
    a.status = status;
    a.scale = scale;
    a.num_seqs = num_seqs;
    a.num_tokens = num_tokens;
    a.max_seqlen = max_seqlen;
    a.num_heads = num_heads;
    a.head_dim = head_dim;
    a.window = window;
    a.causal = causal;
    a.chunk = 0;
    a.mbps = 0;
    a.num_blocks = 0;
    return PKA_OK;
}

}  // namespace

extern "C" {

const char *pka_status_string(pka_status s)
{
    switch (s) {
    case PKA_OK: return "PKA_OK";
    case PKA_ERR_INVALID_ARG: return "PKA_ERR_INVALID_ARG";
    case PKA_ERR_UNSUPPORTED: return "PKA_ERR_UNSUPPORTED";
    case PKA_ERR_CUDA: return "PKA_ERR_CUDA";
    case PKA_ERR_WORKSPACE: return "PKA_ERR_WORKSPACE";
    }
    return "PKA_ERR_UNKNOWN";
}

int pka_version(void) { return 100; }

pka_status pka_reshape_and_cache(const void *key, const void *value, void *k_cache, void *v_cache,
                                 const int64_t *slot_mapping, int num_tokens, int num_heads,
                                 int head_dim, int block_size, int num_blocks, pka_dtype dtype,
                                 int32_t *status, void *stream)
{
    if (num_tokens < 0 || num_heads < 1 || num_blocks < 1 || !dtype_ok(dtype)) return PKA_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return PKA_ERR_UNSUPPORTED;
    if (block_size != 16) return PKA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PKA_OK;
    if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PKA_ERR_INVALID_ARG;
    if (!aligned(key, 16) || !aligned(value, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(slot_mapping, 8) || !aligned(status, 4))
        return PKA_ERR_INVALID_ARG;
    return from_cuda(pka::launch_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, num_tokens,
                                                   num_heads, head_dim, block_size, num_blocks,
                                                   elt_bytes(dtype), status,
                                                   static_cast<cudaStream_t>(stream)));
}

size_t pka_paged_attn_decode_workspace_size(int num_seqs, int num_heads, int head_dim, int max_context_len,
                                            int sliding_window)
{
    if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || max_context_len < 0) return 0;
    const pka::DecodePlan plan = pka::decode_plan(max_context_len, sliding_window, 16);
    return pka::decode_workspace_bytes(num_seqs, num_heads, head_dim, plan);
}

pka_status pka_paged_attn_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
                                 const int32_t *block_tables, const int32_t *context_lens,
                                 const float *attn_bias, int sliding_window, float scale,
                                 int block_size, int num_seqs, int num_heads, int head_dim,
                                 int max_blocks_per_seq, int bias_row_stride, int num_blocks,
                                 int max_context_len, pka_dtype dtype, void *workspace,
                                 size_t workspace_bytes, int32_t *status, void *stream)
{
    const pka_decode_problem p = {out, q, k_cache, v_cache, block_tables, context_lens, attn_bias, nullptr, 0,
                                  sliding_window, scale, num_seqs, max_blocks_per_seq, bias_row_stride,
                                  num_blocks, max_context_len, workspace, workspace_bytes};
    pka::DecodeArgs a;
    pka::DecodePlan plan;
    const pka_status st = prepare_decode(p, block_size, num_heads, head_dim, dtype, status, a, plan);
    if (st != PKA_OK || a.num_seqs == 0) return st;
    return from_cuda(pka::launch_paged_decode(a, plan, static_cast<cudaStream_t>(stream)));
}

pka_status pka_paged_attn_decode_t5bias(void *out, const void *q, const void *k_cache, const void *v_cache,
                                        const int32_t *block_tables, const int32_t *context_lens,
                                        const float *bias_table, int num_buckets, int sliding_window, float scale,
                                        int block_size, int num_seqs, int num_heads, int head_dim,
                                        int max_blocks_per_seq, int num_blocks, int max_context_len, pka_dtype dtype,
                                        void *workspace, size_t workspace_bytes, int32_t *status, void *stream)
{
    if (!bias_table) return PKA_ERR_INVALID_ARG;
    const pka_decode_problem p = {out, q, k_cache, v_cache, block_tables, context_lens, nullptr, bias_table,
                                  num_buckets, sliding_window, scale, num_seqs, max_blocks_per_seq, 0,
                                  num_blocks, max_context_len, workspace, workspace_bytes};
    pka::DecodeArgs a;
    pka::DecodePlan plan;
    const pka_status st = prepare_decode(p, block_size, num_heads, head_dim, dtype, status, a, plan);
    if (st != PKA_OK || a.num_seqs == 0) return st;
    return from_cuda(pka::launch_paged_decode(a, plan, static_cast<cudaStream_t>(stream)));
}

pka_status pka_paged_attn_decode_multi(const pka_decode_problem *problems, int num_problems, int block_size,
                                       int num_heads, int head_dim, pka_dtype dtype, int32_t *status, void *stream)
{
    if (!problems || num_problems < 1) return PKA_ERR_INVALID_ARG;
    if (num_problems > 2) return PKA_ERR_UNSUPPORTED;
    pka::DecodeArgs a[2];
    pka::DecodePlan plan[2];
    size_t need[2] = {0, 0};
    int n = 0;
    for (int i = 0; i < num_problems; ++i) {
        const pka_status st = prepare_decode(problems[i], block_size, num_heads, head_dim, dtype, status, a[n],
                                             plan[n]);
        if (st != PKA_OK) return st;
        if (a[n].num_seqs == 0) continue;
        need[n] = pka::decode_workspace_bytes(a[n].num_seqs, num_heads, head_dim, plan[n]);
        ++n;
    }
    if (n == 2) {
        auto overlap = [](const void *p, size_t pn, const void *q, size_t qn) {
            const uintptr_t x = reinterpret_cast<uintptr_t>(p), y = reinterpret_cast<uintptr_t>(q);
            return x < y + qn && y < x + pn;
        };
        const size_t out_bytes = (size_t)num_heads * head_dim * elt_bytes(dtype);
        if (overlap(a[0].out, out_bytes * a[0].num_seqs, a[1].out, out_bytes * a[1].num_seqs))
            return PKA_ERR_INVALID_ARG;
        if (overlap(a[0].workspace, need[0], a[1].workspace, need[1])) return PKA_ERR_WORKSPACE;
        if (a[0].bias_table && a[1].bias_table &&
            (a[0].bias_table != a[1].bias_table || a[0].num_buckets != a[1].num_buckets))
            return PKA_ERR_UNSUPPORTED;
    }
    if (n == 0) return PKA_OK;
    return from_cuda(pka::launch_paged_decode_multi(a, plan, n, static_cast<cudaStream_t>(stream)));
}

pka_status pka_swa_prefill(void *out, const void *q, const void *k, const void *v, const int32_t *cu_seqlens,
                           int num_seqs, int num_tokens, int max_seqlen, int num_heads, int head_dim, int window,
                           int causal, float scale, pka_dtype dtype, int32_t *status, void *stream)
{
    pka::PrefillArgs a;
    const pka_status st = prepare_prefill(out, q, k, v, cu_seqlens, num_seqs, num_tokens, max_seqlen, num_heads,
                                          head_dim, window, causal, scale, dtype, status, a, true);
    if (st != PKA_OK || a.num_tokens == 0) return st;
    return from_cuda(pka::launch_swa_prefill(a, static_cast<cudaStream_t>(stream)));
}

pka_status pka_chunked_prefill(void *out, const void *q, const void *k, const void *v, const int32_t *cu_seqlens,
                               int num_seqs, int num_tokens, int max_seqlen, int num_heads, int head_dim, int chunk,
                               int causal, float scale, pka_dtype dtype, int32_t *status, void *stream)
{
    if (chunk < 1) return PKA_ERR_INVALID_ARG;
    pka::PrefillArgs a;
    const pka_status st = prepare_prefill(out, q, k, v, cu_seqlens, num_seqs, num_tokens, max_seqlen, num_heads,
                                          head_dim, -1, causal, scale, dtype, status, a, true);
    if (st != PKA_OK || a.num_tokens == 0) return st;
    a.chunk = chunk;
    return from_cuda(pka::launch_swa_prefill(a, static_cast<cudaStream_t>(stream)));
}

pka_status pka_prefill_biased(void *out, const void *q, const void *k, const void *v, const int32_t *cu_seqlens,
                              int num_seqs, int num_tokens, int max_seqlen, int num_heads, int head_dim, int window,
                              int causal, const float *rel_bias, int num_buckets, float scale, pka_dtype dtype,
                              int32_t *status, void *stream)
{
    if (!rel_bias || num_buckets < 1 || !aligned(rel_bias, 4)) return PKA_ERR_INVALID_ARG;
    pka::PrefillArgs a;
    const pka_status st = prepare_prefill(out, q, k, v, cu_seqlens, num_seqs, num_tokens, max_seqlen, num_heads,
                                          head_dim, window, causal, scale, dtype, status, a);
    if (st != PKA_OK || a.num_tokens == 0) return st;
    a.rel_bias = rel_bias;
    a.num_buckets = num_buckets;
    return from_cuda(pka::launch_swa_prefill(a, static_cast<cudaStream_t>(stream)));
}

pka_status pka_paged_prefill(void *out, const void *q, const void *k_cache, const void *v_cache,
                             const int32_t *block_tables, const int32_t *cu_seqlens_q, const int32_t *context_lens,
                             int num_seqs, int num_tokens, int max_query_len, int num_heads, int head_dim,
                             int block_size, int max_blocks_per_seq, int num_blocks, int window, int causal,
                             const float *rel_bias, int num_buckets, float scale, pka_dtype dtype, int32_t *status,
                             void *stream)
{
    if (rel_bias && (num_buckets < 1 || !aligned(rel_bias, 4))) return PKA_ERR_INVALID_ARG;
    if (max_blocks_per_seq < 1 || num_blocks < 1) return PKA_ERR_INVALID_ARG;
    pka::PrefillArgs a;
    const pka_status st = prepare_prefill(out, q, k_cache, v_cache, cu_seqlens_q, num_seqs, num_tokens, max_query_len,
                                          num_heads, head_dim, window, causal, scale, dtype, status, a);
    if (st != PKA_OK) return st;
    if (block_size != 16) return PKA_ERR_UNSUPPORTED;
    if (a.num_tokens == 0) return PKA_OK;
    if (!block_tables || !context_lens || !aligned(block_tables, 4) || !aligned(context_lens, 4))
        return PKA_ERR_INVALID_ARG;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.mbps = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.rel_bias = rel_bias;
    a.num_buckets = rel_bias ? num_buckets : 0;
    return from_cuda(pka::launch_swa_prefill(a, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
