// pka_launch.h — host-side launchers behind the C ABI (internal to libpka).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pka.h"

namespace pka {

// The driver's handle of the CUDA context current on this thread (NULL when
// none is).  Host code that caches a device address of a static __device__
// array keys the cache on it: a context created anew (after cudaDeviceReset)
// loads the module again, at a new address.
void *current_context();

// ---- reshape_and_cache ------------------------------------------------------
cudaError_t launch_reshape_and_cache(const void *key, const void *value, void *k_cache, void *v_cache,
                                     const int64_t *slot_mapping, int num_tokens, int num_heads,
                                     int head_dim, int block_size, int num_blocks, int elt_bytes,
                                     int32_t *status, cudaStream_t stream);

// ---- paged decode -----------------------------------------------------------
// How a decode call is split: each (sequence, head) range of visible key
// blocks is cut into partitions of `part_blocks` cache blocks; at most
// `max_parts` partitions per (sequence, head).
struct DecodePlan {
    int part_blocks;
    int max_parts;
};

DecodePlan decode_plan(int max_context_len, int sliding_window, int block_size);

// Workspace layout: [counters: int32 S*H | pad 256][m,l: float2 S*H*P | pad][acc: f32 S*H*P*D]
size_t decode_workspace_bytes(int num_seqs, int num_heads, int head_dim, const DecodePlan &plan);

struct DecodeArgs {
    void *out;
    const void *q, *k_cache, *v_cache;
    const int32_t *block_tables, *context_lens;
    const float *bias;
    const float *bias_table;   // T5 relative-position table [H, num_buckets] or NULL
    int num_buckets;
    const void *k_new, *v_new; // [S, H, D] newest token's K/V to append at position ctx-1, or NULL
    int32_t *status;
    float scale;
    int window, num_seqs, num_heads, head_dim, max_blocks_per_seq, num_blocks, max_context_len;
    long long bias_row_stride;
    pka_dtype dtype;
    void *workspace;
};

cudaError_t launch_paged_decode(const DecodeArgs &a, const DecodePlan &plan, cudaStream_t stream);

// Up to two problems (same heads, head_dim and dtype, num_seqs >= 1 each) in
// one grid; a.status of the first problem is the status word of the launch.
cudaError_t launch_paged_decode_multi(const DecodeArgs *a, const DecodePlan *plans, int n, cudaStream_t stream);

// ---- sliding-window prefill ----------------------------------------------------
struct PrefillArgs {
    void *out;
    const void *q;
    const void *k, *v;                 // packed [T, H, 64], or the paged caches [num_blocks, H, 16, 64]
    const int32_t *cu_seqlens;         // query rows (packed: key rows too)
    const int32_t *context_lens;       // paged only: keys per sequence
    const int32_t *block_tables;       // paged only: [num_seqs, mbps]; NULL selects packed keys
    const float *rel_bias;             // [H, 2 * num_buckets - 1] or NULL
    int num_buckets;
    int32_t *status;
    float scale;
    int num_seqs, num_tokens, max_seqlen, num_heads, head_dim, window, causal;
    int chunk;   // > 0: chunked local attention (window must be -1; packed only)
    int mbps, num_blocks;              // paged only
    pka_dtype dtype;                   // PKA_BF16 or PKA_F16
};

cudaError_t launch_swa_prefill(const PrefillArgs &a, cudaStream_t stream);

}  // namespace pka
