// reshape_and_cache.cu — scatter new K/V token rows into the paged caches.
//
// The KV-caching step of "Add Encoder-decoder model support and T5 Model
// support" (its split-out cross-attention KV caching item): token t, head h
// goes to cache[slot / bs, h, slot % bs, :] with slot = slot_mapping[t], both
// for K and V; a negative slot skips the token.
//
// Pure data movement, HBM-bound: 2 x (read + write) of num_tokens * H * D
// elements.  One thread moves one 16-byte chunk of K and the same chunk of V;
// a row of head_dim elements is ROW/16 consecutive threads, so both the reads
// (token-major) and the writes (one row per (block, head, offset)) are whole
// 16-byte vectors in runs of at least 128 bytes.
#include "pka_device.cuh"
#include "pka_launch.h"

namespace pka {
namespace {

__global__ void __launch_bounds__(256) reshape_and_cache_kernel(
    const uint4 *__restrict__ key, const uint4 *__restrict__ value, uint4 *__restrict__ k_cache,
    uint4 *__restrict__ v_cache, const int64_t *__restrict__ slot_mapping, long long total_chunks,
    int chunks_per_row, int num_heads, int block_size, long long num_slots, int32_t *status)
{
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total_chunks; i += stride) {
        const long long row = i / chunks_per_row;           // t * H + h
        const int c = (int)(i - row * chunks_per_row);
        const long long t = row / num_heads;
        const int h = (int)(row - t * num_heads);
        const int64_t slot = __ldg(slot_mapping + t);
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (c == 0 && h == 0) flag_status(status, PKA_DEVCHK_SLOT);
            continue;
        }
        const long long blk = slot / block_size;
        const int off = (int)(slot - blk * block_size);
        const long long dst = (((blk * num_heads + h) * block_size + off) * chunks_per_row) + c;
        const uint4 kv = __ldcs(key + i);
        const uint4 vv = __ldcs(value + i);
        __stcg(k_cache + dst, kv);
        __stcg(v_cache + dst, vv);
    }
}

}  // namespace

cudaError_t launch_reshape_and_cache(const void *key, const void *value, void *k_cache, void *v_cache,
                                     const int64_t *slot_mapping, int num_tokens, int num_heads,
                                     int head_dim, int block_size, int num_blocks, int elt_bytes,
                                     int32_t *status, cudaStream_t stream)
{
    const int chunks_per_row = head_dim * elt_bytes / 16;
    const long long total = (long long)num_tokens * num_heads * chunks_per_row;
    if (total == 0) return cudaSuccess;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int threads = 256;
    long long blocks = (total + threads - 1) / threads;
    const long long cap = (long long)sms * 8;              // 8 x 256 threads resident per SM
    if (blocks > cap) blocks = cap;
    reshape_and_cache_kernel<<<(unsigned)blocks, threads, 0, stream>>>(
        static_cast<const uint4 *>(key), static_cast<const uint4 *>(value), static_cast<uint4 *>(k_cache),
        static_cast<uint4 *>(v_cache), slot_mapping, total, chunks_per_row, num_heads, block_size,
        (long long)num_blocks * block_size, status);
    return cudaGetLastError();
}

}  // namespace pka
