// paged_decode_noalloc.cu — paged decode for callers that cannot allocate
// device memory.
//
// pka_paged_attn_decode needs a caller-provided scratch workspace.  Some
// callers have no way to get one: code embedded in a host framework that owns
// every byte of device memory through its own pool and forbids allocations
// outside it, or a latency-critical loop where a cudaMalloc could stall the
// whole device.  This entry point runs the same decode kernel with its scratch
// taken from one fixed, file-scope device array instead, so the caller passes
// only inputs and outputs and nothing is allocated at call time.
//
// Costs and rules of the fixed array:
//  * Every GPU that loads libpka holds PKA_NOALLOC_SCRATCH_BYTES for it until
//    the process exits.
//  * A call whose scratch need (pka_paged_attn_decode_workspace_size) exceeds
//    that size is rejected with PKA_ERR_WORKSPACE before anything is enqueued.
//  * All calls on a device share the one array, and it keeps whatever the last
//    call left in it.  Each call clears the part that must start at zero -- the
//    first 256 bytes (the unit hand-out counter) and the split-K arrival
//    counters after them -- on its own stream before the kernel runs.  Two
//    calls whose work overlaps on the GPU (different streams, not ordered by
//    events) race on the array and give wrong results.
//  * The array's device address is looked up once per device, on the first
//    call made while that device is current (and again if the device's
//    context was created anew, e.g. after cudaDeviceReset, since the module
//    then lives at a new address); make that first call before any stream
//    capture begins.
#include <cuda_runtime.h>

#include <mutex>

#include "pka_launch.h"

namespace {

static __device__ __align__(256) unsigned char pka_noalloc_scratch[PKA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 128;
std::mutex g_scratch_mu;
struct ScratchAddr {
    void *ctx;    // the context the address belongs to
    void *addr;   // device address of the array in that context
};
ScratchAddr g_scratch_addr[kMaxDevices];   // per device ordinal

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, never a device address, so
// the address comes from the runtime, once per device (and once more for a
// context that replaced the one the cached address belongs to).
pka_status scratch_address(void **addr)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return PKA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PKA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchAddr &c = g_scratch_addr[dev];
    void *ctx = pka::current_context();
    if (c.addr == nullptr || ctx == nullptr || c.ctx != ctx) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, pka_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) return PKA_ERR_CUDA;
        c.addr = p;
        c.ctx = pka::current_context();   // the lookup made the context current if none was
    }
    *addr = c.addr;
    return PKA_OK;
}

}  // namespace

extern "C" PKA_API pka_status pka_paged_attn_decode_noalloc(
    void *out, const void *q, const void *k_cache, const void *v_cache, const int32_t *block_tables,
    const int32_t *context_lens, const float *attn_bias, int sliding_window, float scale, int block_size,
    int num_seqs, int num_heads, int head_dim, int max_blocks_per_seq, int bias_row_stride, int num_blocks,
    int max_context_len, pka_dtype dtype, int32_t *status, void *stream)
{
    // Check every argument first, with no workspace: a valid call with work to
    // do answers PKA_ERR_WORKSPACE; anything else (an argument error, or OK
    // for zero sequences) is the answer as is, with nothing enqueued.
    const pka_status probe = pka_paged_attn_decode(
        out, q, k_cache, v_cache, block_tables, context_lens, attn_bias, sliding_window, scale, block_size,
        num_seqs, num_heads, head_dim, max_blocks_per_seq, bias_row_stride, num_blocks, max_context_len, dtype,
        nullptr, 0, status, stream);
    if (probe != PKA_ERR_WORKSPACE) return probe;

    const size_t need = pka_paged_attn_decode_workspace_size(num_seqs, num_heads, head_dim, max_context_len,
                                                             sliding_window);
    if (need > (size_t)PKA_NOALLOC_SCRATCH_BYTES) return PKA_ERR_WORKSPACE;

    void *scratch = nullptr;
    const pka_status st = scratch_address(&scratch);
    if (st != PKA_OK) return st;

    // the unit hand-out counter (the first 256 bytes of the workspace) and the
    // arrival counters after it (int32 per (sequence, head)) must start at zero
    const size_t counter_bytes = 256 + (size_t)num_seqs * num_heads * sizeof(int32_t);
    if (cudaMemsetAsync(scratch, 0, counter_bytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PKA_ERR_CUDA;
    return pka_paged_attn_decode(out, q, k_cache, v_cache, block_tables, context_lens, attn_bias, sliding_window,
                                 scale, block_size, num_seqs, num_heads, head_dim, max_blocks_per_seq,
                                 bias_row_stride, num_blocks, max_context_len, dtype, scratch,
                                 (size_t)PKA_NOALLOC_SCRATCH_BYTES, status, stream);
}
