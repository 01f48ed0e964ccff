// swa_prefill.cu — sliding-window / full attention prefill over a packed
// variable-length batch ("[V1] Add sliding window support to Flex Attention
// backend": bidirectional attention with a sliding window for encoder-only
// models, and its causal counterpart).
//
// For query position r of a sequence of length L, keys c with
//   window <= 0: all c (causal: c <= r);  window > 0: |r - c| < W (causal: 0 <= r - c < W).
// Only key tiles that intersect that band are visited.
//
// This translation unit holds the CUDA-core kernel: one thread per query row,
// 64-key tiles staged in shared memory, online softmax in f32.
#include <algorithm>
#include <cmath>

#include "pka_device.cuh"
#include "pka_launch.h"

namespace pka {
namespace {

constexpr int QT = 128;   // query rows per CTA (one per thread)
constexpr int KT = 64;    // keys per shared-memory tile

template <int D>
__global__ void __launch_bounds__(QT) swa_prefill_simt_kernel(
    __nv_bfloat16 *__restrict__ out, const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
    const __nv_bfloat16 *__restrict__ v, const int32_t *__restrict__ cu_seqlens, int num_tokens, int H,
    int window, int causal, float scale_log2, int32_t *status)
{
    __shared__ __align__(16) float ks[KT][D];
    __shared__ __align__(16) float vs[KT][D];
    const int seq = blockIdx.z, h = blockIdx.y;
    const int s0 = cu_seqlens[seq], s1 = cu_seqlens[seq + 1];
    if (s0 < 0 || s1 < s0 || s1 > num_tokens) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) flag_status(status, PKA_DEVCHK_CU_SEQLENS);
        return;
    }
    const int L = s1 - s0;
    if (L > (int)gridDim.x * QT && blockIdx.x == 0 && threadIdx.x == 0) flag_status(status, PKA_DEVCHK_CU_SEQLENS);
    const int r0 = blockIdx.x * QT;
    if (r0 >= L) return;
    const int r = r0 + threadIdx.x;
    const bool row_ok = r < L;
    const int r_last = min(r0 + QT, L) - 1;
    // key range touched by this tile of rows
    int c_lo = 0, c_hi = L - 1;
    if (window > 0) { c_lo = max(0, r0 - window + 1); c_hi = min(L - 1, r_last + window - 1); }
    if (causal) c_hi = min(c_hi, r_last);

    float qf[D], acc[D];
    if (row_ok) {
        const uint4 *qp = reinterpret_cast<const uint4 *>(q + ((size_t)(s0 + r) * H + h) * D);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) Vec<__nv_bfloat16>::to_f32(qp[c], qf + c * 8);
    } else {
#pragma unroll
        for (int d = 0; d < D; ++d) qf[d] = 0.f;
    }
#pragma unroll
    for (int d = 0; d < D; ++d) acc[d] = 0.f;
    float m = -INFINITY, l = 0.f;

    for (int t0 = c_lo; t0 <= c_hi; t0 += KT) {
        __syncthreads();
        for (int i = threadIdx.x; i < KT * (D / 8); i += QT) {
            const int kr = i / (D / 8), kc = i % (D / 8);
            const int c = t0 + kr;
            if (c <= c_hi) {
                const size_t off = ((size_t)(s0 + c) * H + h) * D;
                Vec<__nv_bfloat16>::to_f32(reinterpret_cast<const uint4 *>(k + off)[kc], &ks[kr][kc * 8]);
                Vec<__nv_bfloat16>::to_f32(reinterpret_cast<const uint4 *>(v + off)[kc], &vs[kr][kc * 8]);
            }
        }
        __syncthreads();
        if (!row_ok) continue;
        const int n = min(KT, c_hi - t0 + 1);
        for (int j = 0; j < n; ++j) {
            const int c = t0 + j;
            bool keep = true;
            if (causal && c > r) keep = false;
            if (window > 0 && (r - c >= window || c - r >= window)) keep = false;
            if (!keep) continue;
            float d0 = 0.f, d1 = 0.f;
#pragma unroll
            for (int d = 0; d < D; d += 2) {
                d0 = fmaf(qf[d], ks[j][d], d0);
                d1 = fmaf(qf[d + 1], ks[j][d + 1], d1);
            }
            const float x = (d0 + d1) * scale_log2;
            const float mn = fmaxf(m, x);
            const float corr = ex2(m - mn), p = ex2(x - mn);
            l = l * corr + p;
#pragma unroll
            for (int d = 0; d < D; ++d) acc[d] = fmaf(p, vs[j][d], acc[d] * corr);
            m = mn;
        }
    }
    if (!row_ok) return;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    uint4 *op = reinterpret_cast<uint4 *>(out + ((size_t)(s0 + r) * H + h) * D);
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
        float o[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) o[e] = acc[c * 8 + e] * inv;
        op[c] = Vec<__nv_bfloat16>::from_f32(o);
    }
}

}  // namespace

cudaError_t launch_swa_prefill(const PrefillArgs &a, cudaStream_t stream)
{
    if (a.head_dim != 64) return cudaErrorInvalidValue;
    dim3 grid((a.max_seqlen + QT - 1) / QT, a.num_heads, a.num_seqs);
    if (grid.x == 0) return cudaSuccess;
    swa_prefill_simt_kernel<64><<<grid, QT, 0, stream>>>(
        static_cast<__nv_bfloat16 *>(a.out), static_cast<const __nv_bfloat16 *>(a.q),
        static_cast<const __nv_bfloat16 *>(a.k), static_cast<const __nv_bfloat16 *>(a.v), a.cu_seqlens,
        a.num_tokens, a.num_heads, a.window, a.causal, a.scale * 1.4426950408889634f, a.status);
    return cudaGetLastError();
}

}  // namespace pka
