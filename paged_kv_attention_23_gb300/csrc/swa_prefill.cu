// swa_prefill.cu — full / sliding-window attention prefill over a packed
// variable-length batch on the 5th-generation tensor cores (tcgen05, TMEM,
// TMA), bf16 in / bf16 out, f32 softmax and accumulation.
//
// What it computes ("[V1] Add sliding window support to Flex Attention
// backend": bidirectional attention with a sliding window for encoder-only
// models, layers alternating full / window): for query position r of a
// sequence of length L, the keys c with
//   window <= 0: all c (causal: c <= r);  window > 0: |r - c| < W (causal: 0 <= r - c < W)
//   O_r = sum_c softmax_c(scale * q_r . k_c) v_c
// Only key tiles that intersect the band are visited: a 128-row query tile at
// r0 reads keys [r0 - W + 1, r0 + 127 + W - 1] (two 128-key tiles for W = 64),
// i.e. the "visit only intra-window blocks" principle of the same page.
//
// One persistent CTA per SM, warp-specialised:
//   warp 0      TMA producer: the query tile (128 x 64) into one of two Q
//               buffers, K and V tiles (128 keys x 64) into a 3-stage ring; all
//               tiles land 128-byte swizzled, the layout the MMA reads.
//   warp 1      TMEM owner and MMA issuer (one thread): S = Q K^T as 4 MMAs
//               128x128x16 into one of two S buffers in TMEM, then
//               O_j = P V as 8 MMAs 128x64x16 into one of two O buffers.
//   warps 2..5  softmax, one thread per query row (the TMEM lane): load the S
//               row, mask, online max / sum in the log2 domain, write P (bf16)
//               to shared memory in the swizzled layout, then fold the
//               previous tile's O into an f32 register accumulator with the
//               running-max correction; at the end normalise and store.
// S(j+1) is computed while the softmax works on S(j), and P(j) V(j) runs
// while the softmax works on S(j+1).  Every wait is bounded: on a timeout the
// CTA records PKA_DEVCHK_TIMEOUT, every role stops, TMEM is freed, and the
// kernel returns.
#include <cuda.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "pka_device.cuh"
#include "pka_launch.h"
#include "pka_tc.cuh"

namespace pka {
namespace {

constexpr int BM = 128;        // query rows per tile = TMEM lanes = MMA M
constexpr int BN = 128;        // keys per K/V tile
constexpr int HD = 64;         // head dim
constexpr int NS = 3;          // K/V stages
constexpr int MAX_SEQS = 1024; // sequences per launch (the host splits larger batches)
constexpr int NTHREADS = 192;

constexpr uint32_t TILE_BYTES = BM * HD * 2;          // 16 KB: one Q, K or V tile
constexpr uint32_t P_BYTES = BM * BN * 2;             // 32 KB: P as two 64-key blocks
constexpr uint32_t OFF_Q = 0;                          // 2 x 16 KB
constexpr uint32_t OFF_KV = 2 * TILE_BYTES;            // NS x (K 16 KB, V 16 KB)
constexpr uint32_t OFF_P = OFF_KV + NS * 2 * TILE_BYTES; // 2 x 32 KB
constexpr uint32_t OFF_BAR = OFF_P + 2 * P_BYTES;
constexpr int NBAR = 2 + 2 + NS + NS + 2 + 2 + 2 + 2 + 2;
constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;      // tmem base, abort flag
constexpr uint32_t OFF_SCHED = (OFF_MISC + 16 + 127) / 128 * 128;
constexpr uint32_t SMEM_BYTES = OFF_SCHED + (4 * MAX_SEQS + 1) * 4 + 1024;   // + alignment slack

// TMEM columns: S buffers at 0 and 128, O buffers at 256 and 320
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S = 0, COL_O = 256;

constexpr uint32_t IDESC_QK = tc::idesc_bf16_f32(BM, BN, false, false);  // S = Q K^T, both K-major
constexpr uint32_t IDESC_PV = tc::idesc_bf16_f32(BM, HD, false, true);   // O = P V, V is MN-major

struct Params {
    __nv_bfloat16 *out;
    const int32_t *cu_seqlens;
    int32_t *status;
    float scale_log2;
    int num_seqs, num_tokens, H, window, causal;
};

struct Tile {
    int s0, L, h, r0, c_lo, nkv;
};

struct Sched {
    const int *cum, *start, *len;
    int nseq, H, window, causal;
    __device__ __forceinline__ Tile get(int t) const
    {
        int lo = 0, hi = nseq;                         // cum[lo] <= t < cum[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (cum[mid] <= t) lo = mid; else hi = mid;
        }
        Tile T;
        T.s0 = start[lo];
        T.L = len[lo];
        const int nq = (T.L + BM - 1) / BM;
        const int r = t - cum[lo];
        T.h = r / nq;                                  // q tiles of one head are neighbours: shared K/V in L2
        T.r0 = (r - T.h * nq) * BM;
        const int r_last = min(T.r0 + BM, T.L) - 1;
        int c_lo = 0, c_hi = T.L - 1;
        if (window > 0) {
            c_lo = max(0, T.r0 - window + 1);
            c_hi = min(T.L - 1, r_last + window - 1);
        }
        if (causal) c_hi = min(c_hi, r_last);
        T.c_lo = c_lo;
        T.nkv = (c_hi - c_lo) / BN + 1;
        return T;
    }
};

// bounded wait that also gives up once another role has aborted
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                              int32_t *status)
{
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (clock64() - t0 > (1ll << 31)) {
            *abort_flag = 1;
            flag_status(status, PKA_DEVCHK_TIMEOUT);
            return false;
        }
    }
    return true;
}

__global__ void __launch_bounds__(NTHREADS, 1)
swa_prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const Params P)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte alignment for the swizzled tiles
    unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
    const uint32_t bar0 = sb + OFF_BAR;
    auto BAR = [&](int i) { return bar0 + 8u * i; };
    // barrier indices
    const int Q_FULL = 0, Q_EMPTY = 2, KV_FULL = 4, KV_EMPTY = 4 + NS, S_FULL = 4 + 2 * NS, S_EMPTY = S_FULL + 2,
              P_FULL = S_EMPTY + 2, O_FULL = P_FULL + 2, O_EMPTY = O_FULL + 2;
    uint32_t *tmem_base_sm = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_MISC + 4);
    int *cum = reinterpret_cast<int *>(smem + OFF_SCHED);
    int *start = cum + MAX_SEQS + 1;
    int *len = start + MAX_SEQS;
    int *rank_tmp = len + MAX_SEQS;

    // ---- schedule: sequences by decreasing length (longest work first) -------
    const int S = P.num_seqs;
    for (int s = threadIdx.x; s < S; s += NTHREADS) {
        int a = P.cu_seqlens[s], b = P.cu_seqlens[s + 1];
        if (a < 0 || b < a || b > P.num_tokens) {
            flag_status(P.status, PKA_DEVCHK_CU_SEQLENS);
            a = 0; b = 0;
        }
        rank_tmp[s] = b - a;
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < NBAR; ++i) {
            const bool by_softmax = (i >= S_EMPTY && i < S_EMPTY + 2) || (i >= P_FULL && i < P_FULL + 2) ||
                                    (i >= O_EMPTY && i < O_EMPTY + 2);
            mbar_init(BAR(i), by_softmax ? 128 : 1);
        }
        *abort_flag = 0;
    }
    fence_barrier_init();
    if (warp == 1) tc::tmem_alloc(sb + OFF_MISC, TMEM_COLS);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    for (int s = threadIdx.x; s < S; s += NTHREADS) {
        const int Ls = rank_tmp[s];
        int rk = 0;
        for (int t = 0; t < S; ++t) {
            const int Lt = rank_tmp[t];
            rk += (Lt > Ls) || (Lt == Ls && t < s);
        }
        int a = P.cu_seqlens[s];
        start[rk] = a < 0 ? 0 : a;
        len[rk] = Ls;
    }
    __syncthreads();
    if (warp == 0) {
        const int per = (S + 31) / 32;
        const int a = min(lane * per, S), b = min(a + per, S);
        int local = 0;
        for (int i = a; i < b; ++i) local += (len[i] + BM - 1) / BM * P.H;
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - local;
        for (int i = a; i < b; ++i) { cum[i] = run; run += (len[i] + BM - 1) / BM * P.H; }
        if (lane == 31) cum[S] = incl;
    }
    __syncthreads();
    const Sched sched{cum, start, len, S, P.H, P.window, P.causal};
    const int total_tiles = cum[S];
    const uint32_t tmem = *tmem_base_sm;

    if (warp == 0 && lane == 0) {
        // ======================= TMA producer =======================
        tc::prefetch_tensormap(&tm_q);
        tc::prefetch_tensormap(&tm_k);
        tc::prefetch_tensormap(&tm_v);
        uint32_t g = 0, wq = 0;
        for (int t = blockIdx.x; t < total_tiles && !*abort_flag; t += gridDim.x, ++wq) {
            const Tile T = sched.get(t);
            const uint32_t qb = wq & 1;
            if (!wait_or_abort(BAR(Q_EMPTY + qb), ((wq >> 1) & 1) ^ 1, abort_flag, P.status)) break;
            mbar_arrive_expect_tx(BAR(Q_FULL + qb), TILE_BYTES);
            tc::tma_load_3d(sb + OFF_Q + qb * TILE_BYTES, &tm_q, 0, T.h, T.s0 + T.r0, BAR(Q_FULL + qb));
            bool ok = true;
            for (int j = 0; j < T.nkv; ++j, ++g) {
                const uint32_t st = g % NS;
                if (!wait_or_abort(BAR(KV_EMPTY + st), ((g / NS) & 1) ^ 1, abort_flag, P.status)) { ok = false; break; }
                const int row = T.s0 + T.c_lo + j * BN;
                mbar_arrive_expect_tx(BAR(KV_FULL + st), 2 * TILE_BYTES);
                tc::tma_load_3d(sb + OFF_KV + st * 2 * TILE_BYTES, &tm_k, 0, T.h, row, BAR(KV_FULL + st));
                tc::tma_load_3d(sb + OFF_KV + st * 2 * TILE_BYTES + TILE_BYTES, &tm_v, 0, T.h, row,
                                BAR(KV_FULL + st));
            }
            if (!ok) break;
        }
    } else if (warp == 1 && lane == 0) {
        // ======================= MMA issuer =======================
        uint32_t g = 0, wq = 0;
        auto issue_pv = [&](uint32_t gg) -> bool {
            const uint32_t pb = gg & 1;
            if (!wait_or_abort(BAR(P_FULL + pb), (gg >> 1) & 1, abort_flag, P.status)) return false;
            if (!wait_or_abort(BAR(O_EMPTY + pb), ((gg >> 1) & 1) ^ 1, abort_flag, P.status)) return false;
            tc::fence_after_sync();
            const uint32_t pa = sb + OFF_P + pb * P_BYTES;
            const uint32_t va = sb + OFF_KV + (gg % NS) * 2 * TILE_BYTES + TILE_BYTES;
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
                tc::mma_bf16(tmem + COL_O + pb * HD, tc::sw128_desc(pa + (kk >> 2) * (P_BYTES / 2) + (kk & 3) * 32),
                             tc::sw128_desc(va + kk * 2048), IDESC_PV, kk > 0);
            tc::commit(BAR(O_FULL + pb));
            tc::commit(BAR(KV_EMPTY + gg % NS));
            return true;
        };
        for (int t = blockIdx.x; t < total_tiles && !*abort_flag; t += gridDim.x, ++wq) {
            const Tile T = sched.get(t);
            const uint32_t qb = wq & 1;
            if (!wait_or_abort(BAR(Q_FULL + qb), (wq >> 1) & 1, abort_flag, P.status)) break;
            const uint32_t qa = sb + OFF_Q + qb * TILE_BYTES;
            bool ok = true;
            for (int j = 0; j < T.nkv; ++j, ++g) {
                const uint32_t st = g % NS, sbuf = g & 1;
                if (!wait_or_abort(BAR(KV_FULL + st), (g / NS) & 1, abort_flag, P.status) ||
                    !wait_or_abort(BAR(S_EMPTY + sbuf), ((g >> 1) & 1) ^ 1, abort_flag, P.status)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                const uint32_t ka = sb + OFF_KV + st * 2 * TILE_BYTES;
#pragma unroll
                for (int kk = 0; kk < HD / 16; ++kk)
                    tc::mma_bf16(tmem + COL_S + sbuf * BN, tc::sw128_desc(qa + kk * 32), tc::sw128_desc(ka + kk * 32),
                                 IDESC_QK, kk > 0);
                tc::commit(BAR(S_FULL + sbuf));
                if (j > 0 && !issue_pv(g - 1)) { ok = false; break; }
            }
            if (!ok || !issue_pv(g - 1)) break;
            tc::commit(BAR(Q_EMPTY + qb));
        }
    } else if (warp >= 2) {
        // ======================= softmax =======================
        const int quarter = warp & 3;                  // TMEM lanes this warp may touch
        const int row = quarter * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        uint32_t g = 0;
        for (int t = blockIdx.x; t < total_tiles && !*abort_flag; t += gridDim.x) {
            const Tile T = sched.get(t);
            const int rr = T.r0 + row;                 // query position within its sequence
            int lo = 0, hi = T.L;                      // keys [lo, hi) kept for this row
            if (P.window > 0) { lo = max(lo, rr - P.window + 1); hi = min(hi, rr + P.window); }
            if (P.causal) hi = min(hi, rr + 1);
            float O[HD];
#pragma unroll
            for (int i = 0; i < HD; ++i) O[i] = 0.f;
            float m = -INFINITY, l = 0.f, corr_prev = 1.f;
            bool ok = true;
            auto fold_o = [&](uint32_t gg, float c) -> bool {
                const uint32_t ob = gg & 1;
                if (!wait_or_abort(BAR(O_FULL + ob), (gg >> 1) & 1, abort_flag, P.status)) return false;
                tc::fence_after_sync();
                float o[HD];
                tc::tmem_ld64(tmem + lane_addr + COL_O + ob * HD, o);
                tc::fence_before_sync();
                mbar_arrive(BAR(O_EMPTY + ob));
#pragma unroll
                for (int i = 0; i < HD; ++i) O[i] = fmaf(O[i], c, o[i]);
                return true;
            };
            for (int j = 0; j < T.nkv; ++j, ++g) {
                const uint32_t sbuf = g & 1;
                if (!wait_or_abort(BAR(S_FULL + sbuf), (g >> 1) & 1, abort_flag, P.status)) { ok = false; break; }
                tc::fence_after_sync();
                float x[BN];
                tc::tmem_ld64(tmem + lane_addr + COL_S + sbuf * BN, x);
                tc::tmem_ld64(tmem + lane_addr + COL_S + sbuf * BN + 64, x + 64);
                tc::fence_before_sync();
                mbar_arrive(BAR(S_EMPTY + sbuf));
                // mask to the kept key range, scale into the log2 domain, tile max
                const int c0 = T.c_lo + j * BN;
                const int ilo = lo - c0, ihi = hi - c0;
                float mt = -INFINITY;
                if (ilo <= 0 && ihi >= BN) {
#pragma unroll
                    for (int i = 0; i < BN; ++i) { x[i] *= P.scale_log2; mt = fmaxf(mt, x[i]); }
                } else {
#pragma unroll
                    for (int i = 0; i < BN; ++i) {
                        x[i] = (i >= ilo && i < ihi) ? x[i] * P.scale_log2 : -INFINITY;
                        mt = fmaxf(mt, x[i]);
                    }
                }
                const float m_new = fmaxf(m, mt);
                const float m_use = m_new == -INFINITY ? 0.f : m_new;
                const float corr = ex2(m - m_use);
                // P = 2^(x - m) as bf16 into the swizzled P buffer; row sum in f32
                const uint32_t pbase = sb + OFF_P + sbuf * P_BYTES + (row >> 3) * 1024 + (row & 7) * 128;
                float lt = 0.f;
#pragma unroll
                for (int c = 0; c < BN / 8; ++c) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float p0 = ex2(x[c * 8 + 2 * e] - m_use), p1 = ex2(x[c * 8 + 2 * e + 1] - m_use);
                        lt += p0 + p1;
                        __nv_bfloat162 hb = __floats2bfloat162_rn(p0, p1);
                        w[e] = *reinterpret_cast<uint32_t *>(&hb);
                    }
                    const uint32_t kb = c >> 3, ch = c & 7;
                    const uint32_t addr = pbase + kb * (P_BYTES / 2) + ((ch ^ (row & 7)) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]), "r"(w[1]),
                                 "r"(w[2]), "r"(w[3])
                                 : "memory");
                }
                l = fmaf(l, corr, lt);
                m = m_new;
                fence_proxy_async();                   // P is read by the tensor cores (async proxy)
                mbar_arrive(BAR(P_FULL + sbuf));
                if (j > 0 && !fold_o(g - 1, corr_prev)) { ok = false; break; }
                corr_prev = corr;
            }
            if (!ok || !fold_o(g - 1, corr_prev)) break;
            if (rr < T.L) {
                const float inv = l > 0.f ? 1.f / l : 0.f;
                uint4 *dst = reinterpret_cast<uint4 *>(P.out + ((size_t)(T.s0 + rr) * P.H + T.h) * HD);
#pragma unroll
                for (int c = 0; c < HD / 8; ++c) {
                    float v[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = O[c * 8 + e] * inv;
                    dst[c] = Vec<__nv_bfloat16>::from_f32(v);
                }
            }
        }
    }

    // ---- teardown: every role is done with TMEM --------------------------------
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---- host: tensor maps ---------------------------------------------------------
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// [T, H, 64] bf16 rows -> boxes of 128 tokens x 64 dims of one head, 128-byte swizzle
bool make_map(CUtensorMap *m, const void *base, int T, int H)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)HD, (cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)HD * 2, (cuuint64_t)H * HD * 2};
    const cuuint32_t box[3] = {HD, 1, BM};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_swa_prefill(const PrefillArgs &a, cudaStream_t stream)
{
    if (a.head_dim != HD) return cudaErrorInvalidValue;
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, a.q, a.num_tokens, a.num_heads) || !make_map(&mk, a.k, a.num_tokens, a.num_heads) ||
        !make_map(&mv, a.v, a.num_tokens, a.num_heads))
        return cudaErrorInvalidValue;
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
        attr = cudaFuncSetAttribute(swa_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    });
    if (attr != cudaSuccess) return attr;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    Params P;
    P.out = static_cast<__nv_bfloat16 *>(a.out);
    P.status = a.status;
    P.scale_log2 = a.scale * 1.4426950408889634f;
    P.num_tokens = a.num_tokens;
    P.H = a.num_heads;
    P.window = a.window;
    P.causal = a.causal;
    for (int base = 0; base < a.num_seqs; base += MAX_SEQS) {
        P.num_seqs = std::min(MAX_SEQS, a.num_seqs - base);
        P.cu_seqlens = a.cu_seqlens + base;
        const long long tiles_upper = (long long)P.num_seqs * ((a.max_seqlen + BM - 1) / BM) * a.num_heads;
        const int grid = (int)std::max<long long>(1, std::min<long long>(sms, tiles_upper));
        swa_prefill_tc_kernel<<<grid, NTHREADS, SMEM_BYTES, stream>>>(mq, mk, mv, P);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace pka
