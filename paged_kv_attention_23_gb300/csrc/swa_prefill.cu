// swa_prefill.cu — full / sliding-window attention prefill over a packed
// variable-length batch on the 5th-generation tensor cores (tcgen05, TMEM,
// TMA), bf16 in / bf16 out, f32 softmax and accumulation.
//
// What it computes ("[V1] Add sliding window support to Flex Attention
// backend": bidirectional attention with a sliding window for encoder-only
// models, layers alternating full / window): for query position r of a
// sequence of length L, the keys c with
//   window <= 0: all c (causal: c <= r);  window > 0: |r - c| < W (causal: 0 <= r - c < W)
//   chunk > 0 (chunked local attention, same page): c in r's chunk of C positions (causal: c <= r)
//   O_r = sum_c softmax_c(scale * q_r . k_c) v_c
// Only key tiles that intersect the band are visited ("visit only
// intra-window blocks", same page).
//
// Two template switches widen it ("Add Encoder-decoder model support and T5
// Model support": T5's custom attention bias; prefill kernels that read
// cross-attention keys through their block table):
//   BIAS   adds rel[h, cap + clamp(d, -cap, cap)] to q.k before the scale,
//          d = query position - key position (the T5 relative-position bias);
//          every head's table, widened by a key tile's span with its clamped
//          end values, is copied to shared memory when it fits, so a score's
//          bias is one shared load at a constant offset.
//   PAGED  reads K/V from the paged cache [num_blocks, H, 16, 64] through the
//          block table, for each sequence's last Lq queries: query row r sits
//          at key position ctx - Lq + r, and the masks and the bias use it.
//
// Work item = two consecutive 128-row query tiles of one (sequence, head)
// sharing one stream of 128-key K/V tiles (for W = 64: three key tiles per
// 256 rows, each query tile multiplying only the two it needs).  One
// persistent CTA per SM, warp-specialised (warp numbers of the plain
// instances; the bias and paged instances put both MMA threads in warpgroup 0
// and the softmax in warps 4..11, with registers moved from warpgroup 0 to
// the softmax warpgroups):
//   warp 0      TMA producer: both query tiles, then the K/V tiles into a
//               ring of 3 stages (4 for paged keys; there the whole warp
//               issues a key tile's 16 cache-block boxes at once); everything
//               lands 128-byte swizzled.
//   warp 1      TMEM owner; with warp 10, one MMA-issuing thread per query
//               tile (each blocks only on its own tile's barriers): per key
//               tile, S = Q K^T (4 x 128x128x16) into that tile's S columns,
//               then O += P V (8 x 128x64x16, P read from TMEM, V MN-major
//               from shared memory) into its O columns.  QK of key tile j+1
//               is issued before PV of j, so scores are ready when the
//               softmax finishes tile j.
//   warps 2..5  softmax of query tile 0, warps 6..9 of query tile 1 (the two
//               groups ping-pong on the tensor core): one thread per row
//               loads its S row, frees the S columns at once, masks, takes
//               the max (two-input max chains), and writes P = 2^(scale*s - m)
//               as bf16 pairs into the tile's P columns of TMEM (tcgen05.st);
//               the scale is folded into the exponent's FMA.  Without bias the
//               exponentials run before the wait for the previous key tile's
//               P V, P held in registers until the store.  O stays in
//               TMEM: the running max is raised only when a row's max grows
//               by more than 2^8, and only then is that row of O rescaled in
//               TMEM (rows never see P > 256).  Each warp normalises its 32
//               rows of O and writes them with one TMA store.
// Sliding-window layers run an instance that sorts each 32-key chunk of a
// tile into kept by no row of the warp (no max, no exponentials: P = 0), kept
// whole, or kept in part (masked key by key).
// Head dim 128 (packed keys, no bias): a work item is one query tile (two
// tiles' S and O do not fit the 512 TMEM columns), and the two softmax
// warpgroups split its S tile by columns: warpgroup h takes keys 64 h .. 64 h
// + 63 of every key tile, with its own running max and sum, P and O
// accumulator (P V of a half: the half's 64 keys of V into its own O), and the
// two halves of a row are merged at the end of the item, each warpgroup
// writing 64 of the row's 128 output dims.  Every tile is two 64-dim boxes
// (the 128-byte swizzle spans 64 elements), QK takes 8 key-dim steps, and P V
// one N = 128 MMA per 16 keys across both boxes of V.  MMA thread 0 issues
// every QK; on full attention thread 1 issues both halves' P V, on banded
// masks each thread its own half's (issuing, not the tensor pipe, set the
// pace).  K and V stream into separate slots (two K, three V), each freed by
// its own MMAs; outputs leave by plain stores.
// Every wait is bounded: on a timeout the CTA records PKA_DEVCHK_TIMEOUT,
// every role stops, TMEM is freed, and the kernel returns.
#include <cuda.h>

#include <algorithm>
#include <cmath>
#include <atomic>
#include <mutex>
#include <type_traits>

#include "pka_device.cuh"
#include "pka_launch.h"
#include "pka_tc.cuh"

namespace pka {
namespace {

constexpr int BM = 128;        // query rows per tile = TMEM lanes = MMA M
constexpr int BN = 128;        // keys per K/V tile
constexpr int HD = 64;         // head dim of one 128-byte-swizzled box (a 64-dim tile, or half of a 128-dim one)
constexpr int MAX_SEQS = 1024; // sequences per launch (the host splits larger batches)
// Threads: the plain instances run 11 warps (producer, MMA of tile 0, 2 x 4
// softmax warps, MMA of tile 1) at the 168 registers a thread that 3 warps on a
// sub-partition leave.  The bias and paged instances run 12 warps: warpgroup 0
// (producer, MMA of tile 0, MMA of tile 1, one idle warp) gives registers to the
// two softmax warpgroups (setmaxnreg): 72 + 2 x 216 = 3 x 168, so the softmax's
// table loads, bias adds and block bookkeeping fit without spills (T5 encoder
// layer 0.440 -> 0.422 ms, paged self-attention 0.418 -> 0.404 ms; the plain
// instances gained nothing from it).
template <bool SPLIT> constexpr int nthreads() { return SPLIT ? 384 : 352; }
constexpr uint32_t REGS_COPY = 72, REGS_SOFTMAX = 216, REGS_AT_LAUNCH = 168;
static_assert(REGS_COPY + 2 * REGS_SOFTMAX <= 3 * REGS_AT_LAUNCH, "the split fits the registers of the launch");
constexpr float RESCALE_LOG2 = 8.f;
constexpr int LONG_ITEM_TILES = 8;              // key tiles per query tile that make an item long
constexpr long long TILE1_DELAY_CLOCKS = 1000;  // second query tile's start offset on long items

constexpr uint32_t TILE_BYTES = BM * HD * 2;             // 16 KB: one Q, K or V tile
// Shared memory and barriers of an instance with NS K/V stages.  The paged
// instances stream one 2 KB box per cache block and keep a fourth tile in
// flight (paged self- and cross-attention 4-5 % faster); the packed
// instances keep three (a fourth slowed the window and T5 encoder layers).
// At head dim 128 the "stages" are five 32 KB slots: two for K, three for V
// (K and V released separately: a K slot once its QK is done, a V slot once
// both halves' P V are done; three K and two V measured the same on full
// attention and 0.7 % slower on window 64).
template <bool PAGED, int D = 64> constexpr int nstages() { return D == 128 ? 5 : PAGED ? 4 : 3; }
constexpr int KSLOTS_128 = 2, VSLOTS_128 = 3;
constexpr uint32_t TAB_FLOATS = 2 * TILE_BYTES / 4;   // widened bias tables held in shared memory, at most
// Layout<NS, TAB>: TAB gives the bias table a region of its own (else it
// takes the output staging tiles' place and the outputs go out by plain stores)
// D is the head dim: 64, or 128 with every tile two 64-dim boxes (32 KB), one
// query tile, 2 K + 3 V slots and no staging tiles (outputs by plain stores;
// their space holds the column halves' (m, l) exchange instead).
template <int NS, bool TAB, int D = 64> struct Layout {
    static constexpr uint32_t TQ = BM * D * 2, TKV = BN * D * 2;    // bytes of a Q tile and of a K or V tile
    static constexpr uint32_t OFF_Q = 0;                             // 2 query tiles (1 at head dim 128)
    static constexpr uint32_t OFF_KV = (D == 128 ? 1 : 2) * TQ;      // NS x (K, V), or the K and V slots
    static constexpr uint32_t OFF_OST = OFF_KV + (D == 128 ? NS : 2 * NS) * TKV;   // 2 output staging tiles
    // (head dim 128: no staging tiles; the two column halves' (m, l) per row, 2 KB)
    static constexpr uint32_t OFF_BAR = OFF_OST + (D == 64 ? 2 * TILE_BYTES : 2 * BM * 8);
    // barriers: q_full, q_empty, kv_full[NS], kv_empty[NS], s_full[2], s_empty[2], p_full[2], o_full[2],
    // o_empty[2], item ring full[2] / empty[2]
    static constexpr int B_QF = 0, B_QE = 1, B_KVF = 2, B_KVE = 2 + NS, B_SF = 2 + 2 * NS, B_SE = B_SF + 2,
                         B_PF = B_SE + 2, B_OF = B_PF + 2, B_OE = B_OF + 2, B_IF = B_OE + 2, B_IE = B_IF + 2,
                         B_MX = B_IE + 2, NBAR = B_IE + 2 + (D == 128 ? 2 : 0);   // ml_full[2] at 128
    static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;         // tmem base, abort flag, item ring [2]
    static constexpr uint32_t OFF_RING = (OFF_MISC + 16 + 127) / 128 * 128;   // the two ring entries' items (64 B each)
    static constexpr uint32_t OFF_SCHED = OFF_RING + 128;
    static constexpr uint32_t OFF_TAB = (OFF_SCHED + (6 * MAX_SEQS + 1) * 4 + 15) / 16 * 16;
    static constexpr uint32_t SMEM_BYTES = OFF_TAB + (TAB ? TAB_FLOATS * 4 : 0) + 1024;   // + alignment slack
    static_assert(SMEM_BYTES <= 227u * 1024u, "dynamic shared memory per CTA");
};
// the packed bias instances give the table its own region, and their outputs
// leave by TMA stores instead of strided plain stores (T5 encoder layer 0.417
// -> 0.373 ms); the paged bias instance, with its fourth K/V stage, has no
// room left and keeps plain stores (most of its rows end in partial warps,
// and trading the fourth stage for the table measured 7 % slower)
template <bool PAGED, bool BIAS> constexpr bool own_table() { return BIAS && !PAGED; }
constexpr int CBS = 16;                   // paged cache block: 16 key rows of one head
constexpr uint32_t CBLK_BYTES = CBS * HD * 2;                                  // 2 KB per block and head

// TMEM columns of query tile w: S (f32) at 128 w, O (f32) at 256 + 64 w, P
// (bf16 pairs) at 384 + 64 w: the 512 columns exactly.  At head dim 128 (one
// tile, two column halves h): S at 0, P of half h at 128 + 32 h, O of half h
// at 256 + 128 h
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S = 0, COL_O = 256, COL_P = 384;
constexpr uint32_t COL_P_128 = 128;                 // head dim 128: P of the two column halves

// S = Q K^T (both K-major) and O += P V (V MN-major), for bf16 or f16 operands
template <typename T> __host__ __device__ constexpr bool is_bf16() { return std::is_same<T, __nv_bfloat16>::value; }
template <typename T> __host__ __device__ constexpr uint32_t idesc_qk() { return tc::idesc_16_f32(BM, BN, false, false, is_bf16<T>()); }
template <typename T> __host__ __device__ constexpr uint32_t idesc_pv() { return tc::idesc_16_f32(BM, HD, false, true, is_bf16<T>()); }
template <typename T> __host__ __device__ constexpr uint32_t idesc_pv128() { return tc::idesc_16_f32(BM, 2 * HD, false, true, is_bf16<T>()); }

struct Params {
    void *out;                       // [T, H, 64] of the operand type
    const int32_t *cu_seqlens;       // query rows (packed keys too)
    const int32_t *context_lens;     // paged: keys of each sequence
    const int32_t *block_tables;     // paged: [num_seqs, mbps] cache blocks
    const float *rel_bias;           // [H, 2 * num_buckets - 1] relative-position bias, or NULL
    int32_t *status;
    unsigned *items;                 // [2] item hand-out and finished-CTA counters, zero between launches
    float scale_log2;
    int num_seqs, num_tokens, H, window, causal, chunk;
    int mbps, num_blocks, num_buckets;
};

// One work item: two query tiles [r0, r0+128) and [r0+128, r0+256) of a
// (sequence, head) and the key tiles c_lo + 128 j, j < nkv, covering both.
// Query tile w multiplies key tiles jb[w] .. je[w] (empty when jb > je).
// Query row r sits at key position r + qoff (qoff = Lk - L: the queries are
// the sequence's last L positions); keys at k_end and beyond are not needed.
struct alignas(16) Item {
    int s0, L, Lk, qoff, seq, h, r0, c_lo, nkv, k_end;
    int jb[2], je[2];
    int pad[2];
};
static_assert(sizeof(Item) == 64, "an item is four 16-byte words in the ring");

// 32-bit words of shared memory by their shared-space address (a 32-bit
// register instead of a 64-bit generic pointer), read and written volatile
__device__ __forceinline__ int lds_volatile(uint32_t addr)
{
    int v;
    asm volatile("ld.volatile.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void sts_volatile(uint32_t addr, int v)
{
    asm volatile("st.volatile.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// An item's description read in place from its ring entry (the layout that
// the producer writes: s0, L, Lk, qoff | seq, h, r0, c_lo | nkv, k_end, jb[2] | je[2];
// the softmax warps never need seq).
struct RingItem {
    uint32_t a;    // shared-space address of the entry
    __device__ __forceinline__ int f(int i) const { return lds_volatile(a + 4u * i); }
    __device__ __forceinline__ int s0() const { return f(0); }
    __device__ __forceinline__ int L() const { return f(1); }
    __device__ __forceinline__ int Lk() const { return f(2); }
    __device__ __forceinline__ int qoff() const { return f(3); }
    __device__ __forceinline__ int h() const { return f(5); }
    __device__ __forceinline__ int r0() const { return f(6); }
    __device__ __forceinline__ int c_lo() const { return f(7); }
    __device__ __forceinline__ int nkv() const { return f(8); }
    __device__ __forceinline__ int k_end() const { return f(9); }
    __device__ __forceinline__ int jb(int w) const { return f(10 + w); }
    __device__ __forceinline__ int je(int w) const { return f(12 + w); }
};

struct Sched {
    const int *cum, *start, *len, *lenk, *seqid;
    int nseq, H, window, causal, chunk;
    bool paged;
    int qt;                                            // query tiles per item: 2, or 1 at head dim 128
    __device__ __forceinline__ Item get(int t) const
    {
        int lo = 0, hi = nseq;                         // cum[lo] <= t < cum[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (cum[mid] <= t) lo = mid; else hi = mid;
        }
        Item I;
        I.s0 = start[lo];
        I.L = len[lo];
        I.Lk = paged ? lenk[lo] : I.L;
        I.seq = seqid[lo];
        I.qoff = I.Lk - I.L;
        const int np = (I.L + qt * BM - 1) / (qt * BM);
        const int r = t - cum[lo];
        I.h = r / np;                                  // pairs of one head are neighbours: shared K/V in L2
        I.r0 = (r - I.h * np) * qt * BM;
        int c_lo = 0x7fffffff, c_hi = -1;
        int lo_w[2], hi_w[2];
        for (int w = 0; w < 2; ++w) {
            lo_w[w] = 0; hi_w[w] = -1;
            const int a = I.r0 + w * BM;
            if (w >= qt || a >= I.L) continue;
            const int pa = a + I.qoff, pb = min(a + BM, I.L) - 1 + I.qoff;   // key positions of the tile's rows
            int kl = 0, kh = I.Lk - 1;
            if (chunk > 0) { kl = pa / chunk * chunk; kh = min(I.Lk - 1, pb / chunk * chunk + chunk - 1); }
            else if (window > 0) { kl = max(0, pa - window + 1); kh = min(I.Lk - 1, pb + window - 1); }
            if (causal) kh = min(kh, pb);
            if (kh < kl) continue;                     // no key for any row of this tile
            lo_w[w] = kl;
            hi_w[w] = kh;
            c_lo = min(c_lo, kl);
            c_hi = max(c_hi, kh);
        }
        if (c_hi < 0) {                                // neither tile has a key
            I.c_lo = 0; I.nkv = 0; I.k_end = 0;
            I.jb[0] = I.jb[1] = 1; I.je[0] = I.je[1] = 0;
            return I;
        }
        if (paged) c_lo = c_lo / CBS * CBS;            // paged key tiles are whole cache blocks
        I.c_lo = c_lo;
        I.nkv = (c_hi - c_lo) / BN + 1;
        I.k_end = c_hi + 1;
        for (int w = 0; w < 2; ++w) {
            if (hi_w[w] < lo_w[w]) { I.jb[w] = 1; I.je[w] = 0; continue; }
            I.jb[w] = (lo_w[w] - c_lo) / BN;
            I.je[w] = (hi_w[w] - c_lo) / BN;
        }
        if (qt == 1) {                                 // the two column halves of the one tile
            I.jb[1] = I.jb[0];
            I.je[1] = I.je[0];
        }
        return I;
    }
};

// (y0, y1) = (x0, x1) * s + (c, c) and (a0, a1) += (y0, y1) as single packed
// f32x2 instructions (sm_100+): the softmax is issue-bound, so pairs halve
// the FMA and add work per score.
__device__ __forceinline__ void fma2(float x0, float x1, float s, float c, float &y0, float &y1)
{
    asm("{\n\t.reg .b64 a, m, k, d;\n\t"
        "mov.b64 a, {%2, %3};\n\tmov.b64 m, {%4, %4};\n\tmov.b64 k, {%5, %5};\n\t"
        "fma.rn.f32x2 d, a, m, k;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(y0), "=f"(y1)
        : "f"(x0), "f"(x1), "f"(s), "f"(c));
}

__device__ __forceinline__ void add2(float &a0, float &a1, float y0, float y1)
{
    asm("{\n\t.reg .b64 a, y;\n\t"
        "mov.b64 a, {%0, %1};\n\tmov.b64 y, {%2, %3};\n\t"
        "add.rn.f32x2 a, a, y;\n\tmov.b64 {%0, %1}, a;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(y0), "f"(y1));
}

// P = 2^(scale * s - m) for one tile row as bf16 pairs into the row's TMEM
// lane (64 columns, key 2c in the low half of column c), 16 columns per store
// (fewer live registers than one wide store); returns the f32 row sum.
template <typename T, bool SKIP>
__device__ __forceinline__ float write_p_tmem(const float *x, float scale_log2, float mneg, uint32_t tP, uint32_t dead)
{
    float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t pk[BN / 8];
        if (SKIP && ((dead >> q4) & 1u)) {
            // no row of the warp keeps a key of these 32 columns: P = 0
#pragma unroll
            for (int c = 0; c < BN / 8; ++c) pk[c] = 0u;
            tc::tmem_st16(tP + q4 * (BN / 8), pk);
            continue;
        }
#pragma unroll
        for (int c = 0; c < BN / 8; ++c) {
            const int i = q4 * (BN / 4) + 2 * c;
            float a0, a1;
            fma2(x[i], x[i + 1], scale_log2, mneg, a0, a1);
            const float p0 = ex2(a0), p1 = ex2(a1);
            add2(ls[(c & 1) * 2], ls[(c & 1) * 2 + 1], p0, p1);
            if constexpr (is_bf16<T>()) {
                __nv_bfloat162 hb = __floats2bfloat162_rn(p0, p1);
                pk[c] = *reinterpret_cast<uint32_t *>(&hb);
            } else {
                __half2 hh = __floats2half2_rn(p0, p1);
                pk[c] = *reinterpret_cast<uint32_t *>(&hh);
            }
        }
        tc::tmem_st16(tP + q4 * (BN / 8), pk);
    }
    return (ls[0] + ls[1]) + (ls[2] + ls[3]);
}

// The same P for one tile row into registers (pk[c] = keys 2c, 2c + 1), the
// TMEM stores left to the caller; returns the f32 row sum
template <typename T, bool SKIP, int NC = BN>
__device__ __forceinline__ float exp_pack(const float *x, float scale_log2, float mneg, uint32_t *pk, uint32_t dead)
{
    float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int q4 = 0; q4 < NC / 32; ++q4) {
        if (SKIP && ((dead >> q4) & 1u)) {
#pragma unroll
            for (int c = 0; c < BN / 8; ++c) pk[q4 * (BN / 8) + c] = 0u;
            continue;
        }
#pragma unroll
        for (int c = 0; c < BN / 8; ++c) {
            const int i = q4 * (BN / 4) + 2 * c;
            float a0, a1;
            fma2(x[i], x[i + 1], scale_log2, mneg, a0, a1);
            const float p0 = ex2(a0), p1 = ex2(a1);
            add2(ls[(c & 1) * 2], ls[(c & 1) * 2 + 1], p0, p1);
            if constexpr (is_bf16<T>()) {
                __nv_bfloat162 hb = __floats2bfloat162_rn(p0, p1);
                pk[q4 * (BN / 8) + c] = *reinterpret_cast<uint32_t *>(&hb);
            } else {
                __half2 hh = __floats2half2_rn(p0, p1);
                pk[q4 * (BN / 8) + c] = *reinterpret_cast<uint32_t *>(&hh);
            }
        }
    }
    return (ls[0] + ls[1]) + (ls[2] + ls[3]);
}

// setmaxnreg: a warpgroup raises or lowers its registers a thread (all its
// warps execute it); a raise waits until lowered registers are free
template <uint32_t N> __device__ __forceinline__ void regs_raise() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }
template <uint32_t N> __device__ __forceinline__ void regs_lower() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }

// bounded wait that also gives up once another role has aborted (the abort
// flag is the shared word at abort_addr)
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, uint32_t abort_addr, int32_t *status)
{
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (lds_volatile(abort_addr)) return false;
        if (clock64() - t0 > (1ll << 31)) {
            sts_volatile(abort_addr, 1);
            flag_status(status, PKA_DEVCHK_TIMEOUT);
            return false;
        }
    }
    return true;
}

// PAGED: keys come from the paged cache [num_blocks, H, 16, 64] through the
// block tables (tm_k / tm_v are 4-D maps with one cache block per box);
// otherwise from the packed [T, H, 64] keys of the same rows as the queries.
// BIAS: the relative-position bias is added to the scores.
template <typename T, bool PAGED, bool BIAS, bool BAND, int D>
__global__ void __launch_bounds__(nthreads<PAGED || BIAS>(), 1)
swa_prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                      const Params P)
{
    constexpr bool SPLIT = PAGED || BIAS;             // registers moved to the softmax warpgroups
    static_assert(D == 64 || (D == 128 && !PAGED && !BIAS), "head dim 128: packed keys, no bias");
    // Head dim 128: one query tile per item, its S tile split by columns
    // between the two softmax warpgroups (warpgroup h takes keys 64 h .. 64 h
    // + 63 of every key tile), each with its own running max and sum, P and O
    // accumulator; the two halves are merged per row at the end of the item.
    // TMEM: S at 0, P of half h at 128 + 32 h, O of half h at 256 + 128 h.
    constexpr bool WIDE = D == 128;
    constexpr int QT = WIDE ? 1 : 2;                  // query tiles per item
    constexpr int NCOL = WIDE ? BN / 2 : BN;          // score columns of a softmax warp's row
    // head dim 128, full attention: MMA thread 0 issues only the QKs and thread
    // 1 the P V of both halves (the issuing threads, not the tensor pipe, had
    // set the pace: 5.42 -> 4.54 ms); the banded instance, whose items are a
    // few key tiles long, keeps one half's P V per thread (0.456 -> 0.506 ms
    // the other way)
    constexpr bool PV_BY_1 = WIDE && !BAND;
    // MMA descriptors built once per tile and stepped by offset adds (window
    // 64 layer -1 %, paged -2 to -3 %, head dim 128 -2.5 to -3.6 %), except on
    // the plain 64-dim instance, where that measured 1-2 % slower
    constexpr bool DSTEP = PAGED || BIAS || BAND || WIDE;
    // no bias: a key tile's exponentials run before the wait for the previous
    // tile's P V, P held in registers until then (full-attention layer 1.737 ->
    // 1.638 ms, window-64 layer 0.161 -> 0.157 ms, paged cross-attention 0.181
    // -> 0.178 ms; chunked unchanged).  The bias instances measured slightly
    // slower with it
    constexpr bool EARLYP = !BIAS;
    // a row of S read from TMEM by one 128-column load and one wait on the bias
    // instances (T5 encoder 0.373 -> 0.369 ms); the others spill more with it
    // and measured 1-5 % slower, and keep two 64-column loads
    constexpr bool LD128 = BIAS;
    constexpr int NS = nstages<PAGED, D>();
    constexpr bool TAB = own_table<PAGED, BIAS>();
    constexpr bool TMA_OUT = (!BIAS || TAB) && !WIDE;   // outputs through the staging tiles
    using LY = Layout<NS, TAB, D>;
    constexpr uint32_t TQ = LY::TQ, TKV = LY::TKV;
    constexpr uint32_t OFF_Q = LY::OFF_Q, OFF_KV = LY::OFF_KV, OFF_OST = LY::OFF_OST, OFF_BAR = LY::OFF_BAR,
                       OFF_MISC = LY::OFF_MISC, OFF_RING = LY::OFF_RING, OFF_SCHED = LY::OFF_SCHED;
    constexpr int B_QF = LY::B_QF, B_QE = LY::B_QE, B_KVF = LY::B_KVF, B_KVE = LY::B_KVE, B_SF = LY::B_SF,
                  B_SE = LY::B_SE, B_PF = LY::B_PF, B_OF = LY::B_OF, B_OE = LY::B_OE, B_IF = LY::B_IF, B_IE = LY::B_IE,
                  B_MX = LY::B_MX, NBAR = LY::NBAR;
    constexpr int NTHREADS = nthreads<SPLIT>();
    constexpr int SOFTMAX_WARP0 = SPLIT ? 4 : 2;      // the 8 softmax warps follow
    constexpr int MMA1_WARP = SPLIT ? 2 : NTHREADS / 32 - 1;   // issues the MMAs of query tile 1
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte alignment for the swizzled tiles
    unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const uint32_t sb = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bar0 = sb + OFF_BAR;
    auto BAR = [&](int i) { return bar0 + 8u * i; };
    uint32_t *tmem_base_sm = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    const uint32_t abort_flag = sb + OFF_MISC + 4;    // shared word: a role gave up, all stop
    int *cum = reinterpret_cast<int *>(smem + OFF_SCHED);
    int *start = cum + MAX_SEQS + 1;
    int *len = start + MAX_SEQS;
    int *rank_tmp = len + MAX_SEQS;
    int *lenk = rank_tmp + MAX_SEQS;
    int *seqid = lenk + MAX_SEQS;

    // ---- schedule: sequences by decreasing length (longest work first) -------
    const int S = P.num_seqs;
    for (int s = threadIdx.x; s < S; s += NTHREADS) {
        int a = P.cu_seqlens[s], b = P.cu_seqlens[s + 1];
        if (a < 0 || b < a || b > P.num_tokens) {
            flag_status(P.status, PKA_DEVCHK_CU_SEQLENS);
            a = 0; b = 0;
        }
        rank_tmp[s] = b - a;
        if (PAGED) {
            const int c = P.context_lens[s];
            if (c < 0 || c > P.mbps * CBS) flag_status(P.status, PKA_DEVCHK_CONTEXT_LEN);
            // paged: order by the work of the sequence, query tiles x key tiles
            const unsigned qt = (unsigned)min((b - a + BM - 1) / BM, 65535);
            const unsigned kt = (unsigned)min((min(max(c, 0), P.mbps * CBS) + BN - 1) / BN, 65535);
            rank_tmp[s] = (int)min(qt * kt * 65536u + (unsigned)min(b - a, 65535), 0x7fffffffu);
        }
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < NBAR; ++i) {
            // (head dim 128: both warpgroups read both O accumulators, so o_empty
            // takes the 256 threads of both, and ml_full the 128 of one)
            const bool by_both_softmax = WIDE && i >= B_OE && i < B_OE + 2;
            const bool by_softmax = (i >= B_SE && i < B_SE + 2) || (i >= B_PF && i < B_PF + 2) ||
                                    (i >= B_OE && i < B_OE + 2) || (WIDE && i >= B_MX && i < B_MX + 2);
            // (head dim 128, thread 1 issuing both halves' P V: a K slot is released
            // by thread 0's QK alone)
            const bool by_both_mma = i == B_QE || (i >= B_KVE + (PV_BY_1 ? KSLOTS_128 : 0) && i < B_KVE + NS);
            const bool by_item_readers = i >= B_IE && i < B_IE + 2;   // 2 MMA threads + 8 softmax warps
            mbar_init(BAR(i), by_both_softmax ? 256 : by_softmax ? 128 : by_both_mma ? 2 : by_item_readers ? 10 : 1);
        }
        sts_volatile(abort_flag, 0);
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
        const int a = P.cu_seqlens[s];
        start[rk] = a < 0 ? 0 : a;
        len[rk] = PAGED ? (a < 0 || P.cu_seqlens[s + 1] < a || P.cu_seqlens[s + 1] > P.num_tokens ? 0
                                                                                                 : P.cu_seqlens[s + 1] - a)
                        : Ls;
        seqid[rk] = s;
        if (PAGED) lenk[rk] = min(max(P.context_lens[s], 0), P.mbps * CBS);
    }
    // The bias instances hold every head's relative-position table in shared
    // memory (a region of its own, or the staging tiles' space), widened to the
    // distances a key tile in the band can present (|d| < cap + BN) with the
    // clamped values, so a score's bias is one shared load at a constant
    // offset: no clamp, no global load.  Tables too large for it stay in
    // global memory (read through the clamp, as before).
    const int bias_cap = BIAS ? P.num_buckets - 1 : 0;
    const int tab_span = 2 * (bias_cap + BN) - 1;
    const bool tab_sm = BIAS && (long long)P.H * tab_span <= (long long)TAB_FLOATS;
    float *tab = reinterpret_cast<float *>(smem + (TAB ? LY::OFF_TAB : OFF_OST));
    if (tab_sm) {
        for (int i = threadIdx.x; i < P.H * tab_span; i += NTHREADS) {
            const int h = i / tab_span, d = i - h * tab_span - (bias_cap + BN - 1);
            tab[i] = __ldg(P.rel_bias + (size_t)h * (2 * bias_cap + 1) + bias_cap + min(max(d, -bias_cap), bias_cap));
        }
    }
    __syncthreads();
    if (warp == 0) {
        const int per = (S + 31) / 32;
        const int a = min(lane * per, S), b = min(a + per, S);
        int local = 0;
        for (int i = a; i < b; ++i) local += (len[i] + QT * BM - 1) / (QT * BM) * P.H;
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - local;
        for (int i = a; i < b; ++i) { cum[i] = run; run += (len[i] + QT * BM - 1) / (QT * BM) * P.H; }
        if (lane == 31) cum[S] = incl;
    }
    __syncthreads();
    const Sched sched{cum, start, len, lenk, seqid, S, P.H, P.window, P.causal, P.chunk, PAGED, QT};
    const int total_items = cum[S];
    const uint32_t tmem = *tmem_base_sm;
    // Items: CTA c takes item c, then items from a global counter one at a
    // time: CTAs that finish early take more, where a static deal left the
    // last CTA 5-20 % behind the average (full layer 1.97 -> 1.92 ms, chunked
    // layer 0.41 -> 0.37 ms).  A launch given no counter pair (P.items == NULL)
    // deals statically: c, c + G, c + 2G, ...  The producer thread hands each
    // id and its item's description to the MMA threads and softmax warps
    // through a two-entry ring in shared memory; an id >= total_items ends the
    // CTA's work.  Sequences are ordered longest first (paged: by query tiles
    // x key tiles, an estimate of their work).
    volatile int *item_ring = reinterpret_cast<volatile int *>(smem + OFF_MISC + 8);
    // the producer also writes each published item's description (the roles
    // then skip the schedule search): ring entry e's item at OFF_RING + 64 e
    auto put_item = [&](uint32_t slot, const Item &it) {
        int4 *dst = reinterpret_cast<int4 *>(smem + OFF_RING + slot * sizeof(Item));
        dst[0] = make_int4(it.s0, it.L, it.Lk, it.qoff);
        dst[1] = make_int4(it.seq, it.h, it.r0, it.c_lo);
        dst[2] = make_int4(it.nkv, it.k_end, it.jb[0], it.jb[1]);
        dst[3] = make_int4(it.je[0], it.je[1], 0, 0);
    };
    auto get_item = [&](uint32_t slot) {
        const int4 *src = reinterpret_cast<const int4 *>(smem + OFF_RING + slot * sizeof(Item));
        const int4 a = src[0], b = src[1], c = src[2], d = src[3];
        Item it;
        it.s0 = a.x; it.L = a.y; it.Lk = a.z; it.qoff = a.w;
        it.seq = b.x; it.h = b.y; it.r0 = b.z; it.c_lo = b.w;
        it.nkv = c.x; it.k_end = c.y; it.jb[0] = c.z; it.jb[1] = c.w;
        it.je[0] = d.x; it.je[1] = d.y;
        return it;
    };
    const bool dyn = P.items != nullptr && total_items > (int)gridDim.x;

    auto producer = [&]() {
        // ======================= TMA producer =======================
        // Paged keys: the whole warp runs the producer, lane 0 doing every wait,
        // arrival and item hand-out and each of lanes 0-15 issuing one cache
        // block's K or V box of a key tile (16 boxes a tile, issued at once
        // instead of one after another by one thread).  Otherwise one thread.
        constexpr bool WP = PAGED;
        const bool lead = !WP || lane == 0;
        auto wwait = [&](uint32_t bar, uint32_t parity) -> bool {
            if constexpr (WP) {
                int r = 1;
                if (lane == 0) r = wait_or_abort(bar, parity, abort_flag, P.status) ? 1 : 0;
                return __shfl_sync(kFull, r, 0) != 0;
            } else {
                return wait_or_abort(bar, parity, abort_flag, P.status);
            }
        };
        auto aborted = [&]() -> bool {
            int v = lds_volatile(abort_flag);
            if constexpr (WP) v = __shfl_sync(kFull, v, 0);
            return v != 0;
        };
        if (lead) {
            tc::prefetch_tensormap(&tm_q);
            tc::prefetch_tensormap(&tm_k);
            tc::prefetch_tensormap(&tm_v);
            tc::prefetch_tensormap(&tm_o);
        }
        uint32_t g = 0, wq = 0, ik = 0;
        auto publish = [&](int id, const Item &it) -> bool {
            const uint32_t slot = ik & 1;
            if (!wwait(BAR(B_IE + slot), ((ik >> 1) & 1) ^ 1)) return false;
            if (lead) {
                item_ring[slot] = id;
                if (id < total_items) put_item(slot, it);
                mbar_arrive(BAR(B_IF + slot));
            }
            ++ik;
            return true;
        };
        auto next_ahead = [&]() -> unsigned {
            unsigned a = 0;
            if (lead) a = atomicAdd(P.items, 1u);
            if constexpr (WP) a = __shfl_sync(kFull, a, 0);
            return a;
        };
        int t = (int)blockIdx.x < total_items ? (int)blockIdx.x : total_items;
        unsigned ahead = 0;                                // the counter's answer for the item after t
        if (dyn && t < total_items) ahead = next_ahead();
        for (;; ++wq) {
            Item I;
            if (t < total_items) I = sched.get(t);
            if (!publish(t, I) || t >= total_items || aborted()) break;
            t = dyn ? (int)gridDim.x + (int)ahead : t + (int)gridDim.x;
            if (dyn && t < total_items) ahead = next_ahead();
            if (!wwait(BAR(B_QE), (wq & 1) ^ 1)) break;
            const bool two = !WIDE && I.r0 + BM < I.L;
            if (lead) {
                mbar_arrive_expect_tx(BAR(B_QF), (two ? 2 : 1) * TQ);
#pragma unroll
                for (int x = 0; x < D; x += HD) {      // a 128-dim tile is two 64-dim boxes, 16 KB apart
                    tc::tma_load_3d(sb + OFF_Q + x * 256, &tm_q, x, I.h, I.s0 + I.r0, BAR(B_QF));
                    if (two) tc::tma_load_3d(sb + OFF_Q + TQ + x * 256, &tm_q, x, I.h, I.s0 + I.r0 + BM, BAR(B_QF));
                }
            }
            bool ok = true;
            // paged: the block-table entry of this lane's block of key tile j + 1 is
            // read while tile j waits for its stage, so the table's latency leaves
            // the copy path
            auto tile_blocks = [&](int j) { return min(BN / CBS, (I.k_end - (I.c_lo + j * BN) + CBS - 1) / CBS); };
            const int lb = lane & (BN / CBS - 1);        // the lane's block within a key tile
            auto read_table = [&](int j) -> int {
                const int32_t *bt = P.block_tables + (size_t)I.seq * P.mbps + (I.c_lo + j * BN) / CBS;
                return lb < tile_blocks(j) ? __ldg(bt + lb) : 0;
            };
            int id_next = 0;
            if constexpr (PAGED) id_next = read_table(0);
            // head dim 128: V of key tile number gv (global count) into its V slot
            auto load_v = [&](uint32_t gv, int row) -> bool {
                const uint32_t vs = KSLOTS_128 + gv % VSLOTS_128;
                if (!wwait(BAR(B_KVE + vs), ((gv / VSLOTS_128) & 1) ^ 1)) return false;
                mbar_arrive_expect_tx(BAR(B_KVF + vs), TKV);
#pragma unroll
                for (int x = 0; x < D; x += HD)
                    tc::tma_load_3d(sb + OFF_KV + vs * TKV + x * 256, &tm_v, x, I.h, row, BAR(B_KVF + vs));
                return true;
            };
            for (int j = 0; j < I.nkv; ++j, ++g) {
                int phys = 0;
                if constexpr (PAGED) {
                    phys = id_next;
                    if (j + 1 < I.nkv) id_next = read_table(j + 1);
                }
                if constexpr (WIDE) {
                    // K of key tile j, then V of key tile j - 1 (V one tile behind, so a
                    // K slot never waits for a V slot to drain)
                    const uint32_t kslot = g % KSLOTS_128;
                    if (!wwait(BAR(B_KVE + kslot), ((g / KSLOTS_128) & 1) ^ 1)) {
                        ok = false;
                        break;
                    }
                    const int row = I.s0 + I.c_lo + j * BN;
                    mbar_arrive_expect_tx(BAR(B_KVF + kslot), TKV);
#pragma unroll
                    for (int x = 0; x < D; x += HD)
                        tc::tma_load_3d(sb + OFF_KV + kslot * TKV + x * 256, &tm_k, x, I.h, row, BAR(B_KVF + kslot));
                    if (j > 0 && !load_v(g - 1, row - BN)) { ok = false; break; }
                    continue;
                }
                const uint32_t st = g % NS;
                if (!wwait(BAR(B_KVE + st), ((g / NS) & 1) ^ 1)) { ok = false; break; }
                const uint32_t dk = sb + OFF_KV + st * 2 * TKV, dv = dk + TKV;
                if constexpr (PAGED) {
                    // the tile's cache blocks below k_end, one 16-row box each; a
                    // 2 KB box keeps the 1024-byte swizzle atoms of a contiguous tile
                    // (lanes 0-7 the K boxes, lanes 8-15 the V boxes, of block lane % 8)
                    const int nblk = tile_blocks(j);
                    if (lead) mbar_arrive_expect_tx(BAR(B_KVF + st), 2u * nblk * CBLK_BYTES);
                    __syncwarp();                      // the byte count is set before any copy lands
                    if (lane < 2 * (BN / CBS) && lb < nblk) {
                        int pb = phys;
                        if ((unsigned)pb >= (unsigned)P.num_blocks) {
                            flag_status(P.status, PKA_DEVCHK_BLOCK_ID);
                            pb = 0;
                        }
                        if (lane < BN / CBS) tc::tma_load_4d(dk + lb * CBLK_BYTES, &tm_k, 0, 0, I.h, pb, BAR(B_KVF + st));
                        else tc::tma_load_4d(dv + lb * CBLK_BYTES, &tm_v, 0, 0, I.h, pb, BAR(B_KVF + st));
                    }
                } else {
                    const int row = I.s0 + I.c_lo + j * BN;
                    mbar_arrive_expect_tx(BAR(B_KVF + st), 2 * TKV);
#pragma unroll
                    for (int x = 0; x < D; x += HD) {
                        tc::tma_load_3d(dk + x * 256, &tm_k, x, I.h, row, BAR(B_KVF + st));
                        tc::tma_load_3d(dv + x * 256, &tm_v, x, I.h, row, BAR(B_KVF + st));
                    }
                }
            }
            if (WIDE && ok && I.nkv > 0 && !load_v(g - 1, I.s0 + I.c_lo + (I.nkv - 1) * BN)) ok = false;
            if (!ok) break;
        }
    };
    auto mma_issuer = [&]() {
        // ============ MMA issuer of query tile w (one thread per query tile) ============
        // Each issuer blocks only on its own query tile's barriers; both read
        // every K/V stage and query tile, so those are released by two arrivals.
        const int w = warp == 1 ? 0 : 1;
        uint32_t g = 0, wq = 0, cs = 0, co = 0;
        for (;; ++wq) {
            if (!wait_or_abort(BAR(B_IF + (wq & 1)), (wq >> 1) & 1, abort_flag, P.status)) break;
            const int t = item_ring[wq & 1];
            Item I;
            if (t < total_items) I = get_item(wq & 1);
            mbar_arrive(BAR(B_IE + (wq & 1)));
            if (t >= total_items || lds_volatile(abort_flag)) break;
            if (!wait_or_abort(BAR(B_QF), wq & 1, abort_flag, P.status)) break;
            const bool mine = I.jb[w] <= I.je[w];
            // (head dim 128: thread 0 issues every QK, thread 1 only its half's P V)
            if (!mine || (WIDE && w == 1)) mbar_arrive(BAR(B_QE));
            // S_w = Q_w K_j^T, when query tile w needs key tile j
            auto issue_qk = [&](int j) -> bool {
                const uint32_t gg = g + j;
                if constexpr (WIDE) {
                    // key tile j's K slot, released once this QK is done (and, when
                    // thread 1 issues half 1's P V, at once by thread 1; when it issues
                    // both halves' P V it leaves the K slots alone).  The QK waits until
                    // both halves have read S.
                    if (PV_BY_1 && w == 1) return true;
                    const uint32_t ks = gg % KSLOTS_128;
                    if (!wait_or_abort(BAR(B_KVF + ks), (gg / KSLOTS_128) & 1, abort_flag, P.status)) return false;
                    if (w == 1 || j < I.jb[w] || j > I.je[w]) {
                        mbar_arrive(BAR(B_KVE + ks));
                        return true;
                    }
                    const uint32_t c = cs + (j - I.jb[w]);
                    if (!wait_or_abort(BAR(B_SE), (c & 1) ^ 1, abort_flag, P.status) ||
                        !wait_or_abort(BAR(B_SE + 1), (c & 1) ^ 1, abort_flag, P.status))
                        return false;
                    tc::fence_after_sync();
                    // the tile's descriptors once, then stepped by the operands' byte
                    // offsets (>> 4, added to the start-address field)
                    const uint64_t dq = tc::sw128_desc(sb + OFF_Q), dk = tc::sw128_desc(sb + OFF_KV + ks * TKV);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t off = ((kk >> 2) * TILE_BYTES + (kk & 3) * 32) >> 4;
                        tc::mma_bf16(tmem + COL_S, dq + off, dk + off, idesc_qk<T>(), kk > 0);
                    }
                    tc::commit(BAR(B_SF));
                    tc::commit(BAR(B_SF + 1));
                    tc::commit(BAR(B_KVE + ks));
                    if (j == I.je[w]) tc::commit(BAR(B_QE));
                    return true;
                }
                const uint32_t st = gg % NS;
                if (!wait_or_abort(BAR(B_KVF + st), (gg / NS) & 1, abort_flag, P.status)) return false;
                if (j < I.jb[w] || j > I.je[w]) return true;
                const uint32_t c = cs + (j - I.jb[w]);
                if (!wait_or_abort(BAR(B_SE + w), (c & 1) ^ 1, abort_flag, P.status)) return false;
                tc::fence_after_sync();
                // the tile's descriptors once, then stepped by the operands' byte offsets
                // (>> 4, added to the start-address field); the plain instance builds
                // each descriptor from its address (1-2 % faster there)
                const uint32_t qa = sb + OFF_Q + w * TQ, ka = sb + OFF_KV + st * 2 * TKV;
                const uint64_t dq = tc::sw128_desc(qa), dk = tc::sw128_desc(ka);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * TILE_BYTES + (kk & 3) * 32;   // box kk / 4, 16 dims in
                    if constexpr (DSTEP)
                        tc::mma_bf16(tmem + COL_S + w * BN, dq + (off >> 4), dk + (off >> 4), idesc_qk<T>(), kk > 0);
                    else
                        tc::mma_bf16(tmem + COL_S + w * BN, tc::sw128_desc(qa + off), tc::sw128_desc(ka + off),
                                     idesc_qk<T>(), kk > 0);
                }
                tc::commit(BAR(B_SF + w));
                if (j == I.je[w]) tc::commit(BAR(B_QE));         // last read of Q_w in this item
                return true;
            };
            // O_w += P_w V_j, then release the K/V stage (or just release it)
            auto issue_pv = [&](int j) -> bool {
                if constexpr (PV_BY_1) {
                    // head dim 128, full attention: thread 1 issues the P V of both
                    // column halves, thread 0 only the QKs.  Key tile j's V slot (filled
                    // after its K: waited for here) is released by one commit after each
                    // half.  Half h: its 64 keys (16-key groups 4 h .. 4 h + 3 of V) into
                    // its O, P of the half at column 128 + 32 h.
                    if (w == 0) return true;
                    const uint32_t st = KSLOTS_128 + (g + j) % VSLOTS_128;
                    if (!wait_or_abort(BAR(B_KVF + st), ((g + j) / VSLOTS_128) & 1, abort_flag, P.status)) return false;
                    const uint32_t c = cs + (j - I.jb[w]);
                    const uint64_t dv = tc::sw128_desc_mn(sb + OFF_KV + st * TKV, TILE_BYTES);
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (!wait_or_abort(BAR(B_PF + h), c & 1, abort_flag, P.status)) return false;
                        if (j == I.jb[w] && !wait_or_abort(BAR(B_OE + h), (co & 1) ^ 1, abort_flag, P.status))
                            return false;
                        tc::fence_after_sync();
#pragma unroll
                        for (int kk = 0; kk < NCOL / 16; ++kk)
                            tc::mma_bf16_ta(tmem + COL_O + h * D, tmem + COL_P_128 + h * (NCOL / 2) + kk * 8,
                                            dv + (((h * (NCOL / 16) + kk) * 2048) >> 4), idesc_pv128<T>(),
                                            kk > 0 || j > I.jb[w]);
                        tc::commit(BAR(B_OF + h));
                        tc::commit(BAR(B_KVE + st));
                    }
                    return true;
                }
                // head dim 128 (banded): key tile j's V slot (filled after its K: wait
                // for it here), released once this P V is done
                const uint32_t st = WIDE ? KSLOTS_128 + (g + j) % VSLOTS_128 : (g + j) % NS;
                if (WIDE && !wait_or_abort(BAR(B_KVF + st), ((g + j) / VSLOTS_128) & 1, abort_flag, P.status))
                    return false;
                if (j < I.jb[w] || j > I.je[w]) {
                    mbar_arrive(BAR(B_KVE + st));
                    return true;
                }
                const uint32_t c = cs + (j - I.jb[w]);
                if (!wait_or_abort(BAR(B_PF + w), c & 1, abort_flag, P.status)) return false;
                if (j == I.jb[w] && !wait_or_abort(BAR(B_OE + w), (co & 1) ^ 1, abort_flag, P.status)) return false;
                tc::fence_after_sync();
                const uint32_t va = WIDE ? sb + OFF_KV + st * TKV : sb + OFF_KV + st * 2 * TKV + TKV;
                const uint64_t dv = WIDE ? tc::sw128_desc_mn(va, TILE_BYTES) : tc::sw128_desc(va);
                // (head dim 128: half w's 64 keys, 16-key groups 4 w .. 4 w + 3 of V,
                // into half w's O; P of the half at column 128 + 32 w)
                const uint32_t pcol = WIDE ? COL_P_128 + w * (NCOL / 2) : COL_P + w * (BN / 2);
                const int kk0 = WIDE ? w * (NCOL / 16) : 0;
                if constexpr (WIDE) {
                    // one N = 128 MMA per 16 keys over both 64-dim boxes of V (the
                    // descriptor's leading byte offset steps from one box to the next)
#pragma unroll
                    for (int kk = 0; kk < NCOL / 16; ++kk)
                        tc::mma_bf16_ta(tmem + COL_O + w * D, tmem + pcol + kk * 8,
                                        dv + (((kk0 + kk) * 2048) >> 4), idesc_pv128<T>(), kk > 0 || j > I.jb[w]);
                } else {
#pragma unroll
                    for (int kk = 0; kk < NCOL / 16; ++kk)
                        tc::mma_bf16_ta(tmem + COL_O + w * D, tmem + pcol + kk * 8,
                                        DSTEP ? dv + (((kk0 + kk) * 2048) >> 4) : tc::sw128_desc(va + (kk0 + kk) * 2048),
                                        idesc_pv<T>(), kk > 0 || j > I.jb[w]);
                }
                tc::commit(BAR(B_OF + w));
                tc::commit(BAR(B_KVE + st));
                return true;
            };
            if (!WIDE && w == 1 && I.je[0] - I.jb[0] >= LONG_ITEM_TILES - 1 && I.je[1] - I.jb[1] >= LONG_ITEM_TILES - 1) {
                // On a long item the second query tile starts a fraction of a key
                // tile after the first: both softmax warpgroups share each
                // sub-partition's exponential unit, and offset their exponentials
                // interleave instead of colliding (the offset carries through the
                // item; full-attention layer 1.88 -> 1.78 ms at 2000 cycles; with the
                // exponentials ahead of the P V wait 0 / 500 / 1000 / 2000 / 3200
                // cycles gave 1.775 / 1.743 / 1.629 / 1.640 / 1.657 ms).  A bounded
                // wait on the clock.
                const long long t0 = clock64();
                while (clock64() - t0 < TILE1_DELAY_CLOCKS) {}
            }
            bool ok = I.nkv == 0 || issue_qk(0);
            for (int j = 0; j < I.nkv && ok; ++j) {
                if (j + 1 < I.nkv && !issue_qk(j + 1)) ok = false;
                if (ok && !issue_pv(j)) ok = false;
            }
            if (!ok) break;
            g += I.nkv;
            if (mine) { cs += I.je[w] - I.jb[w] + 1; ++co; }
        }
    };
    auto softmax = [&]() {
        // ============ softmax (query tile w; at head dim 128 column half w) ============
        const int w = (warp - SOFTMAX_WARP0) >> 2;
        const int quarter = warp & 3;                  // TMEM lanes this warp may touch
        const int row = quarter * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_addr + COL_S + w * (WIDE ? NCOL : BN);
        const uint32_t tO = tmem + lane_addr + COL_O + w * D;
        const uint32_t tP = tmem + lane_addr + (WIDE ? COL_P_128 + w * (NCOL / 2) : COL_P + w * (BN / 2));
        uint32_t cs = 0, co = 0, g = 0;
        for (uint32_t kq = 0;; ++kq) {
            if (!wait_or_abort(BAR(B_IF + (kq & 1)), (kq >> 1) & 1, abort_flag, P.status)) break;
            const int t = item_ring[kq & 1];
            // the item's description stays in its ring entry, read from shared
            // memory where used (fewer live registers); the entry is released
            // once the item is done
            const RingItem I{sb + OFF_RING + (kq & 1) * (uint32_t)sizeof(Item)};
            auto release_item = [&]() {
                __syncwarp();
                if (lane == 0) mbar_arrive(BAR(B_IE + (kq & 1)));
            };
            if (t >= total_items || lds_volatile(abort_flag)) { release_item(); break; }
            const uint32_t g_item = g;                 // K/V stages of this item start at g_item
            g += I.nkv();
            const int rr = I.r0() + (WIDE ? 0 : w) * BM + row;   // query row within its sequence
            if (I.jb(w) > I.je(w)) {
                // past the sequence, or (paged) no key for any row of the tile: zero rows
                if (PAGED && rr < I.L()) {
                    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<T *>(P.out) + ((size_t)(I.s0() + rr) * P.H + I.h()) * HD);
#pragma unroll
                    for (int c = 0; c < HD / 8; ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
                }
                release_item();
                continue;
            }
            const int pos = rr + I.qoff();               // the row's key position
            int lo = 0, hi = I.Lk();                     // keys [lo, hi) kept for this row
            if (P.chunk > 0) { lo = pos / P.chunk * P.chunk; hi = min(hi, lo + P.chunk); }
            else if (P.window > 0) { lo = max(lo, pos - P.window + 1); hi = min(hi, pos + P.window); }
            if (P.causal) hi = min(hi, pos + 1);
            const float *rel = nullptr;                // rel[d]: bias of a key d positions before the row
            const float *trel = nullptr;               // the same, widened, in shared memory (tab_sm)
            int cap = 0;
            if constexpr (BIAS) {
                cap = P.num_buckets - 1;
                rel = P.rel_bias + (size_t)I.h() * (2 * cap + 1) + cap;
                trel = tab + I.h() * tab_span + (cap + BN - 1);
            }
            float m = -INFINITY, l = 0.f;
            bool ok = true;
            for (int j = I.jb(w); j <= I.je(w); ++j, ++cs) {
                if (!wait_or_abort(BAR(B_SF + w), cs & 1, abort_flag, P.status)) { ok = false; break; }
                tc::fence_after_sync();
                float x[NCOL];
                if constexpr (LD128) {
                    tc::tmem_ld128(tS, x);
                } else {
                    tc::tmem_ld64(tS, x);
                    if constexpr (NCOL == 128) tc::tmem_ld64(tS + 64, x + 64);
                }
                tc::fence_before_sync();
                mbar_arrive(BAR(B_SE + w));            // S columns free: QK of the next key tile may start
                const int c0 = I.c_lo() + j * BN + (WIDE ? w * NCOL : 0);   // the key of column 0
                if constexpr (PAGED) {
                    // V rows at k_end and beyond hold unread blocks or cache rows
                    // past the context (any bits): zero them so that P = 0 there
                    // contributes exactly nothing to P V
                    if (row >= I.k_end() - c0) {
                        const uint32_t vrow = sb + OFF_KV + ((g_item + j) % NS) * 2 * TKV + TKV + row * 128;
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(vrow + c * 16), "r"(0)
                                         : "memory");
                    }
                }
                // the relative-position bias: one value for the whole tile when
                // every key of it lies beyond the table's reach, else per key
                float boff = 0.f;
                if constexpr (BIAS) {
                    const int dhi = pos - c0, dlo = dhi - (BN - 1);
                    if (dlo >= cap) boff = __ldg(rel + cap);
                    else if (dhi <= -cap) boff = __ldg(rel - cap);
                    else if (tab_sm) {
                        const float *tr = trel + dhi;      // |dhi - i| < cap + BN in the band
#pragma unroll
                        for (int i = 0; i < BN; i += 2) add2(x[i], x[i + 1], tr[-i], tr[-i - 1]);
                    } else {
#pragma unroll
                        for (int i = 0; i < BN; ++i) x[i] += __ldg(rel + min(max(dhi - i, -cap), cap));
                    }
                    boff *= P.scale_log2;
                }
                // mask to the kept key range; tile max of the raw scores
                float mx[NCOL / 32];
                uint32_t dead = 0;                     // 32-key chunks no row of the warp keeps
                if constexpr (BAND) {
                    // banded masks (window, chunk, causal): per 32-key chunk, the
                    // warp's rows keep none of it, all of it, or part of it; only a
                    // part-kept chunk is masked key by key, a chunk kept by no row
                    // skips its max and (in write_p_tmem) its exponentials
                    const int ilo = lo - c0, ihi = hi - c0;
#pragma unroll
                    for (int k = 0; k < NCOL / 32; ++k) {
                        const int a = 32 * k;
                        if (__all_sync(kFull, ihi <= a || ilo >= a + 32)) {
                            dead |= 1u << k;
                            mx[k] = -INFINITY;
                            continue;
                        }
                        if (!__all_sync(kFull, ilo <= a && ihi >= a + 32)) {
                            const int lk = min(max(ilo - a, 0), 32), hk = min(max(ihi - a, 0), 32);
                            const uint32_t mw = (hk >= 32 ? 0xffffffffu : ((1u << hk) - 1u)) &
                                                ~(lk >= 32 ? 0xffffffffu : ((1u << lk) - 1u));
#pragma unroll
                            for (int i = 0; i < 32; ++i) x[a + i] = (mw & (1u << i)) ? x[a + i] : -INFINITY;
                        }
                        float a0 = x[a], a1 = x[a + 1];
#pragma unroll
                        for (int i = 2; i < 32; i += 2) { a0 = fmaxf(a0, x[a + i]); a1 = fmaxf(a1, x[a + i + 1]); }
                        mx[k] = fmaxf(a0, a1);
                    }
                } else {
                    const int ilo = lo - c0, ihi = hi - c0;
                    const bool masked = ilo > 0 || ihi < NCOL;
                    if (masked) {
                        uint32_t mw[NCOL / 32];
#pragma unroll
                        for (int k = 0; k < NCOL / 32; ++k) {
                            const int a = min(max(ilo - 32 * k, 0), 32), b = min(max(ihi - 32 * k, 0), 32);
                            const uint32_t hiw = b >= 32 ? 0xffffffffu : ((1u << b) - 1u);
                            const uint32_t low = a >= 32 ? 0xffffffffu : ((1u << a) - 1u);
                            mw[k] = hiw & ~low;
                        }
#pragma unroll
                        for (int i = 0; i < NCOL; ++i) x[i] = (mw[i >> 5] & (1u << (i & 31))) ? x[i] : -INFINITY;
                    }
#pragma unroll
                    for (int k = 0; k < NCOL / 32; ++k) {
                        float a0 = x[k * 32], a1 = x[k * 32 + 1];
#pragma unroll
                        for (int i = 2; i < 32; i += 2) { a0 = fmaxf(a0, x[k * 32 + i]); a1 = fmaxf(a1, x[k * 32 + i + 1]); }
                        mx[k] = fmaxf(a0, a1);
                    }
                }
                float mxt;
                if constexpr (NCOL == 128) mxt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                else mxt = fmaxf(mx[0], mx[1]);
                const float mt = mxt * P.scale_log2 + boff;
                // raise the running max only when it grows by more than 2^8
                const bool raise = mt > m + RESCALE_LOG2;
                const float m_old = m;
                if (raise) m = mt;
                if (!EARLYP && j > I.jb(w)) {
                    // P V of the previous key tile is done: P may be overwritten, O rescaled
                    if (!wait_or_abort(BAR(B_OF + w), (cs - 1) & 1, abort_flag, P.status)) { ok = false; break; }
                    tc::fence_after_sync();
                }
                if (raise) l *= ex2(m_old - m);
                // P = 2^(scale * s - m) as bf16 into the swizzled buffer; row sum in f32
                const float mneg = (m == -INFINITY ? 0.f : -m) + boff;
                if constexpr (EARLYP) {
                    uint32_t pk[NCOL / 2];
                    l += exp_pack<T, BAND, NCOL>(x, P.scale_log2, mneg, pk, dead);
                    if (j > I.jb(w)) {
                        if (!wait_or_abort(BAR(B_OF + w), (cs - 1) & 1, abort_flag, P.status)) { ok = false; break; }
                        tc::fence_after_sync();
                    }
#pragma unroll
                    for (int q4 = 0; q4 < NCOL / 32; ++q4) tc::tmem_st16(tP + q4 * (BN / 8), pk + q4 * (BN / 8));
                } else {
                    l += write_p_tmem<T, BAND>(x, P.scale_log2, mneg, tP, dead);
                }
                if (j > I.jb(w) && __any_sync(kFull, raise)) {
                    // the running max rose: bring this row's O to the new max (in TMEM)
                    const float c = raise ? ex2(m_old - m) : 1.f;
#pragma unroll
                    for (int x = 0; x < D; x += HD) {
                        float o[HD];
                        tc::tmem_ld64(tO + x, o);
#pragma unroll
                        for (int i = 0; i < HD; ++i) o[i] *= c;
                        tc::tmem_st64(tO + x, o);
                    }
                }
                if constexpr (PAGED) fence_proxy_async();   // zeroed V rows are read by the tensor cores
                tc::fence_before_sync();               // orders P and the O rescale before the next P V
                mbar_arrive(BAR(B_PF + w));
            }
            if (!ok) break;
            // all key tiles done: read O, free the O columns, normalise, store
            if (!wait_or_abort(BAR(B_OF + w), (cs - 1) & 1, abort_flag, P.status)) break;
            tc::fence_after_sync();
            if constexpr (WIDE) {
                // the two column halves of each row: trade (m, l) through shared
                // memory, then half w writes output dims 64 w .. 64 w + 63 from both
                // O accumulators, rescaled to the larger max
                float2 *mlx = reinterpret_cast<float2 *>(smem + OFF_OST);
                mlx[w * BM + row] = make_float2(m, l);
                mbar_arrive(BAR(B_MX + w));
                if (!wait_or_abort(BAR(B_MX + (1 - w)), co & 1, abort_flag, P.status)) break;
                const float2 oth = mlx[(1 - w) * BM + row];
                const float M = fmaxf(m, oth.x);
                const float as = M == -INFINITY ? 0.f : ex2(m - M), ao = M == -INFINITY ? 0.f : ex2(oth.x - M);
                const float L = l * as + oth.y * ao;
                const float inv = L > 0.f ? 1.f / L : 0.f;
                float o[HD], q[HD];
                tc::tmem_ld64(tmem + lane_addr + COL_O + w * D + w * HD, o);         // this half's O
                tc::tmem_ld64(tmem + lane_addr + COL_O + (1 - w) * D + w * HD, q);   // the other half's
                tc::fence_before_sync();
                mbar_arrive(BAR(B_OE));                // both O accumulators read by this warpgroup
                mbar_arrive(BAR(B_OE + 1));
                ++co;
                if (rr < I.L()) {
                    uint4 *dst = reinterpret_cast<uint4 *>(static_cast<T *>(P.out) +
                                                           ((size_t)(I.s0() + rr) * P.H + I.h()) * D + w * HD);
#pragma unroll
                    for (int c = 0; c < HD / 8; ++c) {
                        float v[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) v[e] = (o[c * 8 + e] * as + q[c * 8 + e] * ao) * inv;
                        dst[c] = Vec<T>::from_f32(v);
                    }
                }
                release_item();
                continue;
            }
            float o[HD];
            tc::tmem_ld64(tO, o);
            tc::fence_before_sync();
            mbar_arrive(BAR(B_OE + w));
            ++co;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const int tile0 = I.r0() + w * BM;            // the tile's first row within its sequence
            const int wrow0 = tile0 + quarter * 32;     // the warp's first row within its sequence
            if (TMA_OUT && wrow0 + 32 <= I.L()) {
                // the warp's 32 rows, all inside the sequence: into its quarter of the
                // 128-byte-swizzled staging tile, then one TMA store by its lane 0
                if (lane == 0) tc::bulk_wait_read_all();
                __syncwarp();
                const uint32_t srow = sb + OFF_OST + w * TILE_BYTES + row * 128;
#pragma unroll
                for (int c = 0; c < HD / 8; ++c) {
                    float v[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = o[c * 8 + e] * inv;
                    const uint4 u = Vec<T>::from_f32(v);
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(srow + ((c ^ (row & 7)) << 4)),
                                 "r"(u.x), "r"(u.y), "r"(u.z), "r"(u.w)
                                 : "memory");
                }
                fence_proxy_async();                   // the rows are read by the TMA engine
                __syncwarp();
                if (lane == 0) {
                    tc::tma_store_3d(&tm_o, 0, I.h(), I.s0() + wrow0, sb + OFF_OST + w * TILE_BYTES + quarter * 32 * 128);
                    tc::bulk_commit_group();
                }
            } else if (rr < I.L()) {
                // plain stores of the rows inside the sequence (its last, partial tile)
                uint4 *dst = reinterpret_cast<uint4 *>(static_cast<T *>(P.out) + ((size_t)(I.s0() + rr) * P.H + I.h()) * HD);
#pragma unroll
                for (int c = 0; c < HD / 8; ++c) {
                    float v[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) v[e] = o[c * 8 + e] * inv;
                    dst[c] = Vec<T>::from_f32(v);
                }
            }
            release_item();
        }
        (void)co;
        if (TMA_OUT && lane == 0) tc::bulk_wait_all();   // the staging tiles stay valid until the stores are done
    };
    if constexpr (SPLIT) {
        // a warpgroup changes its register count with all of its warps, before
        // its roles' code, so each role's code is compiled to its own count
        if (warp < 4) {
            regs_lower<REGS_COPY>();
            if (warp == 0 && (PAGED || lane == 0)) producer();
            else if ((warp == 1 || warp == MMA1_WARP) && lane == 0) mma_issuer();
            __syncwarp();
        } else {
            regs_raise<REGS_SOFTMAX>();
            softmax();
            __syncwarp();
            regs_lower<REGS_COPY>();                   // the teardown runs at warpgroup 0's count
        }
    } else {
        if (warp == 0 && lane == 0) producer();
        else if ((warp == 1 || warp == MMA1_WARP) && lane == 0) mma_issuer();
        else if (warp >= SOFTMAX_WARP0 && warp < SOFTMAX_WARP0 + 8) softmax();
    }

    // ---- teardown: every role is done with TMEM --------------------------------
    tc::fence_before_sync();
    __syncthreads();
    if (dyn && threadIdx.x == 0) {
        // the last CTA to finish returns the counters to zero (all fetches of
        // every CTA precede its arrival here), also after an abort
        __threadfence();
        if (atomicAdd(P.items + 1, 1u) == gridDim.x - 1) {
            __threadfence();
            P.items[0] = 0u;
            P.items[1] = 0u;
        }
    }
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// Item counters of prefill launches.  An eager launch takes the next of
// PREFILL_SLOTS pairs in turn (zero between launches: the last CTA of a launch
// resets its pair), so eager launches that may run at the same time use
// different pairs as long as fewer than PREFILL_SLOTS are in flight at once.
// A launch captured into a CUDA graph keeps its pair for every replay, so it
// takes a pair of its own from CAPTURE_SLOTS pairs that are never handed out
// again; once those are used up, captured launches get no pair and deal items
// statically (CTA c takes items c, c + G, ...), which needs no counter.
constexpr int PREFILL_SLOTS = 1024;
constexpr int CAPTURE_SLOTS = 8192;
__device__ unsigned g_item_counters[2 * PREFILL_SLOTS];
__device__ unsigned g_capture_counters[2 * CAPTURE_SLOTS];

struct CounterArrays {
    void *ctx;                    // the context the addresses belong to
    unsigned *eager, *captured;   // device addresses of the two arrays there
};

// The two arrays' device addresses in the current context (looked up once per
// device, and again for a context that replaced the cached one).
bool counter_arrays(unsigned **eager, unsigned **captured)
{
    static std::mutex mu;
    static CounterArrays cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> lock(mu);
    CounterArrays &c = cache[dev];
    void *ctx = current_context();
    if (c.eager == nullptr || ctx == nullptr || c.ctx != ctx) {
        void *a = nullptr, *b = nullptr;
        if (cudaGetSymbolAddress(&a, g_item_counters) != cudaSuccess ||
            cudaGetSymbolAddress(&b, g_capture_counters) != cudaSuccess)
            return false;
        c.eager = static_cast<unsigned *>(a);
        c.captured = static_cast<unsigned *>(b);
        c.ctx = current_context();
    }
    *eager = c.eager;
    *captured = c.captured;
    return true;
}

// The counter pair of the next launch on `stream`: *pair = NULL (with true)
// means a captured launch past CAPTURE_SLOTS, which deals items statically.
bool next_item_counters(cudaStream_t stream, unsigned **pair)
{
    static std::atomic<unsigned> next_eager{0}, next_captured{0};
    unsigned *eager = nullptr, *captured = nullptr;
    if (!counter_arrays(&eager, &captured)) return false;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return false;
    if (cs == cudaStreamCaptureStatusActive) {
        const unsigned i = next_captured.fetch_add(1u);
        *pair = i < (unsigned)CAPTURE_SLOTS ? captured + 2 * i : nullptr;
        return true;
    }
    *pair = eager + 2 * (next_eager.fetch_add(1u) % PREFILL_SLOTS);
    return true;
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
bool make_map(CUtensorMap *m, const void *base, int T, int H, CUtensorMapDataType dt, int rows = BM, int d = HD)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)H * d * 2};
    const cuuint32_t box[3] = {HD, 1, (cuuint32_t)rows};   // 64 dims (128 bytes, the swizzle span) per box
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [num_blocks, H, 16, 64] bf16 paged cache -> boxes of one block (16 rows x
// 64 dims) of one head, 128-byte swizzle
bool make_paged_map(CUtensorMap *m, const void *base, int num_blocks, int H, CUtensorMapDataType dt)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)HD, (cuuint64_t)CBS, (cuuint64_t)H, (cuuint64_t)num_blocks};
    const cuuint64_t strides[3] = {(cuuint64_t)HD * 2, (cuuint64_t)CBLK_BYTES, (cuuint64_t)H * CBLK_BYTES};
    const cuuint32_t box[4] = {HD, CBS, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, dt, 4, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T, bool PAGED, bool BIAS, bool BAND, int D = 64>
cudaError_t launch_cfg(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mo,
                       Params P, const PrefillArgs &a, int sms, cudaStream_t stream)
{
    auto kern = swa_prefill_tc_kernel<T, PAGED, BIAS, BAND, D>;
    constexpr bool SPLIT = PAGED || BIAS;
    constexpr uint32_t SMEM_BYTES = Layout<nstages<PAGED, D>(), own_table<PAGED, BIAS>(), D>::SMEM_BYTES;
    constexpr int QT = D == 128 ? 1 : 2;              // query tiles per item
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [&] {
        attr = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (attr == cudaSuccess && SPLIT) {
            // the softmax warpgroups' raise is granted from what warpgroup 0 lowers;
            // a build that launched with fewer registers a thread than the split
            // assumes would leave the raise waiting forever: refuse to launch it
            cudaFuncAttributes fa;
            attr = cudaFuncGetAttributes(&fa, kern);
            if (attr == cudaSuccess && REGS_COPY + 2 * REGS_SOFTMAX > 3u * (unsigned)fa.numRegs)
                attr = cudaErrorLaunchOutOfResources;
        }
    });
    if (attr != cudaSuccess) return attr;
    for (int base = 0; base < a.num_seqs; base += MAX_SEQS) {
        P.num_seqs = std::min(MAX_SEQS, a.num_seqs - base);
        P.cu_seqlens = a.cu_seqlens + base;
        if (PAGED) {
            P.context_lens = a.context_lens + base;
            P.block_tables = a.block_tables + (size_t)base * a.mbps;
        }
        const long long tiles_upper = (long long)P.num_seqs * ((a.max_seqlen + QT * BM - 1) / (QT * BM)) * a.num_heads;
        const int grid = (int)std::max<long long>(1, std::min<long long>(sms, tiles_upper));
        if (!next_item_counters(stream, &P.items)) return cudaErrorInvalidDevice;
        kern<<<grid, nthreads<SPLIT>(), SMEM_BYTES, stream>>>(mq, mk, mv, mo, P);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <typename T>
cudaError_t dispatch(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mo,
                     const Params &P, const PrefillArgs &a, int sms, bool paged, bool bias, cudaStream_t stream)
{
    if (paged) return bias ? launch_cfg<T, true, true, false>(mq, mk, mv, mo, P, a, sms, stream)
                           : launch_cfg<T, true, false, false>(mq, mk, mv, mo, P, a, sms, stream);
    if (bias) return launch_cfg<T, false, true, false>(mq, mk, mv, mo, P, a, sms, stream);
    // packed keys without bias: a sliding window takes the instance that
    // classifies 32-key chunks (a third of a window item's chunks are kept by no
    // row of the warp); full, chunked and causal attention keep the plain one,
    // where few tiles are masked and the extra code costs more than it saves
    if (a.head_dim == 128)
        return a.window > 0 ? launch_cfg<T, false, false, true, 128>(mq, mk, mv, mo, P, a, sms, stream)
                            : launch_cfg<T, false, false, false, 128>(mq, mk, mv, mo, P, a, sms, stream);
    if (a.window > 0) return launch_cfg<T, false, false, true>(mq, mk, mv, mo, P, a, sms, stream);
    return launch_cfg<T, false, false, false>(mq, mk, mv, mo, P, a, sms, stream);
}

}  // namespace

cudaError_t launch_swa_prefill(const PrefillArgs &a, cudaStream_t stream)
{
    const bool paged = a.block_tables != nullptr;
    // head dim 64, or 128 for packed keys without bias
    if (a.head_dim != HD && !(a.head_dim == 128 && !paged && a.rel_bias == nullptr)) return cudaErrorInvalidValue;
    const int d = a.head_dim;
    const CUtensorMapDataType dt =
        a.dtype == PKA_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUtensorMap mq, mk, mv, mo;
    if (!make_map(&mq, a.q, a.num_tokens, a.num_heads, dt, BM, d) ||
        !make_map(&mo, a.out, a.num_tokens, a.num_heads, dt, 32, d))
        return cudaErrorInvalidValue;
    if (paged) {
        if (!make_paged_map(&mk, a.k, a.num_blocks, a.num_heads, dt) ||
            !make_paged_map(&mv, a.v, a.num_blocks, a.num_heads, dt))
            return cudaErrorInvalidValue;
    } else if (!make_map(&mk, a.k, a.num_tokens, a.num_heads, dt, BN, d) ||
               !make_map(&mv, a.v, a.num_tokens, a.num_heads, dt, BN, d)) {
        return cudaErrorInvalidValue;
    }
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    Params P;
    P.out = a.out;
    P.status = a.status;
    P.scale_log2 = a.scale * 1.4426950408889634f;
    P.num_tokens = a.num_tokens;
    P.H = a.num_heads;
    P.window = a.window;
    P.causal = a.causal;
    P.chunk = a.chunk;
    P.context_lens = nullptr;
    P.block_tables = nullptr;
    P.rel_bias = a.rel_bias;
    P.num_buckets = a.rel_bias ? a.num_buckets : 0;
    P.mbps = a.mbps;
    P.num_blocks = a.num_blocks;
    const bool bias = a.rel_bias != nullptr;
    return a.dtype == PKA_F16 ? dispatch<__half>(mq, mk, mv, mo, P, a, sms, paged, bias, stream)
                              : dispatch<__nv_bfloat16>(mq, mk, mv, mo, P, a, sms, paged, bias, stream);
}

}  // namespace pka
