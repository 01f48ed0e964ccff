// paged_decode.cu — single-query paged-KV attention with optional materialised
// bias and optional causal sliding window, split-K over the visible blocks.
//
// Computes, per (sequence s, head h), the formula of "PagedAttention: Support
// custom attention bias for T5 model (1/2)" (opening section):
//   out = softmax(scale * (q K^T + A)) V
// over the keys [start, ctx) with start = max(0, ctx - W) for a window W
// ("[V1] Add sliding window support to Flex Attention backend"), K/V gathered
// through the block table passed in (decoder self-attention and encoder
// cross-attention each pass their own: "Add Encoder-decoder model support and
// T5 Model support").  A NULL bias is a no-op: no bias bytes are touched.
//
// Design (memory-bound; everything below is about keeping HBM busy):
//  * Work unit = (s, h, partition): `part_blocks` consecutive cache blocks of
//    the visible range.  The unit list is the prefix sum over sequences of
//    H * num_partitions(s), built by every CTA into shared memory at start
//    (one read of context_lens); a sequence's units run partition-major, so
//    neighbouring warps stream neighbouring heads of the same cache blocks.
//    Warp gw takes units gw and gw + nwt; any further units are handed out
//    one at a time by a wrapping atomic counter, so the warps that stream
//    faster take more of them.
//  * Persistent grid (SMs x resident CTAs); every warp is an independent
//    streaming pipeline over its units with NSTAGE shared-memory stages.
//    Per stage: the K and V runs of one (block, head) — each a contiguous
//    block_size * D run — arrive by two bulk copies on the TMA engine; the
//    bias slice (16 floats, zero-filled outside [start, ctx)) and, at a
//    unit's first block, the query row arrive by per-lane async copies.  One
//    mbarrier per stage counts both (32 lane arrivals + the bulk bytes).
//    Loads run up to NSTAGE blocks ahead of the math and across unit
//    boundaries; block-table entries of the next unit are fetched one unit
//    ahead, and the math side follows the copy side's unit ids through a
//    ring of lane registers.  Block-table entries and blocks outside the
//    window are never read.
//  * Math per block: 2 lanes per key compute q.k from 16-byte shared loads
//    with mixed-precision FMA (bf16 / f16 operands, f32 accumulate; chunk
//    order rotated per key: no bank conflicts), online softmax in the log2
//    domain (ex2.approx), P.V with one 16-byte V load per lane per row group.
//    In a block at the window's start or the context's end, the V rows of
//    keys outside [start, ctx) are replaced by zeros before P.V: those cache
//    rows may hold any bits (an unwritten tail, NaN included).
//  * Bias: a materialised A (streamed with the keys), or the T5 table read
//    from shared memory at column min(ctx-1-j, buckets-1), or none.
//  * A unit that is its (s, h)'s only partition writes `out` directly.  Else
//    it writes (m, l, acc) to the workspace and bumps a per-(s, h) counter with
//    atomicInc(npart - 1), which wraps to zero: the last partition to arrive
//    merges all partials (every load of a chunk of partials issued at once),
//    writes `out` and zeroes the slots it read.  The unit counter wraps to
//    zero as well, so a call leaves the whole workspace zero, ready for the
//    next call of any shape.
//  * A launch may carry two problems (a decode step's self- and
//    cross-attention, each with its own tables, caches and workspace); the
//    unit list runs over the concatenated sequences.
//  * Fused append: a problem may bring its newest token's K/V (position
//    ctx-1).  The unit that covers the last block patches that row into the
//    staged block once the bulk copy has landed and stores it to the cache
//    slot, so one launch does the KV caching and the attention of a step.
//  * Batches of at most one (sequence, head) pair per SM run a second kernel
//    of the same per-block math: one CTA per pair, its blocks dealt to the
//    CTA's warps, the warps' partial states merged in shared memory.
//  * Both kernels are launched with programmatic stream serialization: each
//    CTA lets the next launch in the stream start at once and waits
//    (griddepcontrol.wait) before its first global read, so a launch's CTAs
//    take the SMs the previous grid's CTAs leave during its split-K tail
//    while every input written by an earlier kernel is read only after that
//    kernel has completed (T5-small-shaped step 11.2 -> 11.0 us).

#include <algorithm>
#include <cmath>
#include <mutex>

#include "pka_device.cuh"
#include "pka_launch.h"

namespace pka {
namespace {

constexpr int BS = 16;                   // tokens per cache block (the only size built)
constexpr int MAX_SEQS_PER_LAUNCH = 1024;
constexpr int MAX_TABLE_FLOATS = PKA_MAX_BIAS_TABLE;   // T5 table cached in shared memory

template <typename T, int D> struct Tr {
    static constexpr int ELT = sizeof(T);
    static constexpr int ROW = D * ELT;              // bytes of one K or V row
    static constexpr int NC = ROW / 16;              // 16-byte chunks per row: 8, 16, 32
    static constexpr int EPC = 16 / ELT;             // elements per chunk
    static constexpr int CHUNK = BS * ROW;           // bytes of one (block, head) run
    static constexpr int QCH = NC / 2;               // chunks per lane in q.k (2 lanes per key)
    static constexpr int QSWZ = QCH >= 8 ? 4 : 0;    // extra chunk rotation of the second half-row
    static constexpr int RPI = 32 / NC;              // V rows per warp-wide 16-byte load
    static constexpr int PV_IT = BS / RPI;           // P.V iterations per block
    static constexpr int DPL = D / 32;               // dims per lane in the partition merge
    static constexpr int MCH = 32 / DPL;             // split-K partials merged per L2 round trip
    // stage layout
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = CHUNK;
    static constexpr int B_OFF = 2 * CHUNK;          // 16 floats of bias
    static constexpr int Q_OFF = 2 * CHUNK + 64;     // one query row
    static constexpr int STAGE = ((Q_OFF + ROW) + 127) / 128 * 128;
    static_assert(NC % 8 == 0 && 32 % NC == 0, "row must be 8, 16 or 32 chunks");
};

// n / d for any 32-bit unsigned n and a divisor fixed per launch, by one
// high multiply, a subtract, an add and two shifts (division by invariant
// integers using multiplication, Granlund and Montgomery 1994): a runtime
// integer division costs a ~200-cycle dependent chain, which the unit lookup
// and the partition counts would otherwise pay on every warp's first load.
struct FastDiv {
    uint32_t m, s1, s2;
    __device__ __forceinline__ uint32_t div(uint32_t n) const
    {
        const uint32_t t = __umulhi(m, n);
        return (t + ((n - t) >> s1)) >> s2;
    }
};

// d in [1, 2^31): l = ceil(log2 d), m = floor(2^32 (2^l - d) / d) + 1.
static inline FastDiv make_fastdiv(uint32_t d)
{
    int l = 0;
    while ((1ull << l) < d) ++l;
    FastDiv f;
    f.m = (uint32_t)((((1ull << 32) * ((1ull << l) - d)) / d) + 1);
    f.s1 = l < 1 ? (uint32_t)l : 1u;
    f.s2 = l > 1 ? (uint32_t)(l - 1) : 0u;
    return f;
}

// One decode problem of a launch: decoder self-attention and encoder
// cross-attention of a step are two problems with their own block tables.
constexpr int MAX_PROBLEMS = 2;
struct Prob {
    void *out;
    const unsigned char *q, *k_cache, *v_cache;
    const int32_t *block_tables, *context_lens;
    const float *bias;
    const float *bias_table;     // [H, num_buckets] T5 relative-position table, or NULL
    const unsigned char *k_new, *v_new;   // [S, H, D] newest token's K/V (position ctx-1), or NULL
    unsigned *counters;
    float2 *ws_ml;
    float *ws_acc;
    float scale_log2;
    int window, seq_base, num_seqs, mbps, num_blocks, max_ctx, part_blocks, max_parts, num_buckets;
    long long bias_stride;
    FastDiv by_part_blocks;
};

struct Params {
    Prob pr[MAX_PROBLEMS];
    int nprob;
    int num_seqs;                // sequences of this launch over all problems (problem 0's first)
    int H;
    FastDiv by_H;
    unsigned *queue;             // unit hand-out counter (problem 0's workspace), zero between calls
    int32_t *status;
};

struct Unit {
    int s;       // sequence index within this launch
    int prob;    // which problem
    int gs;      // sequence index within that problem
    int h, p, npart, ctx, start, b0, nb;
};

__device__ __forceinline__ int prob_of(int s, const Params &P) { return (P.nprob > 1 && s >= P.pr[0].num_seqs) ? 1 : 0; }

// The sequence s of unit u: cum[s] <= u < cum[s + 1].  Called by a whole
// warp with the same u: lane i tests the i-th of 32 evenly spaced candidates,
// so 1024 sequences take two shared-memory rounds.
__device__ __forceinline__ int seq_of_warp(int u, const int *cum, int num_seqs)
{
    int lo = 0, n = num_seqs;                         // cum[lo] <= u < cum[lo + n]
    while (n > 1) {
        const int step = (n + 31) >> 5;
        const int idx = lo + (int)(threadIdx.x & 31) * step;
        const unsigned m = __ballot_sync(kFull, idx < lo + n && cum[idx] <= u);
        const int nlo = lo + (__popc(m) - 1) * step;   // candidates at or below u form a prefix
        n = min(step, lo + n - nlo);
        lo = nlo;
    }
    return lo;
}

// Unit u of sequence s -> (h, p) and its block range.
__device__ __forceinline__ Unit unit_in_seq(int u, int s, const int *cum, const int *ctxs, const Params &P)
{
    Unit U;
    U.s = s;
    U.prob = prob_of(s, P);
    const Prob &R = P.pr[U.prob];
    U.gs = R.seq_base + s - (U.prob ? P.pr[0].num_seqs : 0);
    U.npart = (int)P.by_H.div((uint32_t)(cum[s + 1] - cum[s]));
    const int r = u - cum[s];
    U.p = (int)P.by_H.div((uint32_t)r);
    U.h = r - U.p * P.H;
    U.ctx = ctxs[s];
    U.start = (R.window > 0 && U.ctx > R.window) ? U.ctx - R.window : 0;
    if (U.ctx == 0) {
        U.b0 = 0; U.nb = 0;
    } else {
        const int last = (U.ctx - 1) / BS;
        U.b0 = U.start / BS + U.p * R.part_blocks;
        U.nb = min(R.part_blocks, last + 1 - U.b0);
    }
    return U;
}

__device__ __forceinline__ Unit unit_of(int u, const int *cum, const int *ctxs, const Params &P)
{
    return unit_in_seq(u, seq_of_warp(u, cum, P.num_seqs), cum, ctxs, P);
}

__device__ __forceinline__ int load_bt(const Unit &U, const Params &P, int lane)
{
    if (lane < U.nb)
        return __ldg(P.pr[U.prob].block_tables + (size_t)U.gs * P.pr[U.prob].mbps + U.b0 + lane);
    return 0;
}

// q.k for one key: this lane's half-row (QCH chunks of 16 bytes) against the
// query half-row kept in registers; partial sums in two chains.
template <typename T, int D> struct Dot {
    using R = Tr<T, D>;
    // query registers: packed 16-bit pairs, or f32
    struct Q { uint32_t w[R::QCH][4]; };
    __device__ __forceinline__ static void load_q(Q &q, const unsigned char *qrow, int first, int rot)
    {
#pragma unroll
        for (int m = 0; m < R::QCH; ++m) {
            const uint4 v = *reinterpret_cast<const uint4 *>(qrow + (first + ((m + rot) & (R::QCH - 1))) * 16);
            q.w[m][0] = v.x; q.w[m][1] = v.y; q.w[m][2] = v.z; q.w[m][3] = v.w;
        }
    }
    __device__ __forceinline__ static float dot(const Q &q, const unsigned char *krow, int first, int rot)
    {
        float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int m = 0; m < R::QCH; ++m) {
            const uint4 k = *reinterpret_cast<const uint4 *>(krow + (first + ((m + rot) & (R::QCH - 1))) * 16);
            if constexpr (sizeof(T) == 4) {
                a0 = fmaf(__uint_as_float(q.w[m][0]), __uint_as_float(k.x), a0);
                a1 = fmaf(__uint_as_float(q.w[m][1]), __uint_as_float(k.y), a1);
                a2 = fmaf(__uint_as_float(q.w[m][2]), __uint_as_float(k.z), a2);
                a3 = fmaf(__uint_as_float(q.w[m][3]), __uint_as_float(k.w), a3);
            } else {
                fma2_mixed<T>(q.w[m][0], k.x, a0, a1);
                fma2_mixed<T>(q.w[m][1], k.y, a2, a3);
                fma2_mixed<T>(q.w[m][2], k.z, a0, a1);
                fma2_mixed<T>(q.w[m][3], k.w, a2, a3);
            }
        }
        return (a0 + a1) + (a2 + a3);
    }
};

template <typename T, int D, int NSTAGE, int NW>
__global__ void __launch_bounds__(NW * 32, 1) paged_decode_kernel(const Params P)
{
    using R = Tr<T, D>;
    using DT = Dot<T, D>;
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    unsigned char *stages = smem + (size_t)warp * NSTAGE * R::STAGE;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)NW * NSTAGE * R::STAGE) + warp * NSTAGE;
    int *cum = reinterpret_cast<int *>(smem + (size_t)NW * NSTAGE * R::STAGE + NW * NSTAGE * 8);
    int *ctxs = cum + P.num_seqs + 1;
    float *table_sm = reinterpret_cast<float *>(ctxs + P.num_seqs);
    // the next launch may start its CTAs as this grid's CTAs leave the SMs;
    // nothing an earlier kernel wrote is read before that kernel has finished
    griddep_launch_dependents();
    griddep_wait();

    // ---- per-sequence partition counts -> prefix sums (whole CTA) ----------
    for (int s = threadIdx.x; s < P.num_seqs; s += blockDim.x) {
        const int pi = prob_of(s, P);
        const Prob &R = P.pr[pi];
        int c = __ldg(R.context_lens + R.seq_base + s - (pi ? P.pr[0].num_seqs : 0));
        if (c < 0 || c > R.max_ctx || c > R.mbps * BS) {
            flag_status(P.status, PKA_DEVCHK_CONTEXT_LEN);
            c = c < 0 ? 0 : min(c, min(R.max_ctx, R.mbps * BS));
        }
        ctxs[s] = c;
        int npart = 1;
        if (c > 0) {
            const int start = (R.window > 0 && c > R.window) ? c - R.window : 0;
            const int nblk = (c - 1) / BS - start / BS + 1;
            npart = min((int)R.by_part_blocks.div((uint32_t)(nblk + R.part_blocks - 1)), R.max_parts);
        }
        cum[s + 1] = npart * P.H;
    }
    // a T5 bias table is cached in shared memory; when both problems of a
    // launch use one, the host has checked that it is the same table
    {
        const Prob &TP = P.pr[(P.nprob > 1 && P.pr[0].bias_table == nullptr) ? 1 : 0];
        if (TP.bias_table)
            for (int i = threadIdx.x; i < P.H * TP.num_buckets; i += blockDim.x) table_sm[i] = __ldg(TP.bias_table + i);
    }
    if (lane == 0)
        for (int i = 0; i < NSTAGE; ++i) mbar_init(smem_u32(&bars[i]), 32);
    fence_barrier_init();
    __syncthreads();
    if (warp == 0) {
        // chunked inclusive scan of cum[1..S] by one warp
        const int per = (P.num_seqs + 31) / 32;
        const int a = min(lane * per, P.num_seqs), b = min(a + per, P.num_seqs);
        int local = 0;
        for (int i = a; i < b; ++i) local += cum[i + 1];
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += v;
        }
        int run = incl - local;
        for (int i = a; i < b; ++i) { run += cum[i + 1]; cum[i + 1] = run; }
        if (lane == 0) cum[0] = 0;
    }
    __syncthreads();

    const int total_units = cum[P.num_seqs];
    const int gw = blockIdx.x * NW + warp;
    const int nwt = gridDim.x * NW;
    if (gw >= total_units) return;                    // no CTA-wide sync after this point


    // ---- producer state (issue side) ---------------------------------------
    // A warp takes units gw and gw + nwt; when the launch has more than two
    // rounds of units the rest are handed out one at a time by an atomic
    // counter, so warps that stream faster take more of them (a static
    // round-robin left the slowest warps running alone for the last fifth of
    // a large launch).  The counter wraps to zero after the launch's
    // total_units - nwt requests (each warp's last request overshoots once).
    const bool dyn = total_units > 2 * nwt;
    unsigned fut = 0;                                  // lane 0: the counter's answer for the next request
    auto request = [&]() {
        if (lane == 0) fut = atom_inc_relaxed(P.queue, (unsigned)(total_units - nwt - 1));
    };
    if (dyn) request();
    // The ids of the non-empty units this warp streams, in order: lane i % 32
    // holds the i-th (the copy side is at most NSTAGE blocks ahead).
    int ring = 0;
    uint32_t ring_n = 0;
    auto ring_push = [&](int id) {
        if (lane == (int)(ring_n & 31)) ring = id;
        ++ring_n;
    };
    int pk = 0;                                        // unit ordinal of the issue side
    Unit pu = unit_of(gw, cum, ctxs, P);
    const Unit first_unit = pu;                       // the consumer's first unit, when not empty
    if (pu.nb > 0) ring_push(gw);
    int pbt = load_bt(pu, P, lane);
    int pn_id = gw + nwt;
    bool p_next_ok = pn_id < total_units;
    Unit pn = pu;
    int pnbt = 0;
    if (p_next_ok) {
        pn = unit_of(pn_id, cum, ctxs, P);
        pnbt = load_bt(pn, P, lane);
        if (pn.nb > 0) ring_push(pn_id);
    }
    bool p_active = true;
    int pib = 0;
    auto p_advance_unit = [&]() {
        if (pu.nb == 0 && lane < R::NC)                // a sequence without keys: zero output row
            reinterpret_cast<uint4 *>(static_cast<unsigned char *>(P.pr[pu.prob].out) +
                                      ((size_t)pu.gs * P.H + pu.h) * R::ROW)[lane] = make_uint4(0u, 0u, 0u, 0u);
        ++pk;
        if (!p_next_ok) { p_active = false; return; }
        pu = pn; pbt = pnbt; pib = 0;
        if (dyn && pk + 1 >= 2) {
            pn_id = 2 * nwt + __shfl_sync(kFull, (int)fut, 0);
            if (pn_id < total_units) request();
        } else {
            pn_id = gw + (pk + 1) * nwt;
        }
        p_next_ok = pn_id < total_units;
        if (p_next_ok) {
            pn = unit_of(pn_id, cum, ctxs, P);
            pnbt = load_bt(pn, P, lane);
            if (pn.nb > 0) ring_push(pn_id);
        }
    };
    while (p_active && pu.nb == 0) p_advance_unit();

    // ---- consumer state ------------------------------------------------------
    // q.k lanes: key = lane / 2, half = lane % 2; chunk order rotated per key
    // so the 8 lanes of a quarter-warp always hit 8 different bank groups.
    const int key = lane >> 1, half = lane & 1;
    const int q_first = half * R::QCH;
    const int q_rot = (key & 3) + half * R::QSWZ;
    // P.V lanes: row = it * RPI + vr, 16-byte column vc
    const int vr = lane / R::NC, vc = lane % R::NC;
    typename DT::Q qreg;
    float acc[R::EPC];
    float m_run = -INFINITY, l_run = 0.f;
    uint32_t issued = 0, consumed = 0;
    const uint32_t st_base = smem_u32(stages);

    auto top_up = [&]() {
        while (p_active && issued - consumed < (uint32_t)NSTAGE) {
            const int stage = issued % NSTAGE;
            const uint32_t st = st_base + stage * R::STAGE;
            const uint32_t bar = smem_u32(&bars[stage]);
            const Prob &PP = P.pr[pu.prob];
            int phys = __shfl_sync(kFull, pbt, pib);
            if ((unsigned)phys >= (unsigned)PP.num_blocks) {
                if (lane == 0) flag_status(P.status, PKA_DEVCHK_BLOCK_ID);
                phys = 0;
            }
            const int gs = pu.gs;
            if (lane == 0) {
                mbar_expect_tx(bar, 2 * R::CHUNK);
                const size_t off = ((size_t)phys * P.H + pu.h) * (size_t)R::CHUNK;
                bulk_g2s(st + R::K_OFF, PP.k_cache + off, R::CHUNK, bar);
                bulk_g2s(st + R::V_OFF, PP.v_cache + off, R::CHUNK, bar);
            }
            if (PP.bias != nullptr && lane < BS) {
                const int j = (pu.b0 + pib) * BS + lane;
                const bool ok = j >= pu.start && j < pu.ctx;
                const float *src = PP.bias + ((size_t)gs * P.H + pu.h) * PP.bias_stride + (ok ? j : 0);
                cp_async_4(st + R::B_OFF + lane * 4, src, ok ? 4u : 0u);
            }
            if (pib == 0 && lane < R::NC)
                cp_async_16(st + R::Q_OFF + lane * 16, PP.q + ((size_t)gs * P.H + pu.h) * R::ROW + lane * 16);
            cp_async_arrive_noinc(bar);
            ++issued;
            if (++pib >= pu.nb) {
                p_advance_unit();
                while (p_active && pu.nb == 0) p_advance_unit();
            }
        }
    };

    for (uint32_t ck = 0; ck < ring_n; ++ck) {       // ring_n grows as the copy side advances
        const int u = (ck == 0 && first_unit.nb > 0) ? gw : __shfl_sync(kFull, ring, (int)(ck & 31));
        const Unit cu = u == gw ? first_unit : unit_of(u, cum, ctxs, P);
        const Prob &CP = P.pr[cu.prob];
        const bool has_bias = CP.bias != nullptr, has_table = CP.bias_table != nullptr;
        // append: the sequence's newest token (position ctx-1) lies in the last
        // block of its last partition; its K/V row comes from k_new / v_new,
        // replaces the cache row in the staged block and is written to the cache
        const bool append = CP.k_new != nullptr && cu.p == cu.npart - 1 && cu.nb > 0;
        uint4 kn = make_uint4(0u, 0u, 0u, 0u), vn = kn;
        int app_phys = -1;
        if (append) {
            const size_t rowoff = ((size_t)cu.gs * P.H + cu.h) * R::ROW;
            if (lane < R::NC) {
                kn = __ldg(reinterpret_cast<const uint4 *>(CP.k_new + rowoff) + lane);
                vn = __ldg(reinterpret_cast<const uint4 *>(CP.v_new + rowoff) + lane);
            }
            app_phys = __ldg(CP.block_tables + (size_t)cu.gs * CP.mbps + (cu.ctx - 1) / BS);
        }
        m_run = -INFINITY;
        l_run = 0.f;
#pragma unroll
        for (int e = 0; e < R::EPC; ++e) acc[e] = 0.f;

        for (int cb = 0; cb < cu.nb; ++cb) {
            top_up();
            const int stage = consumed % NSTAGE;
            const unsigned char *stp = stages + stage * R::STAGE;
            if (!mbar_wait_bounded(smem_u32(&bars[stage]), (consumed / NSTAGE) & 1)) {
                if (lane == 0) flag_status(P.status, PKA_DEVCHK_TIMEOUT);
                return;
            }
            if (append && cb == cu.nb - 1) {
                const int r = (cu.ctx - 1) % BS;
                if (lane < R::NC) {
                    unsigned char *row = stages + stage * R::STAGE + r * R::ROW;
                    reinterpret_cast<uint4 *>(row + R::K_OFF)[lane] = kn;
                    reinterpret_cast<uint4 *>(row + R::V_OFF)[lane] = vn;
                    if ((unsigned)app_phys < (unsigned)CP.num_blocks) {
                        const size_t off = (((size_t)app_phys * P.H + cu.h) * BS + r) * R::ROW;
                        reinterpret_cast<uint4 *>(const_cast<unsigned char *>(CP.k_cache) + off)[lane] = kn;
                        reinterpret_cast<uint4 *>(const_cast<unsigned char *>(CP.v_cache) + off)[lane] = vn;
                    } else if (lane == 0) {
                        flag_status(P.status, PKA_DEVCHK_BLOCK_ID);
                    }
                    fence_proxy_async();         // before a later bulk copy refills this stage
                }
                __syncwarp();
            }
            if (cb == 0) DT::load_q(qreg, stp + R::Q_OFF, q_first, q_rot);
            // score of key `key` (both lanes of the pair end with the full sum)
            float d = DT::dot(qreg, stp + R::K_OFF + key * R::ROW, q_first, q_rot);
            d += __shfl_xor_sync(kFull, d, 1);
            const int j = (cu.b0 + cb) * BS + key;
            float bv = 0.f;
            if (has_bias) {
                bv = reinterpret_cast<const float *>(stp + R::B_OFF)[key];
            } else if (has_table) {
                // T5 relative position: distance ctx-1-j, capped at the last column
                const int dist = min(max(cu.ctx - 1 - j, 0), CP.num_buckets - 1);
                bv = table_sm[cu.h * CP.num_buckets + dist];
            }
            const float x = (j >= cu.start && j < cu.ctx) ? (d + bv) * CP.scale_log2 : -INFINITY;
            float mb = fmaxf(x, __shfl_xor_sync(kFull, x, 2));
            mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, 4));
            mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, 8));
            mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, 16));
            const float m_new = fmaxf(m_run, mb);
            const float corr = ex2(m_run - m_new);
            const float p = ex2(x - m_new);
            l_run = fmaf(l_run, corr, p);
            m_run = m_new;
#pragma unroll
            for (int e = 0; e < R::EPC; ++e) acc[e] *= corr;
            // A block at the window's start or the context's end holds rows
            // outside [start, ctx): cache rows that were never written, or
            // were written for another request, may hold any bits (NaN, Inf).
            // Their weight is 0, and their V row is replaced by zeros, so
            // such a row contributes exactly nothing (0 * NaN would be NaN).
            const int jb0 = (cu.b0 + cb) * BS;
            const bool edge = jb0 < cu.start || jb0 + BS > cu.ctx;
#pragma unroll
            for (int it = 0; it < R::PV_IT; ++it) {
                const int row = it * R::RPI + vr;
                const float pr = __shfl_sync(kFull, p, row * 2);
                uint4 raw = *reinterpret_cast<const uint4 *>(stp + R::V_OFF + row * R::ROW + vc * 16);
                if (edge && (jb0 + row < cu.start || jb0 + row >= cu.ctx)) raw = make_uint4(0u, 0u, 0u, 0u);
                float vf[R::EPC];
                Vec<T>::to_f32(raw, vf);
#pragma unroll
                for (int e = 0; e < R::EPC; ++e) acc[e] = fmaf(pr, vf[e], acc[e]);
            }
            __syncwarp();
            ++consumed;
        }

        // ---- unit finished: write out or merge partials ------------------------
        float l = l_run;                                // lanes 2k, 2k+1 hold key k's weights
        l += __shfl_xor_sync(kFull, l, 2);
        l += __shfl_xor_sync(kFull, l, 4);
        l += __shfl_xor_sync(kFull, l, 8);
        l += __shfl_xor_sync(kFull, l, 16);
#pragma unroll
        for (int x = R::NC; x < 32; x <<= 1)
#pragma unroll
            for (int e = 0; e < R::EPC; ++e) acc[e] += __shfl_xor_sync(kFull, acc[e], x);
        const size_t sh = (size_t)cu.gs * P.H + cu.h;
        if (cu.npart == 1) {
            const float inv = l > 0.f ? 1.f / l : 0.f;
            if (lane < R::NC) {
                float o[R::EPC];
#pragma unroll
                for (int e = 0; e < R::EPC; ++e) o[e] = acc[e] * inv;
                reinterpret_cast<uint4 *>(static_cast<unsigned char *>(CP.out) + sh * R::ROW)[lane] =
                    Vec<T>::from_f32(o);
            }
            continue;
        }
        const size_t slot = sh * CP.max_parts + cu.p;
        if (lane < R::NC) {
            float4 *dst = reinterpret_cast<float4 *>(CP.ws_acc + slot * D + lane * R::EPC);
#pragma unroll
            for (int e = 0; e < R::EPC; e += 4)
                __stcg(dst + e / 4, make_float4(acc[e], acc[e + 1], acc[e + 2], acc[e + 3]));
        }
        if (lane == 0) __stcg(CP.ws_ml + slot, make_float2(m_run, l));
        __syncwarp();
        unsigned old = 0;
        if (lane == 0) old = atom_inc_acq_rel(CP.counters + sh, (unsigned)(cu.npart - 1));
        old = __shfl_sync(kFull, old, 0);
        if (old != (unsigned)(cu.npart - 1)) continue;

        // last partition of (s, h): merge, write out, return the slots to zero.
        // Every load of a chunk of up to R::MCH partials is issued before any is
        // used (one L2 round trip per chunk); lane i holds partial i's (m, l).
        const size_t base = sh * CP.max_parts;
        float M = -INFINITY, L = 0.f;
        float o_acc[R::DPL];
#pragma unroll
        for (int e = 0; e < R::DPL; ++e) o_acc[e] = 0.f;
        for (int c0 = 0; c0 < cu.npart; c0 += R::MCH) {
            const int n = min(R::MCH, cu.npart - c0);
            float2 ml = make_float2(-INFINITY, 0.f);
            if (lane < n) ml = __ldcg(CP.ws_ml + base + c0 + lane);
            float a[R::MCH][R::DPL];
#pragma unroll
            for (int i = 0; i < R::MCH; ++i) {
                const float *src = CP.ws_acc + (base + c0 + i) * D + lane * R::DPL;
                if constexpr (R::DPL == 4) {
                    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (i < n) v = __ldcg(reinterpret_cast<const float4 *>(src));
                    a[i][0] = v.x; a[i][1] = v.y; a[i][2] = v.z; a[i][3] = v.w;
                } else {
                    float2 v = make_float2(0.f, 0.f);
                    if (i < n) v = __ldcg(reinterpret_cast<const float2 *>(src));
                    a[i][0] = v.x; a[i][1] = v.y;
                }
            }
            float mc = ml.x;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mc = fmaxf(mc, __shfl_xor_sync(kFull, mc, o));
            const float Mn = fmaxf(M, mc);
            const float corr = M == -INFINITY ? 0.f : ex2(M - Mn);
            const float w = (lane < n && Mn != -INFINITY) ? ex2(ml.x - Mn) : 0.f;
            float lc = ml.y * w;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) lc += __shfl_xor_sync(kFull, lc, o);
            L = L * corr + lc;
#pragma unroll
            for (int e = 0; e < R::DPL; ++e) o_acc[e] *= corr;
#pragma unroll
            for (int i = 0; i < R::MCH; ++i) {
                const float wi = __shfl_sync(kFull, w, i);
#pragma unroll
                for (int e = 0; e < R::DPL; ++e) o_acc[e] = fmaf(wi, a[i][e], o_acc[e]);
            }
            M = Mn;
#pragma unroll
            for (int i = 0; i < R::MCH; ++i) {
                if (i >= n) break;
                float *dst0 = CP.ws_acc + (base + c0 + i) * D + lane * R::DPL;
                if constexpr (R::DPL == 4) __stcg(reinterpret_cast<float4 *>(dst0), make_float4(0.f, 0.f, 0.f, 0.f));
                else __stcg(reinterpret_cast<float2 *>(dst0), make_float2(0.f, 0.f));
            }
            if (lane < n) __stcg(CP.ws_ml + base + c0 + lane, make_float2(0.f, 0.f));
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        T *dst = reinterpret_cast<T *>(static_cast<unsigned char *>(CP.out) + sh * R::ROW) + lane * R::DPL;
#pragma unroll
        for (int e = 0; e < R::DPL; ++e) {
            const float v = o_acc[e] * inv;
            if constexpr (sizeof(T) == 4) dst[e] = v;
            else if constexpr (std::is_same<T, __half>::value) dst[e] = __float2half_rn(v);
            else dst[e] = __float2bfloat16_rn(v);
        }
    }
}

// Small batches: one CTA per (sequence, head) of the launch.  The pair's
// visible blocks are dealt round-robin to the CTA's NW warps (warp w takes
// blocks b0 + w, b0 + w + NW, ...), each warp streams its blocks through its
// own NSTAGE-stage pipeline with the same per-block math as the persistent
// kernel, and the warps' partial softmax states are merged in shared memory:
// no prefix scan over the batch, no global split-K round trip, no workspace.
// Launched only when every pair fits one CTA's warps (at most 32 blocks per
// warp) and the launch has at most one pair per SM (see the launcher).
template <typename T, int D, int NSTAGE, int NW>
__global__ void __launch_bounds__(NW * 32) paged_decode_small_kernel(const Params P)
{
    using R = Tr<T, D>;
    using DT = Dot<T, D>;
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    unsigned char *stages = smem + (size_t)warp * NSTAGE * R::STAGE;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)NW * NSTAGE * R::STAGE) + warp * NSTAGE;
    float2 *mrg_ml = reinterpret_cast<float2 *>(smem + (size_t)NW * NSTAGE * R::STAGE + NW * NSTAGE * 8);
    float *mrg_acc = reinterpret_cast<float *>(mrg_ml + NW);          // [NW][D]
    float *table_sm = mrg_acc + NW * D;                               // this head's T5 table row
    griddep_launch_dependents();
    griddep_wait();

    // ---- the pair: launch sequence sl (problem 0's first), head h ----------------
    const int sl = (int)P.by_H.div((uint32_t)blockIdx.x);
    const int h = (int)blockIdx.x - sl * P.H;
    const int prob = prob_of(sl, P);
    const Prob &CP = P.pr[prob];
    const int gs = CP.seq_base + sl - (prob ? P.pr[0].num_seqs : 0);
    int ctx = __ldg(CP.context_lens + gs);
    if (ctx < 0 || ctx > CP.max_ctx || ctx > CP.mbps * BS) {
        if (threadIdx.x == 0) flag_status(P.status, PKA_DEVCHK_CONTEXT_LEN);
        ctx = ctx < 0 ? 0 : min(ctx, min(CP.max_ctx, CP.mbps * BS));
    }
    const size_t sh = (size_t)gs * P.H + h;
    if (ctx == 0) {                                   // no key: a zero output row
        if (threadIdx.x < R::NC)
            reinterpret_cast<uint4 *>(static_cast<unsigned char *>(CP.out) + sh * R::ROW)[threadIdx.x] =
                make_uint4(0u, 0u, 0u, 0u);
        return;
    }
    const int start = (CP.window > 0 && ctx > CP.window) ? ctx - CP.window : 0;
    const int b0 = start / BS, last = (ctx - 1) / BS, nb = last + 1 - b0;
    const bool has_bias = CP.bias != nullptr, has_table = CP.bias_table != nullptr;
    if (has_table)
        for (int i = threadIdx.x; i < CP.num_buckets; i += blockDim.x)
            table_sm[i] = __ldg(CP.bias_table + (size_t)h * CP.num_buckets + i);
    if (lane == 0)
        for (int i = 0; i < NSTAGE; ++i) mbar_init(smem_u32(&bars[i]), 32);
    fence_barrier_init();
    __syncthreads();

    // ---- this warp's blocks: b0 + warp + k NW, k < myn (myn <= 32) --------------
    const int myn = nb > warp ? (nb - warp + NW - 1) / NW : 0;
    int bt = 0;                                       // lane k: block-table entry of block k
    if (lane < myn) bt = __ldg(CP.block_tables + (size_t)gs * CP.mbps + b0 + warp + lane * NW);
    // append: the block holding position ctx - 1 (the sequence's last) is this
    // warp's when (last - b0) % NW == warp
    const bool append = CP.k_new != nullptr && (last - b0) % NW == warp;
    uint4 kn = make_uint4(0u, 0u, 0u, 0u), vn = kn;
    int app_phys = -1;
    if (append) {
        const size_t rowoff = sh * R::ROW;
        if (lane < R::NC) {
            kn = __ldg(reinterpret_cast<const uint4 *>(CP.k_new + rowoff) + lane);
            vn = __ldg(reinterpret_cast<const uint4 *>(CP.v_new + rowoff) + lane);
        }
        app_phys = __ldg(CP.block_tables + (size_t)gs * CP.mbps + last);
    }
    const uint32_t st_base = smem_u32(stages);
    uint32_t issued = 0;
    bool ok = true;
    auto issue = [&]() {
        const int k = (int)issued;
        const int stage = k % NSTAGE;
        const uint32_t st = st_base + stage * R::STAGE;
        const uint32_t bar = smem_u32(&bars[stage]);
        int phys = __shfl_sync(kFull, bt, k);
        if ((unsigned)phys >= (unsigned)CP.num_blocks) {
            if (lane == 0) flag_status(P.status, PKA_DEVCHK_BLOCK_ID);
            phys = 0;
        }
        if (lane == 0) {
            mbar_expect_tx(bar, 2 * R::CHUNK);
            const size_t off = ((size_t)phys * P.H + h) * (size_t)R::CHUNK;
            bulk_g2s(st + R::K_OFF, CP.k_cache + off, R::CHUNK, bar);
            bulk_g2s(st + R::V_OFF, CP.v_cache + off, R::CHUNK, bar);
        }
        if (has_bias && lane < BS) {
            const int j = (b0 + warp + k * NW) * BS + lane;
            const bool in = j >= start && j < ctx;
            const float *src = CP.bias + sh * CP.bias_stride + (in ? j : 0);
            cp_async_4(st + R::B_OFF + lane * 4, src, in ? 4u : 0u);
        }
        if (k == 0 && lane < R::NC) cp_async_16(st + R::Q_OFF + lane * 16, CP.q + sh * R::ROW + lane * 16);
        cp_async_arrive_noinc(bar);
        ++issued;
    };
    while ((int)issued < myn && issued < (uint32_t)NSTAGE) issue();

    const int key = lane >> 1, half = lane & 1;
    const int q_first = half * R::QCH;
    const int q_rot = (key & 3) + half * R::QSWZ;
    const int vr = lane / R::NC, vc = lane % R::NC;
    typename DT::Q qreg;
    float acc[R::EPC];
#pragma unroll
    for (int e = 0; e < R::EPC; ++e) acc[e] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;
    int consumed = 0;
    for (int k = 0; k < myn; ++k) {
        const int stage = k % NSTAGE;
        const unsigned char *stp = stages + stage * R::STAGE;
        if (!mbar_wait_bounded(smem_u32(&bars[stage]), (k / NSTAGE) & 1)) {
            if (lane == 0) flag_status(P.status, PKA_DEVCHK_TIMEOUT);
            ok = false;
            break;
        }
        consumed = k + 1;
        const int bi = b0 + warp + k * NW;
        if (append && bi == last) {
            const int r = (ctx - 1) % BS;
            if (lane < R::NC) {
                unsigned char *row = stages + stage * R::STAGE + r * R::ROW;
                reinterpret_cast<uint4 *>(row + R::K_OFF)[lane] = kn;
                reinterpret_cast<uint4 *>(row + R::V_OFF)[lane] = vn;
                if ((unsigned)app_phys < (unsigned)CP.num_blocks) {
                    const size_t off = (((size_t)app_phys * P.H + h) * BS + r) * R::ROW;
                    reinterpret_cast<uint4 *>(const_cast<unsigned char *>(CP.k_cache) + off)[lane] = kn;
                    reinterpret_cast<uint4 *>(const_cast<unsigned char *>(CP.v_cache) + off)[lane] = vn;
                } else if (lane == 0) {
                    flag_status(P.status, PKA_DEVCHK_BLOCK_ID);
                }
            }
            __syncwarp();
        }
        if (k == 0) DT::load_q(qreg, stp + R::Q_OFF, q_first, q_rot);
        float d = DT::dot(qreg, stp + R::K_OFF + key * R::ROW, q_first, q_rot);
        d += __shfl_xor_sync(kFull, d, 1);
        const int j = bi * BS + key;
        float bv = 0.f;
        if (has_bias) {
            bv = reinterpret_cast<const float *>(stp + R::B_OFF)[key];
        } else if (has_table) {
            const int dist = min(max(ctx - 1 - j, 0), CP.num_buckets - 1);
            bv = table_sm[dist];
        }
        const float x = (j >= start && j < ctx) ? (d + bv) * CP.scale_log2 : -INFINITY;
        float mb = fmaxf(x, __shfl_xor_sync(kFull, x, 2));
        mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, 4));
        mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, 8));
        mb = fmaxf(mb, __shfl_xor_sync(kFull, mb, 16));
        const float m_new = fmaxf(m_run, mb);
        const float corr = ex2(m_run - m_new);
        const float p = ex2(x - m_new);
        l_run = fmaf(l_run, corr, p);
        m_run = m_new;
#pragma unroll
        for (int e = 0; e < R::EPC; ++e) acc[e] *= corr;
        // rows outside [start, ctx) of an edge block: their V bits are not used
        const int jb0 = bi * BS;
        const bool edge = jb0 < start || jb0 + BS > ctx;
#pragma unroll
        for (int it = 0; it < R::PV_IT; ++it) {
            const int row = it * R::RPI + vr;
            const float pr = __shfl_sync(kFull, p, row * 2);
            uint4 raw = *reinterpret_cast<const uint4 *>(stp + R::V_OFF + row * R::ROW + vc * 16);
            if (edge && (jb0 + row < start || jb0 + row >= ctx)) raw = make_uint4(0u, 0u, 0u, 0u);
            float vf[R::EPC];
            Vec<T>::to_f32(raw, vf);
#pragma unroll
            for (int e = 0; e < R::EPC; ++e) acc[e] = fmaf(pr, vf[e], acc[e]);
        }
        __syncwarp();
        if (append && bi == last && lane < R::NC) fence_proxy_async();   // before a refill of this stage
        __syncwarp();
        if ((int)issued < myn) issue();
    }
    if (!ok) {
        // a copy never landed: give the later stages in flight a bounded wait of
        // their own before the CTA leaves (their shared memory must stay valid)
        for (int k = consumed + 1; k < (int)issued; ++k)
            if (!mbar_wait_bounded(smem_u32(&bars[k % NSTAGE]), (k / NSTAGE) & 1)) break;
    }
    // ---- the warp's partial state -> shared memory, merged by warp 0 --------------
    float l = l_run;
    l += __shfl_xor_sync(kFull, l, 2);
    l += __shfl_xor_sync(kFull, l, 4);
    l += __shfl_xor_sync(kFull, l, 8);
    l += __shfl_xor_sync(kFull, l, 16);
#pragma unroll
    for (int x = R::NC; x < 32; x <<= 1)
#pragma unroll
        for (int e = 0; e < R::EPC; ++e) acc[e] += __shfl_xor_sync(kFull, acc[e], x);
    if (!ok || myn == 0) { m_run = -INFINITY; l = 0.f; }
    if (lane < R::NC) {
#pragma unroll
        for (int e = 0; e < R::EPC; ++e) mrg_acc[warp * D + lane * R::EPC + e] = (ok && myn > 0) ? acc[e] : 0.f;
    }
    if (lane == 0) mrg_ml[warp] = make_float2(m_run, l);
    __syncthreads();
    if (warp != 0) return;
    const float2 ml = lane < NW ? mrg_ml[lane] : make_float2(-INFINITY, 0.f);
    float M = ml.x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
    const float wgt = (lane < NW && M != -INFINITY) ? ex2(ml.x - M) : 0.f;
    float L = ml.y * wgt;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(kFull, L, o);
    float o_acc[R::DPL];
#pragma unroll
    for (int e = 0; e < R::DPL; ++e) o_acc[e] = 0.f;
#pragma unroll
    for (int i = 0; i < NW; ++i) {
        const float wi = __shfl_sync(kFull, wgt, i);
#pragma unroll
        for (int e = 0; e < R::DPL; ++e) o_acc[e] = fmaf(wi, mrg_acc[i * D + lane * R::DPL + e], o_acc[e]);
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    T *dst = reinterpret_cast<T *>(static_cast<unsigned char *>(CP.out) + sh * R::ROW) + lane * R::DPL;
#pragma unroll
    for (int e = 0; e < R::DPL; ++e) {
        const float v = o_acc[e] * inv;
        if constexpr (sizeof(T) == 4) dst[e] = v;
        else if constexpr (std::is_same<T, __half>::value) dst[e] = __float2half_rn(v);
        else dst[e] = __float2bfloat16_rn(v);
    }
}

// ---- host side --------------------------------------------------------------------

// Kernels launched with programmatic stream serialization: a launch may begin
// while the previous kernel in the stream finishes (its CTAs take the SMs the
// previous grid's CTAs leave); the kernels wait (griddepcontrol.wait) before
// reading anything, so every input and workspace write of earlier kernels is
// complete and visible when read.
template <typename K>
cudaError_t launch_programmatic(K kern, unsigned grid, unsigned threads, size_t smem, cudaStream_t stream, const Params &P)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, P);
}

template <typename T, int D, int NSTAGE, int NW> struct Config {
    using R = Tr<T, D>;
    static size_t smem_bytes(int nseq)
    {
        return (size_t)NW * NSTAGE * R::STAGE + (size_t)NW * NSTAGE * 8 + (size_t)(2 * nseq + 1) * 4 +
               (size_t)MAX_TABLE_FLOATS * 4;
    }
    static cudaError_t launch(const Params &P, int sms, cudaStream_t stream)
    {
        auto kern = paged_decode_kernel<T, D, NSTAGE, NW>;
        const size_t smem = smem_bytes(P.num_seqs);
        const size_t smem_max = smem_bytes(MAX_SEQS_PER_LAUNCH);
        static std::once_flag once;
        static cudaError_t attr_err = cudaSuccess;
        static int occ = 1;
        std::call_once(once, [&] {
            attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_max);
            if (attr_err == cudaSuccess)
                attr_err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, NW * 32, smem_max);
            if (occ < 1) occ = 1;
        });
        if (attr_err != cudaSuccess) return attr_err;
        long long units_upper = 0;
        for (int i = 0; i < P.nprob; ++i) units_upper += (long long)P.pr[i].num_seqs * P.H * P.pr[i].max_parts;
        long long grid = std::min<long long>((long long)sms * occ, (units_upper + NW - 1) / NW);
        if (grid < 1) grid = 1;
        return launch_programmatic(kern, (unsigned)grid, NW * 32, smem, stream, P);
    }
};

// The small-batch kernel: NW warps per CTA, one CTA per (sequence, head).
constexpr int SMALL_NW = 4;
constexpr int SMALL_MAX_BLOCKS = 32 * SMALL_NW;   // visible blocks one CTA's warps cover (one table entry per lane)
constexpr int SMALL_SHORT_BLOCKS = 32;           // a pair this short stays cheap on one CTA of 4 warps

template <typename T, int D, int NSTAGE> struct SmallConfig {
    using R = Tr<T, D>;
    static size_t smem_bytes(int table_floats)
    {
        return (size_t)SMALL_NW * NSTAGE * R::STAGE + (size_t)SMALL_NW * NSTAGE * 8 + (size_t)SMALL_NW * 8 +
               (size_t)SMALL_NW * D * 4 + (size_t)table_floats * 4;
    }
    static cudaError_t prepare(int *ctas_per_sm)
    {
        auto kern = paged_decode_small_kernel<T, D, NSTAGE, SMALL_NW>;
        static std::once_flag once;
        static cudaError_t err = cudaSuccess;
        static int occ = 1;
        std::call_once(once, [&] {
            const size_t smax = smem_bytes(MAX_TABLE_FLOATS);
            err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smax);
            if (err == cudaSuccess)
                err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, SMALL_NW * 32, smem_bytes(0));
            if (occ < 1) occ = 1;
        });
        *ctas_per_sm = occ;
        return err;
    }
    static cudaError_t launch(const Params &P, int table_floats, cudaStream_t stream)
    {
        int occ = 1;
        const cudaError_t e = prepare(&occ);
        if (e != cudaSuccess) return e;
        return launch_programmatic(paged_decode_small_kernel<T, D, NSTAGE, SMALL_NW>, (unsigned)(P.num_seqs * P.H),
                                   SMALL_NW * 32, smem_bytes(table_floats), stream, P);
    }
};

template <typename T, int D> using SmallCfg = SmallConfig<T, D, (Tr<T, D>::STAGE <= 9000 ? 3 : 2)>;

template <typename T, int D>
cudaError_t small_slots(int sms, long long *slots)
{
    int occ = 1;
    const cudaError_t e = SmallCfg<T, D>::prepare(&occ);
    *slots = (long long)sms * occ;
    return e;
}

template <typename T, int D>
cudaError_t dispatch_cfg(const Params &P, int sms, cudaStream_t stream, bool small, int table_floats)
{
    if (small) return SmallCfg<T, D>::launch(P, table_floats, stream);
    // one CTA per SM, about 200 KB of stages: 16 warps x 3 stages for 4.3 KB
    // stages (2-byte D=64), 12 x 2 for 8.5 KB, 6 x 2 for 17 KB (f32 D=128)
    if constexpr (Tr<T, D>::STAGE <= 5000)
        return Config<T, D, 3, 16>::launch(P, sms, stream);
    else if constexpr (Tr<T, D>::STAGE <= 9000)
        return Config<T, D, 2, 12>::launch(P, sms, stream);
    else
        return Config<T, D, 2, 6>::launch(P, sms, stream);
}

}  // namespace

DecodePlan decode_plan(int max_context_len, int sliding_window, int block_size)
{
    long long maxvb = (max_context_len + block_size - 1) / block_size;
    if (sliding_window > 0) maxvb = std::min<long long>(maxvb, (sliding_window + block_size - 2) / block_size + 1);
    if (maxvb < 1) maxvb = 1;
    int pb = 4;
    while (pb < 32 && (maxvb + pb - 1) / pb > 16) pb *= 2;
    DecodePlan plan;
    plan.part_blocks = pb;
    plan.max_parts = (int)std::max<long long>(1, (maxvb + pb - 1) / pb);
    return plan;
}

static size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

size_t decode_workspace_bytes(int num_seqs, int num_heads, int head_dim, const DecodePlan &plan)
{
    const size_t sh = (size_t)num_seqs * num_heads;
    const size_t slots = sh * plan.max_parts;
    return 256 + round_up(sh * 4, 256) + round_up(slots * 8, 256) + round_up(slots * head_dim * 4, 256);
}

// Streaming warps per CTA of the configuration dispatch_cfg picks.
static int streaming_warps(pka_dtype dt, int head_dim)
{
    const int stage = dt == PKA_F32 ? (head_dim == 64 ? Tr<float, 64>::STAGE : Tr<float, 128>::STAGE)
                                    : (head_dim == 64 ? Tr<__half, 64>::STAGE : Tr<__half, 128>::STAGE);
    return stage <= 5000 ? 16 : stage <= 9000 ? 12 : 6;
}

static cudaError_t dispatch(const Params &P, pka_dtype dt, int head_dim, int sms, cudaStream_t stream, bool small,
                            int table_floats)
{
    if (head_dim == 64) {
        if (dt == PKA_F32) return dispatch_cfg<float, 64>(P, sms, stream, small, table_floats);
        if (dt == PKA_F16) return dispatch_cfg<__half, 64>(P, sms, stream, small, table_floats);
        return dispatch_cfg<__nv_bfloat16, 64>(P, sms, stream, small, table_floats);
    }
    if (dt == PKA_F32) return dispatch_cfg<float, 128>(P, sms, stream, small, table_floats);
    if (dt == PKA_F16) return dispatch_cfg<__half, 128>(P, sms, stream, small, table_floats);
    return dispatch_cfg<__nv_bfloat16, 128>(P, sms, stream, small, table_floats);
}

// CTAs of the small-batch kernel that fit the GPU at once.
static cudaError_t small_kernel_slots(pka_dtype dt, int head_dim, int sms, long long *slots)
{
    if (head_dim == 64) {
        if (dt == PKA_F32) return small_slots<float, 64>(sms, slots);
        if (dt == PKA_F16) return small_slots<__half, 64>(sms, slots);
        return small_slots<__nv_bfloat16, 64>(sms, slots);
    }
    if (dt == PKA_F32) return small_slots<float, 128>(sms, slots);
    if (dt == PKA_F16) return small_slots<__half, 128>(sms, slots);
    return small_slots<__nv_bfloat16, 128>(sms, slots);
}

cudaError_t launch_paged_decode_multi(const DecodeArgs *a, const DecodePlan *size_plans, int n, cudaStream_t stream)
{
    if (n < 1 || n > MAX_PROBLEMS) return cudaErrorInvalidValue;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int H = a[0].num_heads;
    // Fewer, larger partitions cost fewer split-K merges (each ends with a
    // release and an atomic), while enough units keep every warp busy: double
    // a problem's partition (the one with the most partitions first) while the
    // launch still yields at least 3 units per streaming warp of the GPU.  Each
    // workspace was sized for its size plan, the smallest partitions, so it
    // covers any larger ones.
    DecodePlan plan[MAX_PROBLEMS];
    long long maxvb[MAX_PROBLEMS], sh[MAX_PROBLEMS];
    for (int i = 0; i < n; ++i) {
        plan[i] = size_plans[i];
        long long vb = (a[i].max_context_len + BS - 1) / BS;
        if (a[i].window > 0) vb = std::min<long long>(vb, (a[i].window + BS - 2) / BS + 1);
        maxvb[i] = std::max<long long>(1, std::min((long long)plan[i].max_parts * plan[i].part_blocks, vb));
        sh[i] = (long long)a[i].num_seqs * H;
    }
    auto parts = [&](int i, int pb) { return (maxvb[i] + pb - 1) / pb; };
    // Batches of at most one (sequence, head) pair per SM, each pair's visible
    // blocks within one CTA's warps, go to the small-batch kernel: no prefix
    // scan and no global split-K merge (tiny f32 workload 6.7 -> 2.7 us a
    // launch).  So do batches of short contexts (at most SMALL_SHORT_BLOCKS
    // visible blocks a pair) whose pairs fit the GPU's resident small-kernel
    // CTAs at once, several to an SM (T5-small-shaped step 11.0 -> 10.9 us).
    // Other batches stay on the persistent kernel.
    bool small = false;
    {
        long long pairs = 0, vb_max = 0;
        for (int i = 0; i < n; ++i) {
            pairs += sh[i];
            vb_max = std::max(vb_max, maxvb[i]);
        }
        long long slots = 0;
        if (vb_max <= SMALL_MAX_BLOCKS && pairs <= MAX_SEQS_PER_LAUNCH * (long long)H) {
            const cudaError_t e = small_kernel_slots(a[0].dtype, a[0].head_dim, sms, &slots);
            if (e != cudaSuccess) return e;
            small = pairs <= std::min<long long>(slots, sms) || (vb_max <= SMALL_SHORT_BLOCKS && pairs <= slots);
        }
    }
    const long long target = 3ll * sms * streaming_warps(a[0].dtype, a[0].head_dim);
    int pb[MAX_PROBLEMS];
    for (int i = 0; i < n; ++i) pb[i] = plan[i].part_blocks;
    for (;;) {
        long long total = 0;
        for (int i = 0; i < n; ++i) total += sh[i] * parts(i, pb[i]);
        int pick = -1;
        for (int i = 0; i < n; ++i) {
            if (pb[i] >= 32 || sh[i] == 0) continue;
            if (total - sh[i] * (parts(i, pb[i]) - parts(i, 2 * pb[i])) < target) continue;
            if (pick < 0 || parts(i, pb[i]) > parts(pick, pb[pick])) pick = i;
        }
        if (pick < 0) break;
        pb[pick] *= 2;
    }
    Prob pr[MAX_PROBLEMS];
    unsigned *queue = nullptr;
    for (int i = 0; i < n; ++i) {
        if (pb[i] != plan[i].part_blocks) {
            plan[i].part_blocks = pb[i];
            plan[i].max_parts = (int)parts(i, pb[i]);
        }
        const size_t shi = (size_t)sh[i];
        const size_t slots = shi * plan[i].max_parts;
        unsigned char *ws = static_cast<unsigned char *>(a[i].workspace);
        Prob &R = pr[i];
        R.out = a[i].out;
        R.q = static_cast<const unsigned char *>(a[i].q);
        R.k_cache = static_cast<const unsigned char *>(a[i].k_cache);
        R.v_cache = static_cast<const unsigned char *>(a[i].v_cache);
        R.block_tables = a[i].block_tables;
        R.context_lens = a[i].context_lens;
        R.bias = a[i].bias;
        R.bias_table = a[i].bias_table;
        R.num_buckets = a[i].num_buckets;
        R.k_new = static_cast<const unsigned char *>(a[i].k_new);
        R.v_new = static_cast<const unsigned char *>(a[i].v_new);
        // [unit hand-out counter, 256 B | arrival counters | (m, l) | acc]
        R.counters = reinterpret_cast<unsigned *>(ws + 256);
        R.ws_ml = reinterpret_cast<float2 *>(ws + 256 + round_up(shi * 4, 256));
        R.ws_acc = reinterpret_cast<float *>(ws + 256 + round_up(shi * 4, 256) + round_up(slots * 8, 256));
        if (i == 0) queue = reinterpret_cast<unsigned *>(ws);
        R.scale_log2 = a[i].scale * 1.4426950408889634f;
        R.window = a[i].window;
        R.mbps = a[i].max_blocks_per_seq;
        R.num_blocks = a[i].num_blocks;
        R.max_ctx = a[i].max_context_len;
        R.part_blocks = plan[i].part_blocks;
        R.max_parts = plan[i].max_parts;
        R.by_part_blocks = make_fastdiv((uint32_t)plan[i].part_blocks);
        R.bias_stride = a[i].bias_row_stride;
        R.seq_base = 0;
        R.num_seqs = a[i].num_seqs;
    }
    // The sequences of all problems, problem 0's first, go out in launches of
    // at most MAX_SEQS_PER_LAUNCH; a launch may hold the tail of one problem
    // and the head of the next.
    long long total_seqs = 0, first[MAX_PROBLEMS];
    for (int i = 0; i < n; ++i) {
        first[i] = total_seqs;
        total_seqs += a[i].num_seqs;
    }
    for (long long base = 0; base < total_seqs; base += MAX_SEQS_PER_LAUNCH) {
        const long long end = std::min<long long>(total_seqs, base + MAX_SEQS_PER_LAUNCH);
        Params P;
        P.nprob = 0;
        P.num_seqs = 0;
        P.H = H;
        P.by_H = make_fastdiv((uint32_t)H);
        P.queue = queue;
        P.status = a[0].status;
        for (int i = 0; i < n; ++i) {
            const long long lo = std::max(base, first[i]), hi = std::min(end, first[i] + a[i].num_seqs);
            if (lo >= hi) continue;
            Prob R = pr[i];
            R.seq_base = (int)(lo - first[i]);
            R.num_seqs = (int)(hi - lo);
            P.pr[P.nprob++] = R;
            P.num_seqs += R.num_seqs;
        }
        if (P.nprob == 0) continue;
        if (P.nprob < MAX_PROBLEMS) P.pr[1] = P.pr[0];   // never read: keeps the struct defined
        int table_floats = 0;
        for (int i = 0; i < P.nprob; ++i)
            if (P.pr[i].bias_table) table_floats = std::max(table_floats, P.pr[i].num_buckets);
        const cudaError_t e = dispatch(P, a[0].dtype, a[0].head_dim, sms, stream, small, table_floats);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_paged_decode(const DecodeArgs &a, const DecodePlan &size_plan, cudaStream_t stream)
{
    return launch_paged_decode_multi(&a, &size_plan, 1, stream);
}

}  // namespace pka
