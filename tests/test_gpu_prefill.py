"""GPU parity of swa_prefill against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest

import oracle
import synth
from helpers import TOL, max_err, to_dev, to_f64, to_host_storage
from synth import BF16, F16

pytestmark = pytest.mark.gpu


def run_gpu_prefill(pka, case):
    import torch
    if case.device_qkv is not None:
        q, k, v = case.device_qkv
    else:
        q, k, v = (to_dev(a, case.dtype) for a in (case.q, case.k, case.v))
    out = torch.empty_like(q)
    cu = torch.from_numpy(case.cu_seqlens).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pka.swa_prefill(out, q, k, v, cu, case.max_seqlen, case.window, case.causal, case.scale, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return out


def _check(got, ref, what, dtype=BF16):
    assert np.isfinite(got).all(), what
    err = max_err(got, ref)
    assert err <= TOL[dtype], f"{what}: max abs err {err:.3g}"


@pytest.mark.parametrize("window", [-1, 1, 2, 63, 64, 65, 128, 300])
@pytest.mark.parametrize("causal", [0, 1])
def test_prefill_small_parity(cuda_lib, window, causal):
    lens = [1, 2, 127, 128, 129, 255, 300, 513]
    case = synth.make_prefill_case("small", 200 + max(window, 0) + causal, lens, 3, 64, window, causal, BF16,
                                   scale=1 / 8)
    got = to_f64(run_gpu_prefill(cuda_lib, case), BF16)
    ref = oracle.prefill(case.q, case.k, case.v, case.cu_seqlens, window, causal, case.scale, BF16)
    _check(got, ref, f"W={window} causal={causal}")


def _sample_rows(case, rng, per_seq=48):
    rows = []
    cu = case.cu_seqlens
    for b in range(case.num_seqs):
        a, e = int(cu[b]), int(cu[b + 1])
        L = e - a
        pick = {0, L - 1, min(L - 1, 127), min(L - 1, 128)}
        pick |= set(rng.choice(L, size=min(L, per_seq), replace=False).tolist())
        rows += [a + p for p in sorted(pick)]
    return np.array(rows, dtype=np.int64)


def test_prefill_encoder_workload_sampled(cuda_lib):
    """The encoder workload (32 sequences, lengths U[128, 8192], 12 heads,
    head_dim 64) at full size, full-attention layer 0: the oracle checks every
    sequence's first/last rows, the rows at the 128-row tile edge and a
    seeded random sample."""
    case = synth.prefill_workload(0, device="cuda")
    got = run_gpu_prefill(cuda_lib, case)
    q, k, v = (to_host_storage(t, BF16) for t in case.device_qkv)
    rows = _sample_rows(case, np.random.default_rng(400), per_seq=48)
    ref = oracle.prefill(q, k, v, case.cu_seqlens, case.window, case.causal, case.scale, BF16, rows=rows)
    _check(to_f64(got[rows], BF16), ref, "encoder layer 0")


@pytest.mark.parametrize("layer", [1, 2])
def test_prefill_encoder_window_layers_every_row(cuda_lib, layer):
    """The encoder workload's two window-64 layers at full size, every row
    (each row keeps at most 127 keys, so the oracle covers all of them)."""
    case = synth.prefill_workload(layer, device="cuda")
    got = run_gpu_prefill(cuda_lib, case)
    q, k, v = (to_host_storage(t, BF16) for t in case.device_qkv)
    ref = oracle.prefill(q, k, v, case.cu_seqlens, case.window, case.causal, case.scale, BF16)
    _check(to_f64(got, BF16), ref, f"encoder layer {layer}")


def test_prefill_captured_and_eager_launches(cuda_lib):
    """Launches captured into CUDA graphs keep item counters no other launch
    is given: replays of two captured graphs on one stream, while more eager
    launches than the eager counter ring holds run on another, all give the
    eager result bit for bit.  A graph holding more captured launches than
    there are reserved counter pairs ends with launches that deal their items
    statically; those give the same bits too."""
    import torch
    lens = [300] * 40                                  # 2 items per (sequence, head): more items than CTAs
    case = synth.make_prefill_case("capture", 610, lens, 4, 64, 64, 0, BF16, scale=1 / 8)
    q, k, v = (to_dev(a, BF16) for a in (case.q, case.k, case.v))
    cu = torch.from_numpy(case.cu_seqlens).cuda()
    ref = torch.empty_like(q)
    cuda_lib.swa_prefill(ref, q, k, v, cu, case.max_seqlen, case.window, case.causal, case.scale)
    torch.cuda.synchronize()

    def capture(out, n):
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                for _ in range(n):
                    cuda_lib.swa_prefill(out, q, k, v, cu, case.max_seqlen, case.window, case.causal, case.scale)
        torch.cuda.current_stream().wait_stream(s)
        return g

    outs = [torch.zeros_like(q) for _ in range(3)]
    g1, g2 = capture(outs[0], 1), capture(outs[1], 1)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(1100):
            cuda_lib.swa_prefill(outs[2], q, k, v, cu, case.max_seqlen, case.window, case.causal, case.scale)
    for _ in range(20):
        g1.replay()
        g2.replay()
    torch.cuda.synchronize()
    for o in outs:
        assert torch.equal(o.view(torch.int16), ref.view(torch.int16))
    big = torch.zeros_like(q)
    g3 = capture(big, 8192 + 8)                        # at least the last 8 launches find no reserved pair
    g3.replay()
    torch.cuda.synchronize()
    assert torch.equal(big.view(torch.int16), ref.view(torch.int16))


# ---------------------------------------------------------------------------
# chunked local attention
# ---------------------------------------------------------------------------
def run_gpu_chunked(pka, case):
    import torch
    if case.device_qkv is not None:
        q, k, v = case.device_qkv
    else:
        q, k, v = (to_dev(a, case.dtype) for a in (case.q, case.k, case.v))
    out = torch.empty_like(q)
    cu = torch.from_numpy(case.cu_seqlens).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pka.chunked_prefill(out, q, k, v, cu, case.max_seqlen, case.chunk, case.causal, case.scale, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return out


@pytest.mark.parametrize("chunk", [1, 16, 100, 128, 129, 300, 1000])
@pytest.mark.parametrize("causal", [0, 1])
def test_chunked_prefill_small_parity(cuda_lib, chunk, causal):
    lens = [1, 2, 127, 128, 129, 255, 300, 513]
    case = synth.make_prefill_case("chunk", 300 + chunk + causal, lens, 3, 64, -1, causal, BF16, scale=1 / 8)
    case.chunk = chunk
    got = to_f64(run_gpu_chunked(cuda_lib, case), BF16)
    ref = oracle.prefill_chunked(case.q, case.k, case.v, case.cu_seqlens, chunk, causal, case.scale, BF16)
    _check(got, ref, f"chunk={chunk} causal={causal}")


def test_chunked_prefill_workload_sampled(cuda_lib):
    """32 packed sequences U[128,8192], chunks of 1024, causal, full size;
    sampled rows incl. every sequence's first/last and chunk-edge rows."""
    case = synth.chunked_prefill_workload(device="cuda")
    got = run_gpu_chunked(cuda_lib, case)
    q, k, v = (to_host_storage(t, BF16) for t in case.device_qkv)
    rng = np.random.default_rng(444)
    rows = []
    for b in range(case.num_seqs):
        a, e = int(case.cu_seqlens[b]), int(case.cu_seqlens[b + 1])
        pick = {a, e - 1} | {a + p for p in (1023, 1024, 2047, 2048) if a + p < e}
        pick |= set((a + rng.choice(e - a, size=min(e - a, 24), replace=False)).tolist())
        rows += sorted(pick)
    rows = np.array(rows, dtype=np.int64)
    ref = oracle.prefill_chunked(q, k, v, case.cu_seqlens, case.chunk, case.causal, case.scale, BF16, rows=rows)
    _check(to_f64(got[rows], BF16), ref, "chunked workload")


# ---------------------------------------------------------------------------
# relative-position bias in the scores
# ---------------------------------------------------------------------------
def run_gpu_biased(pka, case):
    import torch
    if case.device_qkv is not None:
        q, k, v = case.device_qkv
    else:
        q, k, v = (to_dev(a, case.dtype) for a in (case.q, case.k, case.v))
    out = torch.empty_like(q)
    cu = torch.from_numpy(case.cu_seqlens).cuda()
    rel = torch.from_numpy(case.rel_bias).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pka.prefill_biased(out, q, k, v, cu, case.max_seqlen, rel, case.window, case.causal, case.scale, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return out


@pytest.mark.parametrize("window", [-1, 1, 64, 300])
@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("buckets", [1, 5, 129])
def test_biased_prefill_small_parity(cuda_lib, window, causal, buckets):
    lens = [1, 2, 127, 128, 129, 255, 300, 513]
    case = synth.make_prefill_case("biased", 300 + max(window, 0) + causal + buckets, lens, 3, 64, window, causal,
                                   BF16, scale=1 / 8)
    case.rel_bias = synth.rel_bias_table(buckets, 3, buckets) * np.float32(2.0)
    got = to_f64(run_gpu_biased(cuda_lib, case), BF16)
    ref = oracle.prefill_biased(case.q, case.k, case.v, case.cu_seqlens, window, causal, case.scale, BF16,
                                case.rel_bias)
    _check(got, ref, f"biased W={window} causal={causal} B={buckets}")


@pytest.mark.parametrize("causal", [0, 1])
def test_biased_prefill_table_larger_than_shared_memory(cuda_lib, causal):
    """A relative-position table too wide for the kernel's shared-memory copy
    (4 heads x 1100 buckets) is read from global memory through the clamp;
    sequences longer than the cap reach the saturated columns on both sides."""
    lens = [1, 300, 1300, 2600]
    case = synth.make_prefill_case("biased-wide", 330 + causal, lens, 4, 64, -1, causal, BF16, scale=1 / 8)
    case.rel_bias = synth.rel_bias_table(1100, 4, 1100) * np.float32(2.0)
    got = to_f64(run_gpu_biased(cuda_lib, case), BF16)
    ref = oracle.prefill_biased(case.q, case.k, case.v, case.cu_seqlens, -1, causal, case.scale, BF16,
                                case.rel_bias)
    _check(got, ref, f"biased wide table causal={causal}")


def test_biased_prefill_t5_encoder_workload_sampled(cuda_lib):
    """The T5-large-shaped encoder (256 x 512 tokens, 16 heads, bias table
    [16, 257]) at full size, checked on sampled rows."""
    case = synth.t5_encoder_prefill_workload(device="cuda")
    got = run_gpu_biased(cuda_lib, case)
    q, k, v = (to_host_storage(t, BF16) for t in case.device_qkv)
    rows = _sample_rows(case, np.random.default_rng(410), per_seq=8)
    ref = oracle.prefill_biased(q, k, v, case.cu_seqlens, -1, 0, case.scale, BF16, case.rel_bias, rows=rows)
    _check(to_f64(got[rows], BF16), ref, "t5 encoder")


# ---------------------------------------------------------------------------
# prefill against the paged cache
# ---------------------------------------------------------------------------
class GpuPagedPrefill:
    """A PagedPrefillCase resident on the GPU: caches filled by the library's
    reshape_and_cache, queries packed."""

    def __init__(self, pc, pka):
        import torch
        from helpers import GpuDecode
        self.pc = pc
        self.pka = pka
        self.cache = GpuDecode(pc.cache, pka)
        self.q = pc.device_q if pc.device_q is not None else to_dev(pc.q, pc.dtype)
        self.cu = torch.from_numpy(pc.cu_seqlens_q).cuda()
        self.rel = torch.from_numpy(pc.rel_bias).cuda() if pc.rel_bias is not None else None
        self.out = torch.empty_like(self.q)
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def run(self):
        import torch
        g, pc = self.cache, self.pc
        self.pka.paged_prefill(self.out, self.q, g.k_cache, g.v_cache, g.block_tables, self.cu, g.context_lens,
                               pc.max_query_len, pc.window, pc.causal, self.rel, pc.scale, status=self.status)
        torch.cuda.synchronize()
        return self.out

    def host_caches(self):
        return to_host_storage(self.cache.k_cache, self.pc.dtype), to_host_storage(self.cache.v_cache, self.pc.dtype)


def oracle_paged(gp, rows=None, q=None):
    pc = gp.pc
    kc, vc = gp.host_caches()
    return oracle.paged_prefill(pc.q if q is None else q, kc, vc, pc.cache.block_tables, pc.cu_seqlens_q,
                                pc.cache.context_lens, pc.window, pc.causal, pc.scale, 16, pc.dtype,
                                rel_bias=pc.rel_bias, rows=rows)


PAGED_CTX = (1, 15, 16, 17, 130, 300, 520, 700, 2000)
PAGED_QL = (1, 15, 5, 17, 130, 256, 257, 40, 600)


@pytest.mark.parametrize("window", [-1, 1, 40, 300])
@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("buckets", [0, 129])
def test_paged_prefill_small_parity(cuda_lib, window, causal, buckets):
    pc = synth.make_paged_prefill_case("paged", 500 + max(window, 0) + causal + buckets, BF16, PAGED_CTX, PAGED_QL,
                                       3, 64, window, causal, buckets, scale=1 / 8, pool_blocks=400)
    gp = GpuPagedPrefill(pc, cuda_lib)
    got = to_f64(gp.run(), BF16)
    _check(got, oracle_paged(gp), f"paged W={window} causal={causal} B={buckets}")
    assert int(gp.status.item()) == 0


@pytest.mark.parametrize("window", [-1, 3])
def test_paged_prefill_rows_without_keys_are_zero(cuda_lib, window):
    """Non-causal: more query rows than keys, and a sequence with no keys."""
    pc = synth.make_paged_prefill_case("paged-edge", 520 + window, BF16, (5, 0, 30, 200), (9, 3, 4, 300), 2, 64,
                                       window, 0, 4, scale=1 / 8)
    gp = GpuPagedPrefill(pc, cuda_lib)
    gp.out.fill_(7.0)
    got = to_f64(gp.run(), BF16)
    ref = oracle_paged(gp)
    _check(got, ref, f"paged edge W={window}")
    assert np.all(got[9:12] == 0.0)


def test_paged_prefill_ignores_cache_tails_and_evicted_blocks(cuda_lib):
    """Cache rows past each context hold NaN, and the block-table entries of
    blocks before every row's window hold an id past the pool (evicted): the
    result is unchanged and no status bit is set, so neither was used."""
    import torch
    W = 50
    pc = synth.make_paged_prefill_case("paged-evict", 530, BF16, (700, 333, 129), (100, 20, 129), 2, 64, W, 1, 129,
                                       scale=1 / 8, pool_blocks=120)
    gp = GpuPagedPrefill(pc, cuda_lib)
    ref = to_f64(gp.run(), BF16).copy()
    bt = pc.cache.block_tables.copy()
    kc, vc = gp.cache.k_cache, gp.cache.v_cache
    for s in range(pc.num_seqs):
        ctx, Lq = int(pc.cache.context_lens[s]), int(pc.query_lens[s])
        last = (ctx - 1) // 16
        blk = int(bt[s, last])
        kc[blk, :, ctx % 16 or 16:] = float("nan")
        vc[blk, :, ctx % 16 or 16:] = float("nan")
        first_kept = max(0, ctx - Lq - W + 1)             # the earliest key any row keeps
        bt[s, :first_kept // 16] = 1 << 30
    gp.cache.block_tables.copy_(torch.from_numpy(bt))
    got = to_f64(gp.run(), BF16)
    assert np.isfinite(got).all()
    assert int(gp.status.item()) == 0
    assert max_err(got, ref) == 0.0


def test_paged_prefill_t5_workload_sampled(cuda_lib):
    """A prompt chunk of each sequence of the T5-large-shaped decode workload:
    causal with the T5 bias over the self-attention cache, and unmasked over
    the encoder cache, checked on sampled rows."""
    import torch
    self_c, cross_c = synth.t5_paged_prefill_workload(device="cuda")
    rng = np.random.default_rng(540)
    for pc in (self_c, cross_c):
        gp = GpuPagedPrefill(pc, cuda_lib)
        got = gp.run()
        assert int(gp.status.item()) == 0
        cu = pc.cu_seqlens_q
        rows = []
        for b in range(pc.num_seqs):
            a, e = int(cu[b]), int(cu[b + 1])
            pick = {a, e - 1} | set((a + rng.choice(e - a, size=min(e - a, 6), replace=False)).tolist())
            rows += sorted(pick)
        rows = np.array(rows, dtype=np.int64)
        ref = oracle_paged(gp, rows=rows, q=to_host_storage(gp.q, BF16))
        _check(to_f64(got[rows], BF16), ref, pc.name)
        del gp
        torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# f16 operands (same kernel, f16 MMA and f16 P)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("window", [-1, 1, 64, 300])
@pytest.mark.parametrize("causal", [0, 1])
def test_prefill_f16_small_parity(cuda_lib, window, causal):
    lens = [1, 2, 127, 128, 129, 255, 300, 513]
    case = synth.make_prefill_case("small-f16", 600 + max(window, 0) + causal, lens, 3, 64, window, causal, F16,
                                   scale=1 / 8)
    got = to_f64(run_gpu_prefill(cuda_lib, case), F16)
    ref = oracle.prefill(case.q, case.k, case.v, case.cu_seqlens, window, causal, case.scale, F16)
    _check(got, ref, f"f16 W={window} causal={causal}", F16)


def test_prefill_f16_biased_and_paged_parity(cuda_lib):
    case = synth.make_prefill_case("biased-f16", 610, [1, 130, 300, 513], 2, 64, 40, 0, F16, scale=1 / 8)
    case.rel_bias = synth.rel_bias_table(610, 2, 129)
    got = to_f64(run_gpu_biased(cuda_lib, case), F16)
    ref = oracle.prefill_biased(case.q, case.k, case.v, case.cu_seqlens, 40, 0, case.scale, F16, case.rel_bias)
    _check(got, ref, "f16 biased", F16)
    pc = synth.make_paged_prefill_case("paged-f16", 611, F16, PAGED_CTX, PAGED_QL, 2, 64, -1, 1, 129, scale=1 / 8,
                                       pool_blocks=400)
    gp = GpuPagedPrefill(pc, cuda_lib)
    _check(to_f64(gp.run(), F16), oracle_paged(gp), "f16 paged", F16)
    assert int(gp.status.item()) == 0


def test_prefill_f16_large_logits_stay_finite(cuda_lib):
    """Scores far beyond the f16 range (|q.k| up to ~1e5 before the scale): P
    and the accumulator are f32 and P <= 256, so the f16 outputs stay finite
    (the encoder-decoder page's T5 fp16 overflow report)."""
    case = synth.make_prefill_case("f16-big", 612, [200, 77], 2, 64, -1, 0, F16, scale=1.0)
    case.q = synth.encode(synth.decode_to_f32(case.q, F16) * np.float32(40.0), F16)
    case.k = synth.encode(synth.decode_to_f32(case.k, F16) * np.float32(40.0), F16)
    got = to_f64(run_gpu_prefill(cuda_lib, case), F16)
    ref = oracle.prefill(case.q, case.k, case.v, case.cu_seqlens, -1, 0, 1.0, F16)
    _check(got, ref, "f16 large logits", F16)


def test_prefill_item_counters_are_clean_after_every_launch(cuda_lib):
    """Packed-key launches with more items than CTAs hand items out from one
    of 1024 counter pairs that the library owns, taken in turn by every
    prefill launch; each launch must leave its pair at zero.  A paged launch
    with more items than CTAs, 1023 tiny launches, then a packed launch on
    the paged launch's pair: it still matches the oracle."""
    import torch
    ctx = np.array([16 + 29 * i for i in range(60)])
    ql = np.minimum(ctx, 5 + 3 * np.arange(60))
    pc = synth.make_paged_prefill_case("paged-cycle", 530, BF16, ctx, ql, 3, 64, -1, 1, 0, scale=1 / 8)
    gp = GpuPagedPrefill(pc, cuda_lib)
    case = synth.make_prefill_case("cycle", 531, [256] * 40 + [300, 17], 4, 64, -1, 0, BF16, scale=1 / 8)
    ref = oracle.prefill(case.q, case.k, case.v, case.cu_seqlens, -1, 0, case.scale, BF16)
    tiny = synth.make_prefill_case("tiny", 532, [16], 1, 64, -1, 0, BF16, scale=1 / 8)
    tq, tk, tv = (to_dev(a, BF16) for a in (tiny.q, tiny.k, tiny.v))
    tout = torch.empty_like(tq)
    tcu = torch.from_numpy(tiny.cu_seqlens).cuda()
    for _ in range(2):
        gp.run()                                        # 60 sequences x 3 heads: 180 items
        for _ in range(1023):
            cuda_lib.swa_prefill(tout, tq, tk, tv, tcu, 16, -1, 0, 1 / 8)
        got = to_f64(run_gpu_prefill(cuda_lib, case), BF16)   # 172 items, the paged launch's pair
        _check(got, ref, "packed launch after a full cycle of counter pairs")
    assert int(gp.status.item()) == 0


def test_prefill_more_sequences_than_one_launch(cuda_lib):
    """1300 short sequences: the host splits each call into launches of at
    most 1024 sequences (the kernel's schedule holds 1024).  Every row of the
    full-attention, window-64 (the chunk-classifying instance), biased and
    paged calls against the oracle, across the split."""
    rng = np.random.default_rng(77)
    lens = rng.integers(1, 48, size=1300).tolist()
    for window in (-1, 64):
        case = synth.make_prefill_case("many", 700 + max(window, 0), lens, 2, 64, window, 0, BF16, scale=1 / 8)
        got = to_f64(run_gpu_prefill(cuda_lib, case), BF16)
        ref = oracle.prefill(case.q, case.k, case.v, case.cu_seqlens, window, 0, case.scale, BF16)
        _check(got, ref, f"1300 sequences W={window}")
    case = synth.make_prefill_case("many-biased", 702, lens, 2, 64, -1, 1, BF16, scale=1 / 8)
    case.rel_bias = synth.rel_bias_table(33, 2, 33) * np.float32(2.0)
    got = to_f64(run_gpu_biased(cuda_lib, case), BF16)
    ref = oracle.prefill_biased(case.q, case.k, case.v, case.cu_seqlens, -1, 1, case.scale, BF16, case.rel_bias)
    _check(got, ref, "1300 sequences biased")
    ctx = rng.integers(1, 70, size=1300)
    ql = np.minimum(ctx, rng.integers(1, 40, size=1300))
    pc = synth.make_paged_prefill_case("many-paged", 703, BF16, ctx.tolist(), ql.tolist(), 2, 64, -1, 1, 17,
                                       scale=1 / 8, pool_blocks=int(((ctx + 15) // 16).sum()) + 64)
    gp = GpuPagedPrefill(pc, cuda_lib)
    got = to_f64(gp.run(), BF16)
    _check(got, oracle_paged(gp), "1300 sequences paged")
    assert int(gp.status.item()) == 0


# ---------------------------------------------------------------------------
# head dim 128 (packed keys, no bias): one query tile per work item
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("window", [-1, 1, 63, 64, 65, 128, 300])
@pytest.mark.parametrize("causal", [0, 1])
def test_prefill_head_dim_128_parity(cuda_lib, window, causal):
    lens = [1, 2, 127, 128, 129, 255, 300, 513]
    case = synth.make_prefill_case("d128", 800 + max(window, 0) + causal, lens, 3, 128, window, causal, BF16,
                                   scale=128 ** -0.5)
    got = to_f64(run_gpu_prefill(cuda_lib, case), BF16)
    ref = oracle.prefill(case.q, case.k, case.v, case.cu_seqlens, window, causal, case.scale, BF16)
    _check(got, ref, f"D=128 W={window} causal={causal}")


@pytest.mark.parametrize("chunk", [1, 100, 128, 256])
def test_chunked_prefill_head_dim_128_parity(cuda_lib, chunk):
    lens = [1, 2, 127, 128, 129, 255, 300, 513]
    case = synth.make_prefill_case("d128-chunk", 820 + chunk, lens, 3, 128, -1, 1, BF16, scale=128 ** -0.5)
    case.chunk = chunk
    got = to_f64(run_gpu_chunked(cuda_lib, case), BF16)
    ref = oracle.prefill_chunked(case.q, case.k, case.v, case.cu_seqlens, chunk, 1, case.scale, BF16)
    _check(got, ref, f"D=128 chunk={chunk}")


def test_prefill_head_dim_128_f16_and_long_sequences(cuda_lib):
    """f16 at head dim 128 on ragged lengths up to 1300 (up to 11 key tiles per
    query tile: the running max is raised and O rescaled in TMEM), full and
    window 64; every row against the oracle."""
    lens = [1, 700, 1300]
    for window in (-1, 64):
        case = synth.make_prefill_case("d128-f16", 840 + max(window, 0), lens, 2, 128, window, 0, F16,
                                       scale=128 ** -0.5)
        got = to_f64(run_gpu_prefill(cuda_lib, case), F16)
        ref = oracle.prefill(case.q, case.k, case.v, case.cu_seqlens, window, 0, case.scale, F16)
        _check(got, ref, f"f16 D=128 W={window}", F16)
