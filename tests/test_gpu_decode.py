"""GPU parity of reshape_and_cache and paged_attn_decode against the fp64
oracle, through the C ABI, on seeded synthetic inputs."""
import math

import numpy as np
import pytest

import oracle
import synth
from helpers import TOL, GpuDecode, max_err, oracle_decode, oracle_decode_t5, to_dev, to_f64, to_host_storage, torch_dtype
from synth import BF16, F16, F32

pytestmark = pytest.mark.gpu


def _check(got, ref, dtype, what=""):
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = max_err(got, ref)
    assert err <= TOL[dtype], f"{what}: max abs err {err:.3g} > {TOL[dtype]}"
    return err


# ---------------------------------------------------------------------------
# reshape_and_cache: bit-exact against the oracle's scatter
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", [F32, F16, BF16])
@pytest.mark.parametrize("D", [64, 128])
def test_reshape_and_cache_bitexact(cuda_lib, dtype, D):
    import torch
    case = synth.make_decode_case("rc", 21, dtype, 7, 3, D, context_lens=np.array([1, 15, 16, 17, 40, 0, 33]),
                                  pool_blocks=20)
    slots = case.slot_mapping.copy()
    slots[[0, 5, 17]] = -1
    H, bs = 3, 16
    shape = (case.num_blocks, H, bs, D)
    pat = np.full(int(np.prod(shape)) * case.key.itemsize, 0x5A, np.uint8)
    host_k = pat.view(case.key.dtype).reshape(shape).copy()
    host_v = host_k.copy()
    oracle.reshape_and_cache(host_k, host_v, case.key, case.value, slots, bs)
    kc = to_dev(pat.view(case.key.dtype).reshape(shape), dtype)
    vc = kc.clone()
    cuda_lib.reshape_and_cache(to_dev(case.key, dtype), to_dev(case.value, dtype), kc, vc,
                               torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    assert to_host_storage(kc, dtype).tobytes() == host_k.tobytes()
    assert to_host_storage(vc, dtype).tobytes() == host_v.tobytes()


def test_reshape_and_cache_slot_past_cache_flags_status(cuda_lib):
    import torch
    case = synth.make_decode_case("rc", 22, BF16, 2, 2, 64, context_lens=np.array([5, 9]))
    slots = case.slot_mapping.copy()
    slots[3] = case.num_blocks * 16 + 5           # past the cache: skipped and flagged
    kc = torch.zeros((case.num_blocks, 2, 16, 64), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    cuda_lib.reshape_and_cache(to_dev(case.key, BF16), to_dev(case.value, BF16), kc, vc,
                               torch.from_numpy(slots).cuda(), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & cuda_lib.DEVCHK_SLOT


# ---------------------------------------------------------------------------
# the named decode workloads
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("n", [1, 2, 3])
@pytest.mark.parametrize("bias", [True, False])
def test_decode_workload_parity(cuda_lib, n, bias):
    case = synth.decode_workload(n)
    g = GpuDecode(case, cuda_lib)
    got = to_f64(g.run(bias=bias), case.dtype)
    ref = oracle_decode(case, bias=bias)
    _check(got, ref, case.dtype, f"workload {n} bias={bias}")
    assert int(g.status.item()) == 0


def test_short_context_batch_above_the_small_kernel_slots(cuda_lib):
    """T5-small-shaped contexts (at most 32 cache blocks a pair) run on the
    one-CTA-per-pair kernel while the batch's pairs fit its resident CTAs; 160
    sequences x 8 heads (1280 pairs) exceed them and take the persistent
    kernel with its split-K merge.  Both against the oracle, bias on."""
    case = synth.decode_workload(2, num_seqs=160)
    g = GpuDecode(case, cuda_lib)
    got = to_f64(g.run(bias=True), case.dtype)
    ref = oracle_decode(case, bias=True)
    _check(got, ref, case.dtype, "short contexts, 1280 pairs")
    assert int(g.status.item()) == 0


def test_cross_attention_decode_parity(cuda_lib):
    """Cross-attention decode: its own block table and pool, encoder length
    512, no bias, no window."""
    case = synth.cross_workload()
    g = GpuDecode(case, cuda_lib)
    _check(to_f64(g.run(), case.dtype), oracle_decode(case), case.dtype, "cross")


def test_long_context_window_decode_full_size_sampled(cuda_lib):
    """fp16 / head_dim 128 / window 4096 / NaN-padded bias, at full size
    (512 x 16, contexts log-uniform [16, 8192]); the oracle checks a seeded
    sample of (sequence, head) pairs that includes the longest and shortest
    sequences."""
    import torch
    case = synth.decode_workload(5, device="cuda")
    g = GpuDecode(case, cuda_lib)
    got = to_f64(g.run(), case.dtype)
    assert np.isfinite(got).all()
    assert int(g.status.item()) == 0
    order = np.argsort(case.context_lens)
    rng = np.random.default_rng(55)
    seqs = sorted(set(order[:3].tolist() + order[-5:].tolist() + rng.choice(512, 16, replace=False).tolist()))
    # a compact host case with just those sequences, from the generator's token rows
    sub = _subcase(case, seqs)
    pairs = np.array([[i, h] for i in range(len(seqs)) for h in range(case.num_heads)], dtype=np.int32)
    ref = oracle_decode(sub, pairs=pairs).reshape(len(seqs), case.num_heads, case.head_dim)
    _check(got[seqs], ref, case.dtype, "long-context sample")


def _subcase(case, seqs):
    """Host copy of a few sequences of a device-drawn case, laid out in a
    fresh contiguous pool."""
    key, value = case.device_kv
    ctx = case.context_lens[seqs]
    ks, vs = [], []
    for s in seqs:
        a, b = int(case.tok_offsets[s]), int(case.tok_offsets[s + 1])
        ks.append(to_host_storage(key[a:b], case.dtype))
        vs.append(to_host_storage(value[a:b], case.dtype))
    pool, bt, slot, tok = synth._paged_layout(np.random.default_rng(0), ctx, case.block_size)
    bias = case.bias[seqs] if case.bias is not None else None
    return synth.DecodeCase("sub", case.dtype, len(seqs), case.num_heads, case.head_dim, case.block_size, pool,
                            ctx.astype(np.int32), bt, slot, tok, case.q[seqs], np.concatenate(ks),
                            np.concatenate(vs), bias, case.window, case.scale)


# ---------------------------------------------------------------------------
# edge cases: every dtype and head size, ragged contexts, windows
# ---------------------------------------------------------------------------
EDGE_CTX = (0, 1, 2, 15, 16, 17, 31, 32, 33, 64, 65, 300, 1000)


@pytest.mark.parametrize("dtype", [F32, F16, BF16])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("window", [-1, 1, 7, 16, 17, 100, 5000])
def test_decode_edge_cases(cuda_lib, dtype, D, window):
    case = synth.make_decode_case("edge", 31 + D + window, dtype, len(EDGE_CTX), 3, D,
                                  context_lens=np.array(EDGE_CTX), pool_blocks=120, bias="gauss",
                                  bias_stride=1003, window=window, scale=0.17)
    g = GpuDecode(case, cuda_lib)
    for bias in (True, False):
        got = to_f64(g.run(bias=bias), dtype)
        _check(got, oracle_decode(case, bias=bias), dtype, f"edge bias={bias}")
        np.testing.assert_array_equal(got[0], 0.0)               # ctx 0 -> zero row
    assert int(g.status.item()) == 0


def test_decode_many_sequences_multi_launch(cuda_lib):
    """More sequences than one launch takes (the host splits them)."""
    rng = np.random.default_rng(77)
    ctx = rng.integers(0, 90, size=2600)
    case = synth.make_decode_case("many", 77, BF16, 2600, 2, 64, context_lens=ctx, bias="gauss", bias_stride=90)
    g = GpuDecode(case, cuda_lib)
    _check(to_f64(g.run(), BF16), oracle_decode(case), BF16, "many")


def test_decode_long_unwindowed_many_partitions(cuda_lib):
    """Contexts long enough for the most partitions per (sequence, head)."""
    ctx = np.array([8192, 8191, 7000, 4097, 33])
    case = synth.make_decode_case("long", 78, F16, 5, 2, 128, context_lens=ctx, bias="gauss", bias_stride=8200)
    g = GpuDecode(case, cuda_lib)
    _check(to_f64(g.run(), F16), oracle_decode(case), F16, "long")


@pytest.mark.parametrize("H", [5, 12, 33])
def test_decode_head_counts_not_powers_of_two(cuda_lib, H):
    """Units of a sequence run partition-major (unit - first = p * H + h) and the
    kernel splits them with a precomputed divisor for H: head counts that are
    not powers of two, against contexts from empty to many partitions, and
    more sequences than one CTA's warps so every split lands on every warp."""
    rng = np.random.default_rng(4000 + H)
    ctx = np.concatenate([[0, 1, 16, 17, 2047, 2048], rng.integers(0, 2100, size=40)])
    case = synth.make_decode_case("heads", 4000 + H, BF16, len(ctx), H, 64, context_lens=ctx, bias="gauss",
                                  bias_stride=2100, window=-1 if H != 12 else 1500)
    g = GpuDecode(case, cuda_lib)
    got = to_f64(g.run(), BF16)
    _check(got, oracle_decode(case), BF16, f"H={H}")
    np.testing.assert_array_equal(got[0], 0.0)
    assert int(g.status.item()) == 0


# ---------------------------------------------------------------------------
# poison, invariants, status
# ---------------------------------------------------------------------------
def test_decode_ignores_padding_and_evicted_blocks(cuda_lib):
    """NaN bias outside [start, ctx), block-table entries before the window
    set to -1 (evicted) and junk past the context leave the output as is."""
    import torch
    ctx = np.array([5, 40, 100, 257, 16])
    case = synth.make_decode_case("poison", 90, BF16, 5, 4, 64, context_lens=ctx, bias="gauss", bias_stride=260,
                                  window=20, max_blocks_per_seq=20)
    g = GpuDecode(case, cuda_lib)
    base = to_f64(g.run(), BF16).copy()
    bias = case.bias.copy()
    bt = case.block_tables.copy()
    for s, c in enumerate(ctx):
        start = max(0, c - 20)
        bias[s, :, c:] = np.nan
        bias[s, :, :start] = np.nan
        bt[s, :start // 16] = -1
        bt[s, (c + 15) // 16:] = 1 << 30
    g.bias.copy_(torch.from_numpy(bias))
    g.block_tables.copy_(torch.from_numpy(bt))
    got = to_f64(g.run(), BF16)
    np.testing.assert_array_equal(got, base)
    assert int(g.status.item()) == 0


def _poison_rows_outside_window(case, kc, vc):
    """Fill every cache row of a sequence's visible blocks that lies outside
    [start, ctx) -- the tail of the last block past the context, the head of
    the first visible block before the window -- with NaN, +Inf and -Inf in
    turn.  Each block belongs to one sequence, so no other key is touched."""
    import torch
    bs = case.block_size
    vals = (float("nan"), float("inf"), float("-inf"))
    n = 0
    for s, c in enumerate(case.context_lens.tolist()):
        if c == 0:
            continue
        start = max(0, c - case.window) if case.window > 0 else 0
        rows = [j for j in range(start // bs * bs, start)] + [j for j in range(c, (c - 1) // bs * bs + bs)]
        for j in rows:
            b = int(case.block_tables[s, j // bs])
            kc[b, :, j % bs] = vals[n % 3]
            vc[b, :, j % bs] = vals[(n + 1) % 3]
            n += 1
    torch.cuda.synchronize()
    return n


@pytest.mark.parametrize("dtype", [F32, F16, BF16])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("window", [-1, 20])
def test_decode_stale_cache_rows_contribute_nothing(cuda_lib, dtype, D, window):
    """A serving engine's newest block is only partly written, and a window's
    first block holds keys the window drops: cache rows outside [start, ctx)
    may hold any bits.  With those rows NaN / +Inf / -Inf the output is
    bit-identical to the clean cache's, and matches the oracle (which never
    reads them)."""
    case = synth.make_decode_case("stale", 300 + D + window, dtype, len(EDGE_CTX), 3, D,
                                  context_lens=np.array(EDGE_CTX), pool_blocks=120, bias="gauss",
                                  bias_stride=1003, window=window, scale=0.17)
    g = GpuDecode(case, cuda_lib)
    clean = to_host_storage(g.run(), dtype).copy()
    assert _poison_rows_outside_window(case, g.k_cache, g.v_cache) > 0
    got = g.run()
    assert to_host_storage(got, dtype).tobytes() == clean.tobytes()
    _check(to_f64(got, dtype), oracle_decode(case), dtype, "stale rows")
    assert int(g.status.item()) == 0


@pytest.mark.parametrize("dtype,D", [(BF16, 64), (F16, 128), (F32, 64)])
def test_decode_stale_rows_with_fused_append(cuda_lib, dtype, D):
    """The fused append writes the newest row into a block whose later rows
    hold NaN / Inf: outputs and cache bytes equal scatter + decode on the
    clean cache, bit for bit."""
    import torch
    case = synth.make_decode_case("stale-app", 320 + D, dtype, len(EDGE_CTX), 3, D,
                                  context_lens=np.array(EDGE_CTX), pool_blocks=160, window=40, bias="gauss",
                                  scale=0.2)
    g = GpuDecode(case, cuda_lib)
    ref_out = g.run().clone()
    kc, vc, k_new, v_new = _append_state(case, cuda_lib)
    _poison_rows_outside_window(case, kc, vc)
    kref, vref = g.k_cache.clone(), g.v_cache.clone()
    _poison_rows_outside_window(case, kref, vref)
    out = torch.empty_like(ref_out)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    cuda_lib.paged_attn_decode_multi([dict(g.problem("bias"), out=out, k_cache=kc, v_cache=vc, key_new=k_new,
                                           value_new=v_new)], status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(out.view(torch.uint8), ref_out.view(torch.uint8))
    assert torch.equal(kc.view(torch.uint8), kref.view(torch.uint8))
    assert torch.equal(vc.view(torch.uint8), vref.view(torch.uint8))


def test_decode_block_permutation_is_bitwise_invariant(cuda_lib):
    import torch
    case = synth.decode_workload(2)
    g = GpuDecode(case, cuda_lib)
    base = to_host_storage(g.run(), BF16).copy()
    perm = torch.from_numpy(np.random.default_rng(3).permutation(case.num_blocks)).cuda()
    kc2 = torch.empty_like(g.k_cache); vc2 = torch.empty_like(g.v_cache)
    kc2[perm] = g.k_cache; vc2[perm] = g.v_cache
    bt = g.block_tables.long()
    g.block_tables = torch.where(bt >= 0, perm[bt.clamp(min=0)], bt).int().contiguous()
    g.k_cache, g.v_cache = kc2, vc2
    assert to_host_storage(g.run(), BF16).tobytes() == base.tobytes()


def test_decode_repeat_calls_are_deterministic_and_leave_counters_clean(cuda_lib):
    import torch
    case = synth.decode_workload(3)
    g = GpuDecode(case, cuda_lib)
    need = cuda_lib.paged_attn_decode_workspace_size(case.num_seqs, case.num_heads, case.head_dim,
                                                     case.max_context_len, case.window)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    a = to_host_storage(g.run(workspace=ws), BF16).copy()
    b = to_host_storage(g.run(workspace=ws), BF16).copy()
    assert a.tobytes() == b.tobytes()
    assert int(ws.count_nonzero().item()) == 0          # the whole workspace is zero again


def test_decode_workspace_shared_across_shapes(cuda_lib):
    """One workspace, calls of different (num_seqs, num_heads, partitions) in
    turn: every call must leave it clean for the next."""
    import torch
    cases = [synth.decode_workload(2), synth.decode_workload(3), synth.decode_workload(1),
             synth.make_decode_case("wide", 94, F16, 1500, 4, 128, ctx_range=(1, 300))]
    ws = torch.zeros(64 << 20, dtype=torch.uint8, device="cuda")
    gs = [GpuDecode(c, cuda_lib) for c in cases]
    for rep in range(2):
        for c, g in zip(cases, gs):
            got = to_f64(g.run(workspace=ws), c.dtype)
            _check(got, oracle_decode(c), c.dtype, f"shared workspace {c.name} rep {rep}")
            assert int(ws.count_nonzero().item()) == 0


def test_decode_bad_block_id_sets_status(cuda_lib):
    """A block id past the pool inside the visible range: the kernel reads a
    valid block instead, finishes, and reports PKA_DEVCHK_BLOCK_ID."""
    import torch
    case = synth.make_decode_case("bad", 91, F32, 3, 2, 64, context_lens=np.array([20, 40, 3]))
    g = GpuDecode(case, cuda_lib)
    bt = case.block_tables.copy()
    bt[1, 1] = case.num_blocks + 7
    g.block_tables.copy_(torch.from_numpy(bt))
    g.run()
    torch.cuda.synchronize()
    assert int(g.status.item()) & cuda_lib.DEVCHK_BLOCK_ID


def test_decode_context_len_over_bound_sets_status(cuda_lib):
    import torch
    case = synth.make_decode_case("ctx", 92, F32, 3, 2, 64, context_lens=np.array([20, 40, 3]))
    g = GpuDecode(case, cuda_lib)
    g.context_lens[1] = 41                     # > max_context_len passed (40)
    g.run()
    torch.cuda.synchronize()
    assert int(g.status.item()) & cuda_lib.DEVCHK_CONTEXT_LEN


def test_f16_large_logits_stay_finite(cuda_lib):
    """q.k far beyond the f16 range (the T5-large f16 overflow report): f32
    scores keep the output finite and correct."""
    case = synth.make_decode_case("big", 93, F16, 4, 2, 128, context_lens=np.array([3, 50, 200, 17]),
                                  scale=1.0)
    big_q = (synth.decode_to_f32(case.q, F16) * 40).astype(np.float16)
    big_k = (synth.decode_to_f32(case.key, F16) * 40).astype(np.float16)
    case.q, case.key = big_q, big_k
    g = GpuDecode(case, cuda_lib)
    got = to_f64(g.run(), F16)
    _check(got, oracle_decode(case), F16, "f16 large logits")


def test_api_rejects_bad_arguments(cuda_lib):
    import torch
    case = synth.decode_workload(1)
    g = GpuDecode(case, cuda_lib)
    with pytest.raises(cuda_lib.PkaError):
        g.run(window=0)
    with pytest.raises(cuda_lib.PkaError):
        cuda_lib.paged_attn_decode(g.out, g.q, g.k_cache, g.v_cache, g.block_tables, g.context_lens, g.bias,
                                   max_context_len=65)          # bias stride 64 < 65
    small = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(cuda_lib.PkaError):
        g.run(workspace=small)


# ---------------------------------------------------------------------------
# T5 bias computed in the kernel from its table
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("n", [2, 3])
def test_t5_table_decode_parity(cuda_lib, n):
    """The T5-shaped workloads with the bias read from the [H, 129] table
    inside the kernel: matches the oracle, and the materialised-bias kernel."""
    case = synth.decode_workload(n)
    g = GpuDecode(case, cuda_lib)
    got = to_f64(g.run_t5(), case.dtype).copy()
    _check(got, oracle_decode_t5(case), case.dtype, f"t5 table workload {n}")
    mat = to_f64(g.run(), case.dtype)
    assert max_err(got, mat) <= TOL[case.dtype]
    assert int(g.status.item()) == 0


@pytest.mark.parametrize("window", [-1, 5, 40])
@pytest.mark.parametrize("buckets", [1, 17, 129])
def test_t5_table_decode_edges(cuda_lib, window, buckets):
    case = synth.make_decode_case("t5edge", 60 + buckets, F16, len(EDGE_CTX), 4, 128,
                                  context_lens=np.array(EDGE_CTX), pool_blocks=120, window=window, scale=0.2)
    case.bias_table = np.random.default_rng(buckets).standard_normal((4, buckets)).astype(np.float32)
    g = GpuDecode(case, cuda_lib)
    _check(to_f64(g.run_t5(), F16), oracle_decode_t5(case), F16, "t5 edges")


def test_t5_table_too_large_is_unsupported(cuda_lib):
    import torch
    case = synth.decode_workload(1)
    g = GpuDecode(case, cuda_lib)
    case.bias_table = np.zeros((2, 4000), dtype=np.float32)       # 8000 floats > the shared-memory cache
    with pytest.raises(cuda_lib.PkaError):
        g.run_t5()


# ---------------------------------------------------------------------------
# self- and cross-attention decode in one launch
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("self_mode", ["bias", "t5"])
def test_multi_self_and_cross_parity(cuda_lib, self_mode):
    """The T5-large-shaped step: decoder self-attention (T5 bias, materialised
    or from the table) and encoder cross-attention (its own block table and
    pool, encoder length 512, no bias) in one launch; each matches the oracle
    and the single-problem call."""
    sc, cc = synth.decode_workload(3), synth.cross_workload()
    gs, gc = GpuDecode(sc, cuda_lib), GpuDecode(cc, cuda_lib)
    cuda_lib.paged_attn_decode_multi([gs.problem(self_mode), gc.problem("none")], status=gs.status)
    got_s, got_c = to_f64(gs.out, sc.dtype).copy(), to_f64(gc.out, cc.dtype).copy()
    ref_s = oracle_decode_t5(sc) if self_mode == "t5" else oracle_decode(sc)
    _check(got_s, ref_s, sc.dtype, "multi self")
    _check(got_c, oracle_decode(cc), cc.dtype, "multi cross")
    assert int(gs.status.item()) == 0
    one_s = to_f64(gs.run_t5() if self_mode == "t5" else gs.run(), sc.dtype)
    assert max_err(got_s, one_s) <= TOL[sc.dtype]


@pytest.mark.parametrize("dtype,D", [(F32, 128), (F16, 64)])
def test_multi_spans_launch_boundary(cuda_lib, dtype, D):
    """1300 sequences over two problems take two launches, the first holding
    all of problem 0 and the head of problem 1; the problems differ in window,
    bias, scale, pool and block-table width."""
    a = synth.make_decode_case("multi-a", 71, dtype, 700, 2, D, ctx_range=(0, 70), bias="gauss", bias_stride=80,
                               window=23, scale=0.3)
    b = synth.make_decode_case("multi-b", 72, dtype, 600, 2, D, ctx_range=(1, 200), pool_blocks=5000,
                               max_blocks_per_seq=16, scale=0.05)
    ga, gb = GpuDecode(a, cuda_lib), GpuDecode(b, cuda_lib)
    cuda_lib.paged_attn_decode_multi([ga.problem("bias"), gb.problem("none")], status=ga.status)
    _check(to_f64(ga.out, dtype), oracle_decode(a), dtype, "problem 0")
    _check(to_f64(gb.out, dtype), oracle_decode(b), dtype, "problem 1")
    assert int(ga.status.item()) == 0


def test_multi_empty_problem_and_both_tables(cuda_lib):
    """A problem with no sequences is skipped; two problems may share one T5
    table, cached once."""
    import torch
    a = synth.decode_workload(2)
    b = synth.make_decode_case("multi-c", 73, BF16, 17, 8, 64, ctx_range=(1, 300))
    b.bias_table = a.bias_table
    ga, gb = GpuDecode(a, cuda_lib), GpuDecode(b, cuda_lib)
    pa, pb = ga.problem("t5"), gb.problem("t5")
    pb["bias_table"] = pa["bias_table"]
    cuda_lib.paged_attn_decode_multi([pa, pb], status=ga.status)
    _check(to_f64(ga.out, BF16), oracle_decode_t5(a), BF16, "table problem 0")
    _check(to_f64(gb.out, BF16), oracle_decode_t5(b), BF16, "table problem 1")
    empty = dict(gb.problem("none"), out=gb.out[:0], q=gb.q[:0], block_tables=gb.block_tables[:0],
                 context_lens=gb.context_lens[:0])
    ga.out.zero_()
    cuda_lib.paged_attn_decode_multi([empty, ga.problem("bias")], status=ga.status)
    _check(to_f64(ga.out, BF16), oracle_decode(a), BF16, "after empty problem")
    assert int(ga.status.item()) == 0


def test_multi_rejects_bad_problem_sets(cuda_lib):
    import torch
    a, b = synth.decode_workload(2), synth.make_decode_case("multi-d", 74, BF16, 5, 8, 64)
    ga, gb = GpuDecode(a, cuda_lib), GpuDecode(b, cuda_lib)
    with pytest.raises(cuda_lib.PkaError, match="UNSUPPORTED"):          # three problems
        cuda_lib.paged_attn_decode_multi([ga.problem("none"), gb.problem("none"), gb.problem("none")])
    with pytest.raises(cuda_lib.PkaError, match="INVALID_ARG"):          # overlapping outputs
        cuda_lib.paged_attn_decode_multi([ga.problem("none"), dict(gb.problem("none"), out=ga.out[:5])])
    ws = torch.zeros(1 << 22, dtype=torch.uint8, device="cuda")
    with pytest.raises(cuda_lib.PkaError, match="WORKSPACE"):            # one workspace for both
        cuda_lib.paged_attn_decode_multi([ga.problem("none", workspace=ws), gb.problem("none", workspace=ws)])
    pa, pb = ga.problem("t5"), gb.problem("none")
    pb["bias_table"] = pa["bias_table"].clone()
    with pytest.raises(cuda_lib.PkaError, match="UNSUPPORTED"):          # two different tables
        cuda_lib.paged_attn_decode_multi([pa, pb])
    with pytest.raises(ValueError):                                       # different head counts
        c = synth.make_decode_case("multi-e", 75, BF16, 3, 4, 64)
        cuda_lib.paged_attn_decode_multi([ga.problem("none"), GpuDecode(c, cuda_lib).problem("none")])


# ---------------------------------------------------------------------------
# fused append: the newest token's K/V written and attended in one launch
# ---------------------------------------------------------------------------
def _append_state(case, pka):
    """Caches holding every token but each sequence's newest (those rows NaN),
    and the newest rows as key_new / value_new [S, H, D]."""
    import torch
    H, D, bs = case.num_heads, case.head_dim, case.block_size
    tdt = torch_dtype(case.dtype)
    key, value = to_dev(case.key, case.dtype), to_dev(case.value, case.dtype)
    kc = torch.zeros((case.num_blocks, H, bs, D), dtype=tdt, device="cuda")
    vc = torch.zeros_like(kc)
    slots = case.slot_mapping.copy()
    newest = np.where(case.context_lens > 0, case.tok_offsets[1:] - 1, -1)
    have = newest >= 0
    slots[newest[have]] = -1
    pka.reshape_and_cache(key, value, kc, vc, torch.from_numpy(slots).cuda())
    ns = torch.from_numpy(case.slot_mapping[newest[have]]).cuda()
    kc[ns // bs, :, ns % bs] = float("nan")
    vc[ns // bs, :, ns % bs] = float("nan")
    idx = torch.from_numpy(np.where(have, newest, 0).astype(np.int64)).cuda()
    k_new, v_new = key[idx].contiguous(), value[idx].contiguous()
    return kc, vc, k_new, v_new


@pytest.mark.parametrize("dtype,D,window", [(BF16, 64, -1), (BF16, 64, 40), (F32, 128, 5), (F16, 128, -1)])
def test_multi_append_equals_scatter_then_decode(cuda_lib, dtype, D, window):
    """Outputs and cache bytes of the fused append are bit-identical to
    reshape_and_cache followed by the decode, from caches whose newest rows
    held NaN; and the decode matches the oracle."""
    import torch
    case = synth.make_decode_case("append", 90 + D + max(window, 0), dtype, len(EDGE_CTX), 3, D,
                                  context_lens=np.array(EDGE_CTX), pool_blocks=160, window=window, bias="gauss",
                                  scale=0.2)
    g = GpuDecode(case, cuda_lib)                       # every token scattered by reshape_and_cache
    ref_out = g.run().clone()
    kc, vc, k_new, v_new = _append_state(case, cuda_lib)
    out = torch.empty_like(ref_out)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pr = dict(g.problem("bias"), out=out, k_cache=kc, v_cache=vc, key_new=k_new, value_new=v_new)
    cuda_lib.paged_attn_decode_multi([pr], status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(out.view(torch.uint8), ref_out.view(torch.uint8))
    assert torch.equal(kc.view(torch.uint8), g.k_cache.view(torch.uint8))
    assert torch.equal(vc.view(torch.uint8), g.v_cache.view(torch.uint8))
    _check(to_f64(out, dtype), oracle_decode(case), dtype, "append")


@pytest.mark.parametrize("self_mode", ["bias", "t5"])
def test_multi_append_self_with_unappended_cross(cuda_lib, self_mode):
    """The T5-large-shaped step in one launch: the self-attention problem
    (materialised or in-kernel T5 bias) appends its newest token, the
    cross-attention problem does not."""
    import torch
    sc, cc = synth.decode_workload(3, num_seqs=48), synth.cross_workload(num_seqs=48)
    gs, gc = GpuDecode(sc, cuda_lib), GpuDecode(cc, cuda_lib)
    cuda_lib.paged_attn_decode_multi([gs.problem(self_mode), gc.problem("none")])   # same plan, scattered caches
    ref_s, ref_c = gs.out.clone(), gc.out.clone()
    kc, vc, k_new, v_new = _append_state(sc, cuda_lib)
    out_s, out_c = torch.empty_like(ref_s), torch.empty_like(ref_c)
    cuda_lib.paged_attn_decode_multi([dict(gs.problem(self_mode), out=out_s, k_cache=kc, v_cache=vc,
                                           key_new=k_new, value_new=v_new), dict(gc.problem("none"), out=out_c)])
    torch.cuda.synchronize()
    assert torch.equal(out_s.view(torch.int16), ref_s.view(torch.int16))
    assert torch.equal(out_c.view(torch.int16), ref_c.view(torch.int16))
    assert torch.equal(kc.view(torch.int16), gs.k_cache.view(torch.int16))
    ref = oracle_decode_t5(sc) if self_mode == "t5" else oracle_decode(sc)
    _check(to_f64(out_s, BF16), ref, BF16, "append self")


def test_multi_append_across_the_launch_split(cuda_lib):
    """1300 appending sequences over two problems take two launches; every
    sequence's newest row is written and attended exactly once."""
    import torch
    a = synth.make_decode_case("app-a", 95, F16, 700, 2, 64, ctx_range=(0, 70), bias="gauss", bias_stride=80,
                               window=23, scale=0.3)
    b = synth.make_decode_case("app-b", 96, F16, 600, 2, 64, ctx_range=(1, 200), pool_blocks=5000,
                               max_blocks_per_seq=16, scale=0.05)
    ga, gb = GpuDecode(a, cuda_lib), GpuDecode(b, cuda_lib)
    cuda_lib.paged_attn_decode_multi([ga.problem("bias"), gb.problem("none")])
    ref_a, ref_b = ga.out.clone(), gb.out.clone()
    ka, va, kna, vna = _append_state(a, cuda_lib)
    kb, vb, knb, vnb = _append_state(b, cuda_lib)
    oa, ob = torch.empty_like(ref_a), torch.empty_like(ref_b)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    cuda_lib.paged_attn_decode_multi([dict(ga.problem("bias"), out=oa, k_cache=ka, v_cache=va, key_new=kna,
                                           value_new=vna),
                                      dict(gb.problem("none"), out=ob, k_cache=kb, v_cache=vb, key_new=knb,
                                           value_new=vnb)], status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(oa.view(torch.int16), ref_a.view(torch.int16))
    assert torch.equal(ob.view(torch.int16), ref_b.view(torch.int16))
    assert torch.equal(ka.view(torch.int16), ga.k_cache.view(torch.int16))
    assert torch.equal(vb.view(torch.int16), gb.v_cache.view(torch.int16))


def test_multi_materialised_bias_then_table(cuda_lib):
    """Problem 0 with a materialised bias, problem 1 with the T5 table: the
    launch caches the second problem's table."""
    a = synth.decode_workload(2)
    b = synth.make_decode_case("tab1", 97, BF16, 20, 8, 64, ctx_range=(1, 400))
    b.bias_table = np.random.default_rng(97).standard_normal((8, 33)).astype(np.float32)
    ga, gb = GpuDecode(a, cuda_lib), GpuDecode(b, cuda_lib)
    cuda_lib.paged_attn_decode_multi([ga.problem("bias"), gb.problem("t5")])
    _check(to_f64(ga.out, BF16), oracle_decode(a), BF16, "materialised problem 0")
    _check(to_f64(gb.out, BF16), oracle_decode_t5(b), BF16, "table problem 1")


# ---------------------------------------------------------------------------
# the small-batch kernel (at most one (sequence, head) pair per SM) and the
# persistent kernel take the same problems
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype,D", [(BF16, 64), (F16, 128), (F32, 64), (F32, 128)])
@pytest.mark.parametrize("num_seqs", [9, 400])
def test_decode_small_and_large_batches_two_problems(cuda_lib, dtype, D, num_seqs):
    """A decode step of two problems -- self-attention with a materialised
    bias, a window and the fused append; cross-attention with the T5 table --
    at 9 sequences (the small-batch kernel: 72 pairs) and at 400 (the
    persistent kernel), each against the oracle; contexts reach 2047 keys."""
    import torch
    rng = np.random.default_rng(700 + D + num_seqs)
    ctx_a = rng.integers(0, 2048, size=num_seqs)
    ctx_a[:3] = [0, 1, 2047]
    a = synth.make_decode_case("two-a", 701 + D, dtype, num_seqs, 4, D, context_lens=ctx_a, bias="gauss",
                               bias_stride=2048, window=300, scale=0.15)
    b = synth.make_decode_case("two-b", 702 + D, dtype, num_seqs, 4, D, ctx_range=(1, 700), scale=0.1)
    b.bias_table = np.random.default_rng(703).standard_normal((4, 40)).astype(np.float32)
    ga, gb = GpuDecode(a, cuda_lib), GpuDecode(b, cuda_lib)
    kc, vc, k_new, v_new = _append_state(a, cuda_lib)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    cuda_lib.paged_attn_decode_multi([dict(ga.problem("bias"), k_cache=kc, v_cache=vc, key_new=k_new,
                                           value_new=v_new), gb.problem("t5")], status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _check(to_f64(ga.out, dtype), oracle_decode(a), dtype, f"self {num_seqs}")
    _check(to_f64(gb.out, dtype), oracle_decode_t5(b), dtype, f"cross {num_seqs}")
    assert torch.equal(kc.view(torch.uint8), ga.k_cache.view(torch.uint8))
