"""Pins for the fp64 oracle, independent of the oracle itself (no GPU).

Each check ties the oracle to something it does not contain: brute-force
attention on contiguous (unpaged) numpy arrays, closed forms that follow from
the formula softmax((QK^T + A)/sqrt(d_k)) V ("PagedAttention: Support custom
attention bias for T5 model (1/2)", opening section), invariants of that
formula, the two-table encoder-decoder layout ("Add Encoder-decoder model
support and T5 Model support") and the sliding-window masks ("[V1] Add
sliding window support to Flex Attention backend").
"""
import math
import os

import numpy as np
import pytest

import oracle
import synth
from synth import BF16, F16, F32

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------------------
# helpers that do NOT go through the oracle
# ---------------------------------------------------------------------------
def fill_cache_numpy(case):
    """Scatter the token rows into a [num_blocks, H, bs, D] cache with numpy
    fancy indexing (independent of the oracle's scatter)."""
    H, D, bs = case.num_heads, case.head_dim, case.block_size
    shape = (case.num_blocks, H, bs, D)
    dt = case.key.dtype
    kc = np.zeros(shape, dtype=dt)
    vc = np.zeros(shape, dtype=dt)
    slots = case.slot_mapping
    kc[slots // bs, :, slots % bs, :] = case.key
    vc[slots // bs, :, slots % bs, :] = case.value
    return kc, vc


def brute_decode(case):
    """Contiguous attention per (s, h): the sequence's own token rows, masked
    to the last W keys, softmax in float64 with numpy."""
    S, H, D = case.q.shape
    q = synth.decode_to_f32(case.q, case.dtype).astype(np.float64)
    K = synth.decode_to_f32(case.key, case.dtype).astype(np.float64)
    V = synth.decode_to_f32(case.value, case.dtype).astype(np.float64)
    out = np.zeros((S, H, D))
    for s in range(S):
        c = int(case.context_lens[s])
        lo = max(0, c - case.window) if case.window > 0 else 0
        if c == 0:
            continue
        t0 = int(case.tok_offsets[s])
        Ks = K[t0 + lo:t0 + c]          # [n, H, D]
        Vs = V[t0 + lo:t0 + c]
        logits = np.einsum("hd,nhd->hn", q[s], Ks)
        if case.bias is not None:
            logits = logits + case.bias[s, :, lo:c].astype(np.float64)
        logits = logits * case.scale
        w = np.exp(logits - logits.max(axis=1, keepdims=True))
        w /= w.sum(axis=1, keepdims=True)
        out[s] = np.einsum("hn,nhd->hd", w, Vs)
    return out


def run_oracle_decode(case, **kw):
    kc, vc = fill_cache_numpy(case)
    return oracle.paged_decode(case.q, kc, vc, case.block_tables, case.context_lens, case.bias,
                               case.window, case.scale, case.block_size, case.dtype, **kw)


def small_case(dtype=F32, ctx=(1, 15, 16, 17, 33), H=2, D=64, bias="gauss", window=-1, seed=7,
               scale=None, pool_extra=5):
    ctx = np.array(ctx, dtype=np.int32)
    pool = int(((ctx + 15) // 16).sum()) + pool_extra
    return synth.make_decode_case("pin", seed, dtype, len(ctx), H, D, context_lens=ctx, pool_blocks=pool,
                                  bias=bias, bias_stride=int(ctx.max()) + 3, window=window, scale=scale)


# ---------------------------------------------------------------------------
# widening of the storage encodings
# ---------------------------------------------------------------------------
def test_widen_f16_matches_numpy():
    bits = np.array([0x0000, 0x8000, 0x0001, 0x03ff, 0x0400, 0x3c00, 0xbc00, 0x7bff, 0x7c00, 0xfc00,
                     0x3555, 0x1234, 0x8abc], dtype=np.uint16)
    got = oracle.widen(bits, F16)
    ref = bits.view(np.float16).astype(np.float64)
    np.testing.assert_array_equal(got, ref)


def test_widen_bf16_and_f32():
    x = np.random.default_rng(1).standard_normal(200).astype(np.float32) * 1e3
    b = synth.f32_to_bf16_bits(x)
    np.testing.assert_array_equal(oracle.widen(b, BF16), synth.bf16_bits_to_f32(b).astype(np.float64))
    np.testing.assert_array_equal(oracle.widen(x, F32), x.astype(np.float64))


def test_bf16_rounding_is_rne():
    # 1 + 2^-8 is exactly halfway between bf16 neighbours 1 and 1 + 2^-7: ties to even -> 1
    x = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -2.5], dtype=np.float32)
    got = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(x))
    np.testing.assert_array_equal(got, np.array([1.0, 1 + 2.0 ** -6, -2.5], dtype=np.float32))


# ---------------------------------------------------------------------------
# decode: brute force on contiguous inputs
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", [F32, F16, BF16])
@pytest.mark.parametrize("bias", ["none", "gauss", "t5"])
@pytest.mark.parametrize("window", [-1, 1, 5, 16, 100])
def test_decode_matches_contiguous_bruteforce(dtype, bias, window):
    case = small_case(dtype=dtype, bias=bias, window=window)
    got = run_oracle_decode(case)
    ref = brute_decode(case)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_decode_tiny_workload_matches_bruteforce():
    case = synth.decode_workload(1)
    np.testing.assert_allclose(run_oracle_decode(case), brute_decode(case), rtol=1e-12, atol=1e-12)


def test_decode_thread_count_does_not_change_bits():
    case = small_case(dtype=BF16, ctx=(40, 3, 77, 16), H=3)
    a = run_oracle_decode(case, nthreads=1)
    b = run_oracle_decode(case, nthreads=7)
    np.testing.assert_array_equal(a, b)


def test_decode_pairs_subset_matches_full():
    case = small_case(dtype=F16, ctx=(40, 3, 77, 16), H=3)
    full = run_oracle_decode(case)
    pairs = np.array([[2, 1], [0, 0], [3, 2]], dtype=np.int32)
    sub = run_oracle_decode(case, pairs=pairs)
    np.testing.assert_array_equal(sub, full[pairs[:, 0], pairs[:, 1]])


# ---------------------------------------------------------------------------
# decode: closed forms
# ---------------------------------------------------------------------------
def _vals(case, arr):
    return synth.decode_to_f32(arr, case.dtype).astype(np.float64)


def test_ctx_one_returns_v0_exactly():
    case = small_case(ctx=(1, 1, 1), bias="gauss")
    got = run_oracle_decode(case)
    V = _vals(case, case.value)
    for s in range(3):
        np.testing.assert_array_equal(got[s], V[case.tok_offsets[s]])


def test_window_one_returns_last_value():
    case = small_case(ctx=(1, 9, 16, 40), window=1, bias="gauss")
    got = run_oracle_decode(case)
    V = _vals(case, case.value)
    for s in range(4):
        np.testing.assert_array_equal(got[s], V[case.tok_offsets[s + 1] - 1])


def test_zero_query_zero_bias_is_mean_of_visible_values():
    case = small_case(dtype=F16, ctx=(5, 17, 30), window=12, bias="none")
    case.q[:] = 0
    got = run_oracle_decode(case)
    V = _vals(case, case.value)
    for s in range(3):
        c = int(case.context_lens[s]); lo = max(0, c - 12)
        ref = V[case.tok_offsets[s] + lo:case.tok_offsets[s] + c].mean(axis=0)
        np.testing.assert_allclose(got[s], ref, rtol=0, atol=1e-13)


def test_identical_keys_give_mean_of_values():
    case = small_case(ctx=(9, 20), bias="none")
    case.key[:] = case.key[0]
    got = run_oracle_decode(case)
    V = _vals(case, case.value)
    for s in range(2):
        ref = V[case.tok_offsets[s]:case.tok_offsets[s + 1]].mean(axis=0)
        np.testing.assert_allclose(got[s], ref, rtol=0, atol=1e-13)


def test_one_hot_bias_selects_one_value():
    case = small_case(ctx=(20, 33), bias="gauss", scale=1 / 8)
    case.q[:] = 0
    case.bias[:] = -1e4
    picks = [7, 31]
    for s, j in enumerate(picks):
        case.bias[s, :, j] = 0.0
    got = run_oracle_decode(case)
    V = _vals(case, case.value)
    for s, j in enumerate(picks):
        # every other weight is exp(-1e4 / 8) relative: far below double rounding
        np.testing.assert_allclose(got[s], np.broadcast_to(V[case.tok_offsets[s] + j], got[s].shape),
                                   rtol=0, atol=1e-300)


def test_scale_multiplies_the_bias_two_key_closed_form():
    """Two keys, q = 0: the weights are a logistic function of scale*(a0 - a1).
    A bias left unscaled (or scaled twice) moves the result."""
    case = small_case(ctx=(2,), H=1, bias="gauss", scale=0.3)
    case.q[:] = 0
    case.bias[0, 0, 0] = 1.75          # exactly representable in fp32
    case.bias[0, 0, 1] = -0.375
    got = run_oracle_decode(case)
    V = _vals(case, case.value)
    w0 = 1.0 / (1.0 + math.exp(-0.3 * (1.75 - (-0.375))))
    ref = w0 * V[0, 0] + (1 - w0) * V[1, 0]
    np.testing.assert_allclose(got[0, 0], ref, rtol=1e-14, atol=1e-14)


def test_scale_multiplies_qk_two_key_closed_form():
    """Two keys, no bias, K rows built so q.k0 - q.k1 = delta exactly."""
    case = small_case(ctx=(2,), H=1, bias="none", scale=0.25)
    case.q[:] = 0
    case.q[0, 0, 0] = 1.0
    case.key[:] = 0
    case.key[0, 0, 0] = 3.0
    case.key[1, 0, 0] = -1.0
    got = run_oracle_decode(case)
    V = _vals(case, case.value)
    w0 = 1.0 / (1.0 + math.exp(-0.25 * 4.0))
    np.testing.assert_allclose(got[0, 0], w0 * V[0, 0] + (1 - w0) * V[1, 0], rtol=1e-14, atol=1e-14)


def test_empty_context_gives_zero_row():
    case = small_case(ctx=(0, 5), bias="gauss")
    got = run_oracle_decode(case)
    np.testing.assert_array_equal(got[0], 0.0)
    assert np.isfinite(got).all()


# ---------------------------------------------------------------------------
# decode: invariants
# ---------------------------------------------------------------------------
def test_zero_bias_equals_no_bias():
    case = small_case(dtype=BF16, bias="gauss")
    case.bias[:] = 0
    with_bias = run_oracle_decode(case)
    case.bias = None
    np.testing.assert_array_equal(with_bias, run_oracle_decode(case))


def test_row_constant_added_to_bias_leaves_output():
    case = small_case(dtype=F16, bias="gauss", window=20)
    # bias on a 2^-10 grid and integer shifts: bias + c stays exact in fp32
    case.bias = (np.round(case.bias * 1024) / 1024).astype(np.float32)
    base = run_oracle_decode(case)
    c = np.random.default_rng(3).integers(-50, 51, size=case.bias.shape[:2]).astype(np.float32)
    case.bias = (case.bias + c[:, :, None]).astype(np.float32)
    np.testing.assert_allclose(run_oracle_decode(case), base, rtol=0, atol=1e-12)


def test_block_permutation_leaves_output():
    case = small_case(dtype=BF16, ctx=(40, 3, 77, 16), H=3)
    kc, vc = fill_cache_numpy(case)
    base = oracle.paged_decode(case.q, kc, vc, case.block_tables, case.context_lens, case.bias, -1,
                               case.scale, 16, case.dtype)
    perm = np.random.default_rng(5).permutation(case.num_blocks)      # new position of block b
    kc2 = np.empty_like(kc); vc2 = np.empty_like(vc)
    kc2[perm] = kc; vc2[perm] = vc
    bt2 = np.where(case.block_tables >= 0, perm[np.maximum(case.block_tables, 0)], -1).astype(np.int32)
    got = oracle.paged_decode(case.q, kc2, vc2, bt2, case.context_lens, case.bias, -1, case.scale, 16,
                              case.dtype)
    np.testing.assert_array_equal(got, base)


@pytest.mark.parametrize("extra", [0, 1, 1000])
def test_window_at_least_context_equals_full(extra):
    case = small_case(dtype=F32, ctx=(4, 31, 50))
    full = run_oracle_decode(case)
    case.window = int(case.context_lens.max()) + extra
    np.testing.assert_array_equal(run_oracle_decode(case), full)


def test_bias_outside_window_and_context_is_ignored():
    case = small_case(dtype=F32, ctx=(10, 40), bias="gauss", window=8)
    base = run_oracle_decode(case)
    for s in range(2):
        c = int(case.context_lens[s])
        case.bias[s, :, c:] = np.nan
        case.bias[s, :, :c - 8] = np.nan
    np.testing.assert_array_equal(run_oracle_decode(case), base)


def test_unused_block_table_entries_are_not_read():
    case = small_case(dtype=F32, ctx=(50, 17), window=10, pool_extra=0)
    base = run_oracle_decode(case)
    bt = case.block_tables.copy()
    for s in range(2):
        c = int(case.context_lens[s]); first = (c - 10) // 16
        bt[s, :first] = -1                           # blocks wholly before the window: "evicted"
        bt[s, (c + 15) // 16:] = 2 ** 30              # past the context
    case.block_tables = bt
    np.testing.assert_array_equal(run_oracle_decode(case), base)


# ---------------------------------------------------------------------------
# T5 bias materialisation used by the workloads (golden fixture)
# ---------------------------------------------------------------------------
def test_t5_clamp_fixture():
    path = os.path.join(os.path.dirname(__file__), "golden", "t5_clamp.txt")
    rows = [l.split() for l in open(path) if l.strip() and not l.startswith("#")]
    d = np.array([int(r[0]) for r in rows])
    col = np.array([int(r[1]) for r in rows])
    np.testing.assert_array_equal(synth.t5_bucket(d), col)
    table = np.arange(2 * 129, dtype=np.float32).reshape(2, 129)
    ctx = np.array([300], dtype=np.int32)
    A = synth.t5_bias(table, ctx, 304)
    # key j sits ctx-1-j behind the query
    for j in (299, 298, 171, 170, 0):
        assert A[0, 1, j] == table[1, min(299 - j, 128)]
    assert (A[0, :, 300:] == 0).all()


# ---------------------------------------------------------------------------
# prefill
# ---------------------------------------------------------------------------
def brute_prefill(case):
    H, D = case.num_heads, case.head_dim
    q = synth.decode_to_f32(case.q, case.dtype).astype(np.float64)
    k = synth.decode_to_f32(case.k, case.dtype).astype(np.float64)
    v = synth.decode_to_f32(case.v, case.dtype).astype(np.float64)
    out = np.zeros_like(q)
    cu = case.cu_seqlens
    for b in range(len(cu) - 1):
        a, e = int(cu[b]), int(cu[b + 1])
        L = e - a
        if L == 0:
            continue
        r = np.arange(L)[:, None]; c = np.arange(L)[None, :]
        keep = np.ones((L, L), dtype=bool)
        if case.causal:
            keep &= c <= r
        if case.window > 0:
            keep &= np.abs(r - c) < case.window
        logits = np.einsum("ihd,jhd->hij", q[a:e], k[a:e]) * case.scale
        logits = np.where(keep[None], logits, -np.inf)
        w = np.exp(logits - logits.max(axis=2, keepdims=True))
        w /= w.sum(axis=2, keepdims=True)
        out[a:e] = np.einsum("hij,jhd->ihd", w, v[a:e])
    return out


def run_oracle_prefill(case, rows=None, nthreads=None):
    return oracle.prefill(case.q, case.k, case.v, case.cu_seqlens, case.window, case.causal, case.scale,
                          case.dtype, rows=rows, nthreads=nthreads)


@pytest.mark.parametrize("window", [-1, 1, 3, 64])
@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("dtype", [BF16, F16])
def test_prefill_matches_bruteforce(window, causal, dtype):
    case = synth.make_prefill_case("pin", 11, [1, 7, 70, 130], 2, 64, window, causal, dtype)
    np.testing.assert_allclose(run_oracle_prefill(case), brute_prefill(case), rtol=1e-12, atol=1e-12)


def test_prefill_window_one_is_identity_on_values():
    case = synth.make_prefill_case("pin", 12, [5, 33], 3, 64, 1, 0, BF16)
    got = run_oracle_prefill(case)
    np.testing.assert_array_equal(got, synth.decode_to_f32(case.v, BF16).astype(np.float64))


def test_prefill_causal_first_row_is_v0():
    case = synth.make_prefill_case("pin", 13, [9, 4], 2, 64, -1, 1, BF16)
    got = run_oracle_prefill(case)
    v = synth.decode_to_f32(case.v, BF16).astype(np.float64)
    for a in case.cu_seqlens[:-1]:
        np.testing.assert_array_equal(got[a], v[a])


def test_prefill_zero_query_band_mean():
    case = synth.make_prefill_case("pin", 14, [40], 1, 64, 5, 0, BF16)
    case.q[:] = 0
    got = run_oracle_prefill(case)
    v = synth.decode_to_f32(case.v, BF16).astype(np.float64)
    for i in range(40):
        lo, hi = max(0, i - 4), min(40, i + 5)
        np.testing.assert_allclose(got[i], v[lo:hi].mean(axis=0), rtol=0, atol=1e-13)


def test_prefill_sampled_rows_match_full():
    case = synth.make_prefill_case("pin", 15, [20, 50, 3], 2, 64, 7, 0, BF16)
    full = run_oracle_prefill(case)
    rows = np.array([0, 19, 20, 69, 72, 45], dtype=np.int64)
    np.testing.assert_array_equal(run_oracle_prefill(case, rows=rows), full[rows])


def test_prefill_bidirectional_band_is_symmetric_under_reversal():
    """Reversing a sequence's tokens maps the band |i-j|<W onto itself."""
    case = synth.make_prefill_case("pin", 16, [37], 2, 64, 6, 0, BF16)
    base = run_oracle_prefill(case)
    case.q = case.q[::-1].copy(); case.k = case.k[::-1].copy(); case.v = case.v[::-1].copy()
    np.testing.assert_allclose(run_oracle_prefill(case)[::-1], base, rtol=0, atol=1e-13)


@pytest.mark.parametrize("window", [1, 6, 25, -1])
def test_decode_is_last_row_of_causal_prefill(window):
    """A decode query at position ctx-1 over a paged cache equals the last row
    of a causal (windowed) prefill over the same tokens, when the decode query
    is that last row's query."""
    pre = synth.make_prefill_case("pin", 17, [25, 40], 2, 64, window, 1, BF16)
    ctx = np.array([25, 40], dtype=np.int32)
    dec = small_case(dtype=BF16, ctx=ctx, H=2, bias="none", window=window, scale=pre.scale)
    dec.key = pre.k.copy(); dec.value = pre.v.copy()
    last = pre.cu_seqlens[1:] - 1
    dec.q = pre.q[last].copy()
    got = run_oracle_decode(dec)
    ref = run_oracle_prefill(pre, rows=last.astype(np.int64))
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-13)


# ---------------------------------------------------------------------------
# reshape_and_cache
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", [F32, F16, BF16])
def test_reshape_and_cache_round_trip_and_skip(dtype):
    case = small_case(dtype=dtype, ctx=(5, 40, 16), H=3, pool_extra=3)
    slots = case.slot_mapping.copy()
    slots[[1, 7, 30]] = -1
    shape = (case.num_blocks, 3, 16, 64)
    poison = np.frombuffer(np.full(int(np.prod(shape)) * case.key.itemsize, 0xA5, np.uint8).tobytes(),
                           dtype=case.key.dtype).reshape(shape)
    kc = poison.copy(); vc = poison.copy()
    oracle.reshape_and_cache(kc, vc, case.key, case.value, slots, 16)
    for t, sl in enumerate(slots):
        if sl < 0:
            continue
        assert kc[sl // 16, :, sl % 16, :].tobytes() == case.key[t].tobytes()
        assert vc[sl // 16, :, sl % 16, :].tobytes() == case.value[t].tobytes()
    written = np.zeros(case.num_blocks * 16, dtype=bool)
    written[slots[slots >= 0]] = True
    kb = kc.transpose(0, 2, 1, 3).reshape(case.num_blocks * 16, -1)
    pb = poison.transpose(0, 2, 1, 3).reshape(case.num_blocks * 16, -1)
    assert kb[~written].tobytes() == pb[~written].tobytes()


# ---------------------------------------------------------------------------
# decode with the T5 bias read from its table
# ---------------------------------------------------------------------------
def run_oracle_decode_t5(case, table, **kw):
    kc, vc = fill_cache_numpy(case)
    return oracle.paged_decode_t5(case.q, kc, vc, case.block_tables, case.context_lens, table, case.window,
                                  case.scale, case.block_size, case.dtype, **kw)


@pytest.mark.parametrize("window", [-1, 7, 200])
@pytest.mark.parametrize("buckets", [1, 5, 129])
def test_t5_table_decode_equals_materialised_bias(window, buckets):
    """Reading A from the table equals brute force with A materialised by the
    (fixture-pinned) T5 clamp, for any number of table columns."""
    case = small_case(dtype=BF16, ctx=(1, 3, 16, 17, 150, 260), H=3, bias="none", window=window)
    table = np.random.default_rng(9).standard_normal((3, buckets)).astype(np.float32)
    A = np.zeros((case.num_seqs, 3, 264), dtype=np.float32)
    for s, c in enumerate(case.context_lens):
        d = np.minimum((int(c) - 1) - np.arange(int(c)), buckets - 1)
        A[s, :, :c] = table[:, d]
    got = run_oracle_decode_t5(case, table)
    case.bias = A
    np.testing.assert_allclose(got, brute_decode(case), rtol=1e-12, atol=1e-12)


def test_t5_table_constant_rows_equal_no_bias():
    case = small_case(dtype=F32, ctx=(5, 40, 77), H=2, bias="none")
    table = np.repeat(np.array([[0.75], [-2.5]], dtype=np.float32), 129, axis=1)
    np.testing.assert_allclose(run_oracle_decode_t5(case, table), run_oracle_decode(case), rtol=0, atol=1e-13)


# ---------------------------------------------------------------------------
# chunked local attention prefill
# ---------------------------------------------------------------------------
def _split_into_chunks(cu, C):
    """cu_seqlens of the same tokens cut into chunks of C positions."""
    out = [0]
    for b in range(len(cu) - 1):
        a, e = int(cu[b]), int(cu[b + 1])
        for s in range(a, e, C):
            out.append(min(s + C, e))
    return np.array(out, dtype=np.int32)


@pytest.mark.parametrize("C", [1, 3, 16, 64, 1000])
@pytest.mark.parametrize("causal", [0, 1])
def test_chunked_equals_full_attention_over_the_chunks(C, causal):
    """Chunked attention over a sequence is exactly (causal or full) attention
    over the packed batch of its chunks."""
    case = synth.make_prefill_case("pin", 18, [1, 7, 70, 130], 2, 64, -1, causal, BF16)
    got = oracle.prefill_chunked(case.q, case.k, case.v, case.cu_seqlens, C, causal, case.scale, BF16)
    ref = oracle.prefill(case.q, case.k, case.v, _split_into_chunks(case.cu_seqlens, C), -1, causal,
                         case.scale, BF16)
    np.testing.assert_array_equal(got, ref)


def test_chunked_matches_bruteforce():
    case = synth.make_prefill_case("pin", 19, [5, 40, 100], 2, 64, -1, 0, BF16)
    q = synth.decode_to_f32(case.q, BF16).astype(np.float64)
    k = synth.decode_to_f32(case.k, BF16).astype(np.float64)
    v = synth.decode_to_f32(case.v, BF16).astype(np.float64)
    C = 16
    ref = np.zeros_like(q)
    cu = case.cu_seqlens
    for b in range(len(cu) - 1):
        a, e = int(cu[b]), int(cu[b + 1])
        r = np.arange(e - a)
        keep = (r[:, None] // C) == (r[None, :] // C)
        lg = np.einsum("ihd,jhd->hij", q[a:e], k[a:e]) * case.scale
        lg = np.where(keep[None], lg, -np.inf)
        w = np.exp(lg - lg.max(axis=2, keepdims=True)); w /= w.sum(axis=2, keepdims=True)
        ref[a:e] = np.einsum("hij,jhd->ihd", w, v[a:e])
    got = oracle.prefill_chunked(case.q, case.k, case.v, cu, C, 0, case.scale, BF16)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# relative-position bias in prefill; prefill against the paged cache
# ---------------------------------------------------------------------------
def _rel_cols(rel, d):
    """Columns of the signed table for distances d (any shape), saturated."""
    cap = (rel.shape[1] - 1) // 2
    return cap + np.clip(d, -cap, cap)


def _softmax_rows(lg, keep, V):
    """Masked softmax over the last axis of lg [H, n, m]; rows that keep no key
    give zeros.  V: [m, H, D] -> [n, H, D]."""
    lg = np.where(keep[None], lg, -np.inf)
    m = lg.max(axis=2, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    w = np.where(keep[None], np.exp(lg - m), 0.0)
    tot = w.sum(axis=2, keepdims=True)
    w = np.divide(w, tot, out=np.zeros_like(w), where=tot > 0)
    return np.einsum("hij,jhd->ihd", w, V)


def brute_prefill_biased(case):
    q = synth.decode_to_f32(case.q, case.dtype).astype(np.float64)
    k = synth.decode_to_f32(case.k, case.dtype).astype(np.float64)
    v = synth.decode_to_f32(case.v, case.dtype).astype(np.float64)
    rel = case.rel_bias.astype(np.float64)
    out = np.zeros_like(q)
    cu = case.cu_seqlens
    for b in range(len(cu) - 1):
        a, e = int(cu[b]), int(cu[b + 1])
        if e == a:
            continue
        r = np.arange(e - a)[:, None]; c = np.arange(e - a)[None, :]
        keep = np.ones((e - a, e - a), dtype=bool)
        if case.causal:
            keep &= c <= r
        if case.window > 0:
            keep &= np.abs(r - c) < case.window
        lg = (np.einsum("ihd,jhd->hij", q[a:e], k[a:e]) + rel[:, _rel_cols(rel, r - c)]) * case.scale
        out[a:e] = _softmax_rows(lg, keep, v[a:e])
    return out


def brute_paged_prefill(pc):
    """From the token arrays (no block table): the last Lq positions of each
    sequence against its ctx contiguous keys."""
    c = pc.cache
    q = synth.decode_to_f32(pc.q, pc.dtype).astype(np.float64)
    K = synth.decode_to_f32(c.key, pc.dtype).astype(np.float64)
    V = synth.decode_to_f32(c.value, pc.dtype).astype(np.float64)
    out = np.zeros_like(q)
    for s in range(pc.num_seqs):
        a, e = int(pc.cu_seqlens_q[s]), int(pc.cu_seqlens_q[s + 1])
        ctx = int(c.context_lens[s])
        if e == a or ctx == 0:
            continue
        t0 = int(c.tok_offsets[s])
        p = ctx - (e - a) + np.arange(e - a)[:, None]
        col = np.arange(ctx)[None, :]
        keep = np.ones((e - a, ctx), dtype=bool)
        if pc.causal:
            keep &= col <= p
        if pc.window > 0:
            keep &= np.abs(p - col) < pc.window
        lg = np.einsum("ihd,jhd->hij", q[a:e], K[t0:t0 + ctx])
        if pc.rel_bias is not None:
            rel = pc.rel_bias.astype(np.float64)
            lg = lg + rel[:, _rel_cols(rel, p - col)]
        out[a:e] = _softmax_rows(lg * pc.scale, keep, V[t0:t0 + ctx])
    return out


def run_oracle_paged_prefill(pc, **kw):
    kc, vc = fill_cache_numpy(pc.cache)
    return oracle.paged_prefill(pc.q, kc, vc, pc.cache.block_tables, pc.cu_seqlens_q, pc.cache.context_lens,
                                pc.window, pc.causal, pc.scale, pc.cache.block_size, pc.dtype, rel_bias=pc.rel_bias,
                                **kw)


def biased_case(seqlens, window, causal, buckets=5, dtype=BF16, seed=23):
    case = synth.make_prefill_case("pin", seed, seqlens, 2, 64, window, causal, dtype)
    case.rel_bias = synth.rel_bias_table(seed, 2, buckets)
    return case


def run_oracle_prefill_biased(case, **kw):
    return oracle.prefill_biased(case.q, case.k, case.v, case.cu_seqlens, case.window, case.causal, case.scale,
                                 case.dtype, case.rel_bias, **kw)


PAGED_CTX = (1, 15, 16, 17, 40, 100, 130)
PAGED_QL = (1, 15, 5, 17, 3, 60, 130)


def paged_case(window=-1, causal=1, buckets=0, dtype=BF16, ctx=PAGED_CTX, ql=PAGED_QL, seed=29):
    return synth.make_paged_prefill_case("pin", seed, dtype, ctx, ql, 2, 64, window, causal, buckets,
                                         pool_blocks=40)


@pytest.mark.parametrize("window", [-1, 1, 9, 200])
@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("buckets", [1, 5, 129])
def test_biased_prefill_matches_bruteforce(window, causal, buckets):
    case = biased_case([1, 7, 70, 130], window, causal, buckets)
    np.testing.assert_allclose(run_oracle_prefill_biased(case), brute_prefill_biased(case), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("window", [-1, 1, 7, 300])
@pytest.mark.parametrize("causal", [0, 1])
@pytest.mark.parametrize("buckets", [0, 129])
@pytest.mark.parametrize("dtype", [BF16, F32])
def test_paged_prefill_matches_bruteforce(window, causal, buckets, dtype):
    pc = paged_case(window, causal, buckets, dtype)
    np.testing.assert_allclose(run_oracle_paged_prefill(pc), brute_paged_prefill(pc), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("window", [-1, 3])
def test_paged_prefill_more_queries_than_keys_and_empty_context(window):
    """Without the causal mask a sequence may have more query rows than keys
    (early rows sit at negative positions) or no keys at all (zero rows)."""
    pc = paged_case(window, 0, 4, ctx=(5, 0, 30), ql=(9, 3, 4))
    got = run_oracle_paged_prefill(pc)
    np.testing.assert_allclose(got, brute_paged_prefill(pc), rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(got[9:12], 0.0)


def test_rel_bias_one_hot_selects_previous_key():
    """A huge bias at distance +1 only: every query r >= 1 returns v_{r-1}
    exactly (a sign slip would return v_{r+1})."""
    case = biased_case([12, 30], -1, 0, buckets=4, dtype=F32)
    case.rel_bias[:] = 0
    case.rel_bias[:, 3 + 1] = 1e4
    case.scale = 1.0
    got = run_oracle_prefill_biased(case)
    v = synth.decode_to_f32(case.v, F32).astype(np.float64)
    for a, e in zip(case.cu_seqlens[:-1], case.cu_seqlens[1:]):
        np.testing.assert_array_equal(got[a + 1:e], v[a:e - 1])


def test_paged_rel_bias_one_hot_selects_key_before_the_query_position():
    """Paged and causal: with the huge bias at distance +1, query row r of a
    sequence (position ctx - Lq + r) returns the value at position ctx - Lq + r - 1."""
    pc = paged_case(-1, 1, 4, F32, ctx=(20, 37, 16), ql=(5, 37, 1))
    pc.rel_bias[:] = 0
    pc.rel_bias[:, 3 + 1] = 1e4
    pc.scale = 1.0
    got = run_oracle_paged_prefill(pc)
    V = synth.decode_to_f32(pc.cache.value, F32).astype(np.float64)
    for s in range(pc.num_seqs):
        a, e = int(pc.cu_seqlens_q[s]), int(pc.cu_seqlens_q[s + 1])
        ctx, t0 = int(pc.cache.context_lens[s]), int(pc.cache.tok_offsets[s])
        for r in range(e - a):
            p = ctx - (e - a) + r
            if p >= 1:
                np.testing.assert_array_equal(got[a + r], V[t0 + p - 1])


def test_rel_bias_saturates_at_the_last_column():
    """Zero query, bias b only in the saturated column (distance >= cap):
    the weights take two values, split exactly at distance cap."""
    B, cap, b = 4, 3, 1.5
    case = biased_case([20], -1, 0, buckets=B, dtype=F32)
    case.q[:] = 0
    case.rel_bias[:] = 0
    case.rel_bias[:, 2 * cap] = b
    got = run_oracle_prefill_biased(case)
    v = synth.decode_to_f32(case.v, F32).astype(np.float64)
    for r in range(20):
        wts = np.where(r - np.arange(20) >= cap, math.exp(b * case.scale), 1.0)
        ref = np.einsum("j,jhd->hd", wts, v[:20]) / wts.sum()
        np.testing.assert_allclose(got[r], ref, rtol=1e-13, atol=1e-13)


def test_rel_bias_constant_shift_leaves_output():
    case = biased_case([9, 50], 7, 0, buckets=6)
    case.rel_bias = (np.round(case.rel_bias * 1024) / 1024).astype(np.float32)   # + 3 stays exact in f32
    a = run_oracle_prefill_biased(case)
    case.rel_bias = case.rel_bias + np.float32(3.0)
    np.testing.assert_allclose(run_oracle_prefill_biased(case), a, rtol=0, atol=1e-12)


def test_paged_prefill_of_whole_sequences_equals_packed_causal_prefill():
    """Querying every position (Lq = ctx) through the block table is the
    causal biased prefill over the contiguous tokens."""
    ctx = (1, 16, 17, 90)
    pc = paged_case(-1, 1, 7, ctx=ctx, ql=ctx)
    got = run_oracle_paged_prefill(pc)
    packed = synth.make_prefill_case("pin", 1, list(ctx), 2, 64, -1, 1, BF16, pc.scale)
    packed.q, packed.k, packed.v, packed.rel_bias = pc.q, pc.cache.key, pc.cache.value, pc.rel_bias
    np.testing.assert_allclose(got, run_oracle_prefill_biased(packed), rtol=0, atol=1e-13)


def test_noncausal_paged_prefill_rows_are_paged_decodes():
    """Without mask or bias, every query row is a decode over all ctx keys of
    its sequence (a decoder prompt's cross-attention)."""
    pc = paged_case(-1, 0, 0)
    got = run_oracle_paged_prefill(pc)
    seq = np.repeat(np.arange(pc.num_seqs), pc.query_lens)
    kc, vc = fill_cache_numpy(pc.cache)
    ref = oracle.paged_decode(pc.q, kc, vc, pc.cache.block_tables[seq], pc.cache.context_lens[seq], None, -1,
                              pc.scale, 16, pc.dtype)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-13)


def test_causal_paged_prefill_last_rows_are_t5_decodes():
    """The last query row of each sequence is the decode at position ctx-1
    with the table's non-negative half as the T5 decode table."""
    pc = paged_case(-1, 1, 129)
    last = (pc.cu_seqlens_q[1:] - 1).astype(np.int64)
    got = run_oracle_paged_prefill(pc, rows=last)
    kc, vc = fill_cache_numpy(pc.cache)
    ref = oracle.paged_decode_t5(pc.q[last], kc, vc, pc.cache.block_tables, pc.cache.context_lens,
                                 np.ascontiguousarray(pc.rel_bias[:, 128:]), -1, pc.scale, 16, pc.dtype)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-13)
