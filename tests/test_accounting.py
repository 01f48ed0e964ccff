"""The bench's algorithmic byte and FLOP accounting against brute-force
enumeration on small cases: every roofline fraction divides by these.  No GPU."""
import numpy as np
import pytest

import bench
import synth
from synth import BF16, F16, F32


def _mask_count(L, Lk, qoff, window, causal, chunk):
    """Kept (query, key) pairs by enumeration: query row r at key position r + qoff."""
    n = 0
    for r in range(L):
        p = r + qoff
        for c in range(Lk):
            if causal and c > p:
                continue
            if chunk > 0 and (p // chunk != c // chunk):
                continue
            if window > 0 and abs(p - c) >= window:
                continue
            n += 1
    return n


@pytest.mark.parametrize("window,causal,chunk", [(-1, 0, 0), (-1, 1, 0), (1, 0, 0), (5, 0, 0), (5, 1, 0),
                                                 (300, 0, 0), (-1, 1, 7), (-1, 0, 16)])
def test_prefill_visible_pairs_match_enumeration(window, causal, chunk):
    lens = [1, 2, 17, 40, 129]
    case = synth.make_prefill_case("acct", 1, lens, 1, 64, window, causal, BF16)
    case.chunk = chunk
    want = sum(_mask_count(L, L, 0, window, causal, chunk) for L in lens)
    assert case.visible_pairs() == want
    assert bench.prefill_flops(case) == 4 * 64 * 1 * want
    rows = np.arange(case.num_tokens, dtype=np.int64)
    assert bench._kept_keys(case, rows) == want


@pytest.mark.parametrize("window,causal", [(-1, 1), (-1, 0), (3, 1), (3, 0), (50, 1)])
def test_paged_prefill_kept_pairs_match_enumeration(window, causal):
    ctx, ql = [1, 15, 16, 40, 100, 5, 0], [1, 15, 3, 40, 7, 9, 2]
    if causal:
        ql = [min(a, b) for a, b in zip(ql, ctx)]
    pc = synth.make_paged_prefill_case("acct", 2, BF16, ctx, ql, 2, 64, window, causal, pool_blocks=40)
    want = sum(_mask_count(l, c, c - l, window, causal, 0) for l, c in zip(ql, ctx))
    assert pc.kept_pairs() == want
    rows = np.arange(pc.num_tokens, dtype=np.int64)
    assert bench._kept_keys(pc, rows) == want


@pytest.mark.parametrize("dtype,D,window,bias", [(F32, 64, -1, "gauss"), (BF16, 64, 5, "none"),
                                                 (F16, 128, 20, "gauss")])
def test_decode_algorithmic_bytes_match_a_hand_count(dtype, D, window, bias):
    ctx = [0, 1, 15, 16, 17, 33, 100]
    case = synth.make_decode_case("acct", 3, dtype, len(ctx), 3, D, context_lens=np.array(ctx), window=window,
                                  bias=bias)
    elt = 4 if dtype == F32 else 2
    H = 3
    kv = bias_b = other = 0
    for c in ctx:
        n = min(c, window) if window > 0 else c         # keys [max(0, c - W), c)
        kv += 2 * H * n * D * elt
        if bias != "none":
            bias_b += 4 * H * n
        other += 2 * H * D * elt + 4 * ((n + 15) // 16)
    other += 4 * len(ctx)
    got = bench.decode_alg_bytes(case, bias_on=True)
    assert (got["kv"], got["bias"], got["other"]) == (kv, bias_b, other)
    assert got["total"] == kv + bias_b + other
    assert bench.decode_alg_bytes(case, bias_on=False)["bias"] == 0


def test_t5_table_decode_counts_the_table_not_the_rows():
    case = synth.decode_workload(2)
    got = bench.decode_alg_bytes(case, bias_on=True, t5_table=True)
    assert got["bias"] == 8 * 129 * 4
