"""Planted mistakes: each test copies oracle.c, plants one plausible mistake
(a dropped term, an off-by-one, a transposed index), builds the mutant on the
CPU and checks that at least one pin catches it.  The real oracle is never
modified.  No GPU."""
import ctypes
import os
import subprocess
import tempfile

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "bias_not_scaled": ("x[t] = c->scale * (dot + a);", "x[t] = c->scale * dot + a;"),
    "window_off_by_one": ("start = ctx - c->window;", "start = ctx - c->window + 1;"),
    "block_index": ("[(size_t)s * c->max_blocks_per_seq + j / bs]",
                    "[(size_t)s * c->max_blocks_per_seq + (j + 1) / bs]"),
    "head_and_slot_transposed": ("(((size_t)blk * H + h) * bs + (j % bs)) * D",
                                 "(((size_t)blk * bs + (j % bs)) * H + h) * D"),
    "no_normalisation": ("for (int d = 0; d < D; ++d) out[d] /= l;", ""),
    "q_from_wrong_head": ("const size_t qoff = ((size_t)s * H + h) * D;",
                          "const size_t qoff = ((size_t)s * H + (H - 1 - h)) * D;"),
    "prefill_causal_flipped": ("if (causal && c > r) return 0;", "if (causal && c < r) return 0;"),
    "prefill_window_inclusive": ("if (d >= window) return 0;", "if (d > window) return 0;"),
    "scatter_layout": ("(((size_t)blk * num_heads + h) * block_size + off) * rowb",
                       "(((size_t)blk * block_size + off) * num_heads + h) * rowb"),
    "f16_exponent_bias": ("expo - 25", "expo - 24"),
    "t5_distance_off_by_one": ("int d = (ctx - 1) - j;", "int d = ctx - j;"),
    "chunk_boundary_shifted": ("if (chunk > 0 && r / chunk != c / chunk) return 0;",
                               "if (chunk > 0 && (r + 1) / chunk != (c + 1) / chunk) return 0;"),
    "rel_bias_sign_flipped": ("rel_term(c->rel_bias, c->num_buckets, h, r - col)",
                              "rel_term(c->rel_bias, c->num_buckets, h, col - r)"),
    "rel_bias_clamp_off_by_one": ("if (d > cap) d = cap;", "if (d > cap - 1) d = cap - 1;"),
    "paged_prefill_position_offset_dropped": ("const int pos = ctx - Lq + (int)(i - c->cu_seqlens_q[b]);",
                                              "const int pos = (int)(i - c->cu_seqlens_q[b]);"),
    "paged_prefill_bias_distance_reversed": ("rel_term(c->rel_bias, c->num_buckets, h, pos - col)",
                                             "rel_term(c->rel_bias, c->num_buckets, h, col - pos)"),
}


def _pin_suite():
    """A fixed selection of pins, each called with concrete arguments."""
    yield lambda: pins.test_widen_f16_matches_numpy()
    for dt in (pins.F32, pins.BF16):
        for bias in ("none", "gauss"):
            for w in (-1, 5):
                yield lambda dt=dt, bias=bias, w=w: pins.test_decode_matches_contiguous_bruteforce(dt, bias, w)
    yield pins.test_scale_multiplies_the_bias_two_key_closed_form
    yield pins.test_window_one_returns_last_value
    for w, c in ((-1, 1), (3, 0), (64, 1)):
        yield lambda w=w, c=c: pins.test_prefill_matches_bruteforce(w, c, pins.BF16)
    yield lambda: pins.test_reshape_and_cache_round_trip_and_skip(pins.F16)
    yield lambda: pins.test_t5_table_decode_equals_materialised_bias(-1, 129)
    yield pins.test_chunked_matches_bruteforce
    yield pins.test_rel_bias_one_hot_selects_previous_key
    yield pins.test_paged_rel_bias_one_hot_selects_key_before_the_query_position
    yield pins.test_rel_bias_saturates_at_the_last_column
    for causal in (0, 1):
        yield lambda causal=causal: pins.test_paged_prefill_matches_bruteforce(7, causal, 129, pins.BF16)
        yield lambda causal=causal: pins.test_biased_prefill_matches_bruteforce(9, causal, 5)


def _build_mutant(name, tmpdir):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    path = os.path.join(tmpdir, f"{name}.c")
    open(path, "w").write(src.replace(old, new))
    so = os.path.join(tmpdir, f"lib{name}.so")
    subprocess.check_call(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-pthread", path, "-o", so, "-lm"])
    return so


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    real = oracle._load()
    with tempfile.TemporaryDirectory() as d:
        so = _build_mutant(name, d)
        mut = ctypes.CDLL(so)
        for fn in ("oracle_paged_decode", "oracle_paged_decode_t5", "oracle_prefill", "oracle_prefill_chunked",
                   "oracle_prefill_biased", "oracle_paged_prefill", "oracle_reshape_and_cache", "oracle_widen"):
            getattr(mut, fn).argtypes = getattr(real, fn).argtypes
            getattr(mut, fn).restype = getattr(real, fn).restype
        monkeypatch.setattr(oracle, "_lib", mut)
        caught = 0
        for pin in _pin_suite():
            try:
                pin()
            except AssertionError:
                caught += 1
        assert caught > 0, f"no pin caught the planted mistake {name}"
