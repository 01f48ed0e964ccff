"""fp64 CPU oracle for paged-KV attention — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  It wraps ``oracle.c`` (plain C, double
precision, pthreads) through ctypes and shares nothing with the CUDA library.

Functions and the passages they follow:

* ``paged_decode`` — "PagedAttention: Support custom attention bias for T5
  model (1/2)", the opening formula softmax((QK^T + A)/sqrt(d_k)) V with the
  optional, materialised, padded bias; K/V gathered through the block table
  passed in ("Add Encoder-decoder model support and T5 Model support": one
  table for decoder self-attention, another for encoder cross-attention);
  causal sliding window keeping the W most recent keys ("[V1] Add sliding
  window support to Flex Attention backend").
* ``paged_decode_t5`` — the same with the bias read from a T5 relative-
  position table [H, num_buckets] at column min(ctx - 1 - j, num_buckets - 1)
  (same page: capped distance, last value reused; computing the T5 bias in
  the kernel instead of materialising it).
* ``prefill`` — the same softmax attention for every row of a packed varlen
  batch, mask = full / causal / bidirectional band |i-j| < W / causal band
  ("[V1] Add sliding window support to Flex Attention backend").
* ``prefill_chunked`` — keys restricted to the query's own chunk of C
  positions, bidirectional or causal (the chunked local attention layers the
  same page discusses).
* ``prefill_biased`` — ``prefill`` with an additive relative-position bias
  rel_bias[h, B-1 + clamp(r - c, -(B-1), B-1)] inside the scaled logits: the
  T5 bias of an encoder's bidirectional self-attention ("Add Encoder-decoder
  model support and T5 Model support"; capped distance as in the T5-bias
  page).  A causal layer reads only the non-negative half = the decode table.
* ``paged_prefill`` — prefill of each sequence's newest Lq tokens against its
  ctx keys in the paged cache, read through the block table passed in (same
  encoder-decoder page: prefill and decode kernels both read the separate
  cross-attention blocks); query row r sits at key position ctx - Lq + r.
* ``reshape_and_cache`` — the plain scatter of new K/V rows into cache blocks
  (the cross-attention KV caching step named in "Add Encoder-decoder model
  support and T5 Model support").

Every function is pinned by ``tests/test_oracle_pins.py`` against brute force
on contiguous inputs, closed forms and invariants.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain gcc, strict IEEE double)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I = ctypes.c_int
        lib.oracle_paged_decode.argtypes = [P, P, P, P, P, P, P, I, ctypes.c_double, I, I, I, I, I, I, I,
                                            P, I, I]
        lib.oracle_paged_decode.restype = None
        lib.oracle_paged_decode_t5.argtypes = [P, P, P, P, P, P, P, I, I, ctypes.c_double, I, I, I, I, I, I,
                                               P, I, I]
        lib.oracle_paged_decode_t5.restype = None
        lib.oracle_prefill.argtypes = [P, P, P, P, P, I, I, I, I, I, ctypes.c_double, I, P,
                                       ctypes.c_longlong, I]
        lib.oracle_prefill.restype = None
        lib.oracle_prefill_chunked.argtypes = [P, P, P, P, P, I, I, I, I, I, ctypes.c_double, I, P,
                                               ctypes.c_longlong, I]
        lib.oracle_prefill_chunked.restype = None
        lib.oracle_prefill_biased.argtypes = [P, P, P, P, P, I, I, I, I, I, ctypes.c_double, I, P, I, P,
                                              ctypes.c_longlong, I]
        lib.oracle_prefill_biased.restype = None
        lib.oracle_paged_prefill.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, ctypes.c_double, P, I, I,
                                             P, ctypes.c_longlong, I]
        lib.oracle_paged_prefill.restype = None
        lib.oracle_reshape_and_cache.argtypes = [P, P, P, P, P, ctypes.c_longlong, I, I, I, I]
        lib.oracle_reshape_and_cache.restype = None
        lib.oracle_widen.argtypes = [P, ctypes.c_longlong, I]
        lib.oracle_widen.restype = ctypes.c_double
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype=None):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=dtype) if dtype is not None else np.ascontiguousarray(a)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def widen(a: np.ndarray, dtype: int) -> np.ndarray:
    """The oracle's own exact widening of stored values to double (for pins)."""
    lib = _load()
    a = _c(a)
    return np.array([lib.oracle_widen(_ptr(a), i, dtype) for i in range(a.size)], dtype=np.float64)


def paged_decode(q, k_cache, v_cache, block_tables, context_lens, bias, window, scale, block_size,
                 dtype, pairs=None, nthreads=None) -> np.ndarray:
    """Decode output in double: [S, H, D], or [len(pairs), D] for listed (s, h)."""
    lib = _load()
    q = _c(q); k_cache = _c(k_cache); v_cache = _c(v_cache)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    S, H, D = q.shape
    bias = _c(bias, np.float32) if bias is not None else None
    stride = int(bias.shape[2]) if bias is not None else 0
    pr = _c(pairs, np.int32) if pairs is not None else None
    n = len(pr) if pr is not None else S * H
    out = np.zeros((n, D), dtype=np.float64)
    lib.oracle_paged_decode(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), _ptr(cl), _ptr(bias),
                            int(window), float(scale), int(block_size), S, H, D, int(bt.shape[1]), stride,
                            int(dtype), _ptr(pr), n, int(nthreads or default_threads()))
    return out if pr is not None else out.reshape(S, H, D)


def paged_decode_t5(q, k_cache, v_cache, block_tables, context_lens, bias_table, window, scale, block_size,
                    dtype, pairs=None, nthreads=None) -> np.ndarray:
    """Decode with the T5 bias read from its [H, num_buckets] table."""
    lib = _load()
    q = _c(q); k_cache = _c(k_cache); v_cache = _c(v_cache)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    tab = _c(bias_table, np.float32)
    S, H, D = q.shape
    pr = _c(pairs, np.int32) if pairs is not None else None
    n = len(pr) if pr is not None else S * H
    out = np.zeros((n, D), dtype=np.float64)
    lib.oracle_paged_decode_t5(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), _ptr(cl), _ptr(tab),
                               int(tab.shape[1]), int(window), float(scale), int(block_size), S, H, D,
                               int(bt.shape[1]), int(dtype), _ptr(pr), n, int(nthreads or default_threads()))
    return out if pr is not None else out.reshape(S, H, D)


def prefill(q, k, v, cu_seqlens, window, causal, scale, dtype, rows=None, nthreads=None) -> np.ndarray:
    """Prefill output in double: [T, H, D], or [len(rows), H, D] for listed rows."""
    lib = _load()
    q = _c(q); k = _c(k); v = _c(v)
    cu = _c(cu_seqlens, np.int32)
    T, H, D = q.shape
    rr = _c(rows, np.int64) if rows is not None else None
    nr = len(rr) if rr is not None else int(cu[-1])
    out = np.zeros((nr, H, D), dtype=np.float64)
    lib.oracle_prefill(_ptr(out), _ptr(q), _ptr(k), _ptr(v), _ptr(cu), len(cu) - 1, H, D, int(window),
                       int(causal), float(scale), int(dtype), _ptr(rr), nr, int(nthreads or default_threads()))
    return out


def prefill_chunked(q, k, v, cu_seqlens, chunk, causal, scale, dtype, rows=None, nthreads=None) -> np.ndarray:
    """Chunked local attention prefill in double: [T or len(rows), H, D]."""
    lib = _load()
    q = _c(q); k = _c(k); v = _c(v)
    cu = _c(cu_seqlens, np.int32)
    T, H, D = q.shape
    rr = _c(rows, np.int64) if rows is not None else None
    nr = len(rr) if rr is not None else int(cu[-1])
    out = np.zeros((nr, H, D), dtype=np.float64)
    lib.oracle_prefill_chunked(_ptr(out), _ptr(q), _ptr(k), _ptr(v), _ptr(cu), len(cu) - 1, H, D, int(chunk),
                               int(causal), float(scale), int(dtype), _ptr(rr), nr,
                               int(nthreads or default_threads()))
    return out


def prefill_biased(q, k, v, cu_seqlens, window, causal, scale, dtype, rel_bias, rows=None,
                   nthreads=None) -> np.ndarray:
    """Prefill with the relative-position bias rel_bias [H, 2B-1]:
    x = scale * (q.k + rel_bias[h, B-1 + clamp(r - c, -(B-1), B-1)])."""
    lib = _load()
    q = _c(q); k = _c(k); v = _c(v)
    cu = _c(cu_seqlens, np.int32)
    rb = _c(rel_bias, np.float32)
    T, H, D = q.shape
    assert rb.shape[0] == H and rb.shape[1] % 2 == 1
    rr = _c(rows, np.int64) if rows is not None else None
    nr = len(rr) if rr is not None else int(cu[-1])
    out = np.zeros((nr, H, D), dtype=np.float64)
    lib.oracle_prefill_biased(_ptr(out), _ptr(q), _ptr(k), _ptr(v), _ptr(cu), len(cu) - 1, H, D, int(window),
                              int(causal), float(scale), int(dtype), _ptr(rb), (rb.shape[1] + 1) // 2, _ptr(rr), nr,
                              int(nthreads or default_threads()))
    return out


def paged_prefill(q, k_cache, v_cache, block_tables, cu_seqlens_q, context_lens, window, causal, scale, block_size,
                  dtype, rel_bias=None, rows=None, nthreads=None) -> np.ndarray:
    """Prefill of each sequence's last Lq tokens against its ctx paged keys:
    query row r at key position ctx - Lq + r.  [T or len(rows), H, D] double."""
    lib = _load()
    q = _c(q); kc = _c(k_cache); vc = _c(v_cache)
    bt = _c(block_tables, np.int32)
    cu = _c(cu_seqlens_q, np.int32)
    cl = _c(context_lens, np.int32)
    rb = _c(rel_bias, np.float32) if rel_bias is not None else None
    T, H, D = q.shape
    rr = _c(rows, np.int64) if rows is not None else None
    nr = len(rr) if rr is not None else int(cu[-1])
    out = np.zeros((nr, H, D), dtype=np.float64)
    lib.oracle_paged_prefill(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(cu), _ptr(cl), len(cu) - 1, H, D,
                             int(block_size), bt.shape[1], int(window), int(causal), float(scale), _ptr(rb),
                             (rb.shape[1] + 1) // 2 if rb is not None else 0, int(dtype), _ptr(rr), nr,
                             int(nthreads or default_threads()))
    return out


def reshape_and_cache(k_cache, v_cache, key, value, slot_mapping, block_size) -> None:
    """In-place scatter of key/value [T, H, D] rows into the caches."""
    lib = _load()
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    key = _c(key); value = _c(value)
    sm = _c(slot_mapping, np.int64)
    T, H, D = key.shape
    lib.oracle_reshape_and_cache(_ptr(k_cache), _ptr(v_cache), _ptr(key), _ptr(value), _ptr(sm), T, H, D,
                                 int(block_size), key.itemsize)
