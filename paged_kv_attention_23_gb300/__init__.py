"""paged_kv_attention_23_gb300 — Python binding of libpka.so (sm_103a).

A thin ctypes layer over the C ABI declared in ``include/pka.h``: it turns
torch tensors into device pointers, sizes and dtype codes, passes the current
CUDA stream, and raises on a non-OK status.  Every step of the computation
runs in the library's CUDA kernels; there is no other code path, and calling
any operation without the built library (or without a GPU) raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = ["PkaError", "load", "build", "lib_path", "reshape_and_cache", "paged_attn_decode",
           "paged_attn_decode_t5bias", "paged_attn_decode_multi", "chunked_prefill", "prefill_biased",
           "paged_prefill",
           "paged_attn_decode_workspace_size", "swa_prefill", "DecodeWorkspace", "DTYPE_CODE",
           "DEVCHK_BLOCK_ID", "DEVCHK_CONTEXT_LEN", "DEVCHK_SLOT", "DEVCHK_TIMEOUT", "DEVCHK_CU_SEQLENS",
           "EXPORTED_SYMBOLS"]

_PKG = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(_PKG, "libpka.so")

PKA_OK, PKA_ERR_INVALID_ARG, PKA_ERR_UNSUPPORTED, PKA_ERR_CUDA, PKA_ERR_WORKSPACE = range(5)
DEVCHK_BLOCK_ID, DEVCHK_CONTEXT_LEN, DEVCHK_SLOT, DEVCHK_TIMEOUT, DEVCHK_CU_SEQLENS = 0x1, 0x2, 0x4, 0x8, 0x10

EXPORTED_SYMBOLS = ("pka_status_string", "pka_version", "pka_reshape_and_cache",
                    "pka_paged_attn_decode_workspace_size", "pka_paged_attn_decode",
                    "pka_paged_attn_decode_noalloc", "pka_paged_attn_decode_t5bias",
                    "pka_paged_attn_decode_multi", "pka_swa_prefill", "pka_chunked_prefill", "pka_prefill_biased",
                    "pka_paged_prefill")


class DecodeProblem(ctypes.Structure):
    """The C struct pka_decode_problem (one problem of pka_paged_attn_decode_multi)."""
    _fields_ = [("out", ctypes.c_void_p), ("q", ctypes.c_void_p), ("k_cache", ctypes.c_void_p),
                ("v_cache", ctypes.c_void_p), ("block_tables", ctypes.c_void_p), ("context_lens", ctypes.c_void_p),
                ("attn_bias", ctypes.c_void_p), ("bias_table", ctypes.c_void_p), ("num_buckets", ctypes.c_int),
                ("sliding_window", ctypes.c_int), ("scale", ctypes.c_float), ("num_seqs", ctypes.c_int),
                ("max_blocks_per_seq", ctypes.c_int), ("bias_row_stride", ctypes.c_int),
                ("num_blocks", ctypes.c_int), ("max_context_len", ctypes.c_int),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("key_new", ctypes.c_void_p), ("value_new", ctypes.c_void_p)]

_lib = None
_lock = threading.Lock()


class PkaError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn}: {msg} ({code})")
        self.code = code


def build(force: bool = False, verbose: bool = False) -> str:
    from . import buildlib
    return buildlib.build(force=force, verbose=verbose)


def load():
    """Load libpka.so (built in-tree by ``build()``); raise if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(lib_path):
            raise RuntimeError(f"libpka.so not built at {lib_path}; run paged_kv_attention_23_gb300.build()")
        lib = ctypes.CDLL(lib_path)
        P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.pka_status_string.argtypes = [I]
        lib.pka_status_string.restype = ctypes.c_char_p
        lib.pka_version.argtypes = []
        lib.pka_version.restype = I
        lib.pka_reshape_and_cache.argtypes = [P, P, P, P, P, I, I, I, I, I, I, P, P]
        lib.pka_reshape_and_cache.restype = I
        lib.pka_paged_attn_decode_workspace_size.argtypes = [I, I, I, I, I]
        lib.pka_paged_attn_decode_workspace_size.restype = ctypes.c_size_t
        lib.pka_paged_attn_decode.argtypes = [P, P, P, P, P, P, P, I, F, I, I, I, I, I, I, I, I, I, P,
                                              ctypes.c_size_t, P, P]
        lib.pka_paged_attn_decode.restype = I
        lib.pka_paged_attn_decode_t5bias.argtypes = [P, P, P, P, P, P, P, I, I, F, I, I, I, I, I, I, I, I, P,
                                                     ctypes.c_size_t, P, P]
        lib.pka_paged_attn_decode_t5bias.restype = I
        lib.pka_paged_attn_decode_multi.argtypes = [ctypes.POINTER(DecodeProblem), I, I, I, I, I, P, P]
        lib.pka_paged_attn_decode_multi.restype = I
        lib.pka_swa_prefill.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, F, I, P, P]
        lib.pka_swa_prefill.restype = I
        lib.pka_prefill_biased.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, P, I, F, I, P, P]
        lib.pka_prefill_biased.restype = I
        lib.pka_paged_prefill.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, P, I, F, I, P, P]
        lib.pka_paged_prefill.restype = I
        lib.pka_chunked_prefill.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, F, I, P, P]
        lib.pka_chunked_prefill.restype = I
        _lib = lib
        return lib


def _torch():
    import torch
    return torch


_DTYPES = None


def _dtype_code(t) -> int:
    global _DTYPES
    if _DTYPES is None:
        torch = _torch()
        _DTYPES = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
    return _DTYPES[t.dtype]


DTYPE_CODE = {"f32": 0, "f16": 1, "bf16": 2}


def _ptr(t):
    """Device address of a tensor (an int, which ctypes passes as void *), or None."""
    return None if t is None else t.data_ptr()


_raw_stream = None


def _stream(stream):
    """The cudaStream_t to launch on: the given torch stream, else torch's
    current stream on the current device."""
    global _raw_stream
    torch = _torch()
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is None:
        # the raw handle of the current stream without building a Stream object
        # (where the installed torch has the call), else through current_stream
        _raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None) or \
            (lambda idx: torch.cuda.current_stream(idx).cuda_stream)
    return _raw_stream(torch.cuda.current_device())


def _check(fn: str, code: int):
    if code != PKA_OK:
        raise PkaError(fn, code, load().pka_status_string(code).decode())


def _need(t, name, dtype=None, ndim=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")


# ---------------------------------------------------------------------------
def reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, status=None, stream=None):
    """Scatter key/value [T, H, D] into the caches [num_blocks, H, bs, D]
    at slot_mapping (int64 [T]; negative = skip)."""
    torch = _torch()
    for n, t in (("key", key), ("value", value), ("k_cache", k_cache), ("v_cache", v_cache)):
        _need(t, n, ndim=3 if n in ("key", "value") else 4)
    _need(slot_mapping, "slot_mapping", torch.int64, 1)
    T, H, D = key.shape
    nb, _, bs, _ = k_cache.shape
    lib = load()
    _check("pka_reshape_and_cache",
           lib.pka_reshape_and_cache(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping),
                                     T, H, D, bs, nb, _dtype_code(key), _ptr(status), _stream(stream)))


def paged_attn_decode_workspace_size(num_seqs, num_heads, head_dim, max_context_len, sliding_window=-1) -> int:
    return int(load().pka_paged_attn_decode_workspace_size(num_seqs, num_heads, head_dim, max_context_len,
                                                           sliding_window))


class DecodeWorkspace:
    """A zero-filled device buffer for ``paged_attn_decode``, grown on demand.
    The kernels leave its counter region zero after every call, so it is
    reused without clearing; share one only between calls on one stream."""

    def __init__(self, device=None):
        self.device = device
        self.buf = None

    def get(self, nbytes: int):
        torch = _torch()
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=self.device or "cuda")
        return self.buf


_default_ws = {}


def paged_attn_decode(out, q, k_cache, v_cache, block_tables, context_lens, attn_bias=None, sliding_window=-1,
                      scale=None, max_context_len=None, workspace=None, status=None, stream=None):
    """out[s,h,:] = softmax(scale * (q.K^T + A)) V over each sequence's paged
    keys [max(0, ctx - W), ctx).  ``max_context_len`` defaults to the block
    table's capacity (no device sync); ``workspace`` defaults to a cached
    zero-filled buffer per device."""
    torch = _torch()
    _need(out, "out", ndim=3); _need(q, "q", ndim=3)
    _need(k_cache, "k_cache", ndim=4); _need(v_cache, "v_cache", ndim=4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    if attn_bias is not None:
        _need(attn_bias, "attn_bias", torch.float32, 3)
    S, H, D = q.shape
    nb, _, bs, _ = k_cache.shape
    mbps = block_tables.shape[1]
    stride = attn_bias.shape[2] if attn_bias is not None else 0
    if max_context_len is None:
        max_context_len = mbps * bs if attn_bias is None else min(mbps * bs, stride)
    if scale is None:
        scale = D ** -0.5
    lib = load()
    need = int(lib.pka_paged_attn_decode_workspace_size(S, H, D, int(max_context_len), int(sliding_window)))
    if workspace is None:
        dev = q.device.index if q.device.index is not None else torch.cuda.current_device()
        workspace = _default_ws.setdefault(dev, DecodeWorkspace(q.device)).get(need)
    _check("pka_paged_attn_decode",
           lib.pka_paged_attn_decode(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                     _ptr(context_lens), _ptr(attn_bias), int(sliding_window), float(scale), bs, S,
                                     H, D, mbps, stride, nb, int(max_context_len), _dtype_code(q), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _ptr(status), _stream(stream)))
    return out


def paged_attn_decode_t5bias(out, q, k_cache, v_cache, block_tables, context_lens, bias_table, sliding_window=-1,
                             scale=None, max_context_len=None, workspace=None, status=None, stream=None):
    """Paged decode with the T5 relative-position bias computed in the kernel:
    A[s,h,j] = bias_table[h, min(ctx_s - 1 - j, num_buckets - 1)]."""
    torch = _torch()
    _need(out, "out", ndim=3); _need(q, "q", ndim=3)
    _need(k_cache, "k_cache", ndim=4); _need(v_cache, "v_cache", ndim=4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(context_lens, "context_lens", torch.int32, 1)
    _need(bias_table, "bias_table", torch.float32, 2)
    S, H, D = q.shape
    nb, _, bs, _ = k_cache.shape
    mbps = block_tables.shape[1]
    if max_context_len is None:
        max_context_len = mbps * bs
    if scale is None:
        scale = D ** -0.5
    lib = load()
    need = int(lib.pka_paged_attn_decode_workspace_size(S, H, D, int(max_context_len), int(sliding_window)))
    if workspace is None:
        dev = q.device.index if q.device.index is not None else torch.cuda.current_device()
        workspace = _default_ws.setdefault(dev, DecodeWorkspace(q.device)).get(need)
    _check("pka_paged_attn_decode_t5bias",
           lib.pka_paged_attn_decode_t5bias(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                            _ptr(context_lens), _ptr(bias_table), bias_table.shape[1],
                                            int(sliding_window), float(scale), bs, S, H, D, mbps, nb,
                                            int(max_context_len), _dtype_code(q), _ptr(workspace),
                                            workspace.numel() * workspace.element_size(), _ptr(status),
                                            _stream(stream)))
    return out


def paged_attn_decode_multi(problems, status=None, stream=None):
    """Several paged decodes in one launch (at most two: an encoder-decoder
    step's self- and cross-attention).  ``problems`` is a sequence of dicts
    with the keyword arguments of ``paged_attn_decode`` — out, q, k_cache,
    v_cache, block_tables, context_lens and optionally attn_bias or
    bias_table, sliding_window, scale, max_context_len, workspace — plus
    optionally key_new / value_new [S, H, D]: the newest token's K/V, written
    to the cache at position ctx-1 and attended in the same launch.  All
    share num_heads, head_dim, block size and dtype; each gets its own
    workspace."""
    torch = _torch()
    lib = load()
    arr = (DecodeProblem * max(1, len(problems)))()
    keep = []
    H = D = bs = dt = None
    for i, pr in enumerate(problems):
        out, q, kc, vc = pr["out"], pr["q"], pr["k_cache"], pr["v_cache"]
        bt, cl = pr["block_tables"], pr["context_lens"]
        bias, table = pr.get("attn_bias"), pr.get("bias_table")
        _need(out, "out", ndim=3); _need(q, "q", ndim=3)
        _need(kc, "k_cache", ndim=4); _need(vc, "v_cache", ndim=4)
        _need(bt, "block_tables", torch.int32, 2)
        _need(cl, "context_lens", torch.int32, 1)
        if bias is not None:
            _need(bias, "attn_bias", torch.float32, 3)
        if table is not None:
            _need(table, "bias_table", torch.float32, 2)
        S, h, d = q.shape
        nb, _, b, _ = kc.shape
        if H is not None and (h, d, b, _dtype_code(q)) != (H, D, bs, dt):
            raise ValueError("paged_attn_decode_multi: problems must share num_heads, head_dim, block size and dtype")
        H, D, bs, dt = h, d, b, _dtype_code(q)
        mbps = bt.shape[1]
        stride = bias.shape[2] if bias is not None else 0
        w = int(pr.get("sliding_window", -1))
        mcl = pr.get("max_context_len")
        if mcl is None:
            mcl = mbps * bs if bias is None else min(mbps * bs, stride)
        scale = pr.get("scale")
        if scale is None:
            scale = D ** -0.5
        need = int(lib.pka_paged_attn_decode_workspace_size(S, H, D, int(mcl), w))
        ws = pr.get("workspace")
        if ws is None:
            dev = q.device.index if q.device.index is not None else torch.cuda.current_device()
            ws = _default_ws.setdefault((dev, "multi", i), DecodeWorkspace(q.device)).get(need)
        keep.append(ws)
        kn, vn = pr.get("key_new"), pr.get("value_new")
        if kn is not None or vn is not None:
            _need(kn, "key_new", q.dtype, 3); _need(vn, "value_new", q.dtype, 3)
        arr[i] = DecodeProblem(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(cl), _ptr(bias), _ptr(table),
                               table.shape[1] if table is not None else 0, w, float(scale), S, mbps, stride, nb,
                               int(mcl), _ptr(ws), ws.numel() * ws.element_size(), _ptr(kn), _ptr(vn))
    if not problems:
        raise ValueError("paged_attn_decode_multi needs at least one problem")
    _check("pka_paged_attn_decode_multi",
           lib.pka_paged_attn_decode_multi(arr, len(problems), bs, H, D, dt, _ptr(status), _stream(stream)))
    return [pr["out"] for pr in problems]


def swa_prefill(out, q, k, v, cu_seqlens, max_seqlen, window=-1, causal=0, scale=None, status=None, stream=None):
    """Packed varlen prefill with full / causal / sliding-window (|i-j| < W)
    masks; q/k/v/out [T, H, 64 or 128] bf16 or f16 (one dtype), cu_seqlens int32 [B+1]."""
    torch = _torch()
    for n, t in (("out", out), ("q", q), ("k", k), ("v", v)):
        _need(t, n, ndim=3)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    T, H, D = q.shape
    if scale is None:
        scale = D ** -0.5
    lib = load()
    _check("pka_swa_prefill",
           lib.pka_swa_prefill(_ptr(out), _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), cu_seqlens.numel() - 1, T,
                               int(max_seqlen), H, D, int(window), int(causal), float(scale), _dtype_code(q),
                               _ptr(status), _stream(stream)))
    return out


def chunked_prefill(out, q, k, v, cu_seqlens, max_seqlen, chunk, causal=1, scale=None, status=None, stream=None):
    """Packed varlen prefill with chunked local attention: each token sees the
    keys of its own chunk of ``chunk`` positions (causal: up to itself)."""
    torch = _torch()
    for n, t in (("out", out), ("q", q), ("k", k), ("v", v)):
        _need(t, n, ndim=3)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    T, H, D = q.shape
    if scale is None:
        scale = D ** -0.5
    lib = load()
    _check("pka_chunked_prefill",
           lib.pka_chunked_prefill(_ptr(out), _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), cu_seqlens.numel() - 1,
                                   T, int(max_seqlen), H, D, int(chunk), int(causal), float(scale), _dtype_code(q),
                                   _ptr(status), _stream(stream)))
    return out


def prefill_biased(out, q, k, v, cu_seqlens, max_seqlen, rel_bias, window=-1, causal=0, scale=None, status=None,
                   stream=None):
    """``swa_prefill`` with the relative-position bias rel_bias [H, 2B-1]:
    A[h, r, c] = rel_bias[h, B-1 + clamp(r - c, -(B-1), B-1)] inside the scores."""
    torch = _torch()
    for n, t in (("out", out), ("q", q), ("k", k), ("v", v)):
        _need(t, n, ndim=3)
    _need(cu_seqlens, "cu_seqlens", torch.int32, 1)
    _need(rel_bias, "rel_bias", torch.float32, 2)
    T, H, D = q.shape
    if rel_bias.shape[0] != H or rel_bias.shape[1] % 2 != 1:
        raise ValueError("rel_bias must be [num_heads, 2 * num_buckets - 1]")
    if scale is None:
        scale = D ** -0.5
    lib = load()
    _check("pka_prefill_biased",
           lib.pka_prefill_biased(_ptr(out), _ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), cu_seqlens.numel() - 1, T,
                                  int(max_seqlen), H, D, int(window), int(causal), _ptr(rel_bias),
                                  (rel_bias.shape[1] + 1) // 2, float(scale), _dtype_code(q), _ptr(status),
                                  _stream(stream)))
    return out


def paged_prefill(out, q, k_cache, v_cache, block_tables, cu_seqlens_q, context_lens, max_query_len, window=-1,
                  causal=1, rel_bias=None, scale=None, status=None, stream=None):
    """Prefill of each sequence's last Lq tokens (q/out [T, H, 64], packed by
    cu_seqlens_q) against its context_lens[s] keys in the paged caches
    [num_blocks, H, 16, 64] through block_tables; query row r sits at key
    position ctx - Lq + r.  Optional relative-position bias as in
    ``prefill_biased``."""
    torch = _torch()
    _need(out, "out", ndim=3); _need(q, "q", ndim=3)
    _need(k_cache, "k_cache", ndim=4); _need(v_cache, "v_cache", ndim=4)
    _need(block_tables, "block_tables", torch.int32, 2)
    _need(cu_seqlens_q, "cu_seqlens_q", torch.int32, 1)
    _need(context_lens, "context_lens", torch.int32, 1)
    nb_buckets = 0
    if rel_bias is not None:
        _need(rel_bias, "rel_bias", torch.float32, 2)
        if rel_bias.shape[1] % 2 != 1:
            raise ValueError("rel_bias must be [num_heads, 2 * num_buckets - 1]")
        nb_buckets = (rel_bias.shape[1] + 1) // 2
    T, H, D = q.shape
    nb, _, bs, _ = k_cache.shape
    if scale is None:
        scale = D ** -0.5
    lib = load()
    _check("pka_paged_prefill",
           lib.pka_paged_prefill(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                 _ptr(cu_seqlens_q), _ptr(context_lens), cu_seqlens_q.numel() - 1, T,
                                 int(max_query_len), H, D, bs, block_tables.shape[1], nb, int(window), int(causal),
                                 _ptr(rel_bias), nb_buckets, float(scale), _dtype_code(q), _ptr(status),
                                 _stream(stream)))
    return out
