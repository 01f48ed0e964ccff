"""Seeded synthetic inputs for paged-KV attention, shared by the tests, the
oracle checks and the benchmark.

This module only draws and lays out inputs: context lengths, block
permutations, per-token K/V, queries and the materialised bias.  It holds none
of the attention arithmetic, so neither the CUDA path nor the oracle can
borrow a step of the method from here.

Workload recipes (one per named workload) follow the shapes of the pages:

* "PagedAttention: Support custom attention bias for T5 model (1/2)" — a fully
  materialised fp32 bias A padded to the maximum sequence length, built here
  from a T5 relative-position table whose distances beyond 128 reuse the last
  entry (the reviewer comment on T5-large's maximum relative distance).
* "Add Encoder-decoder model support and T5 Model support" — decoder
  self-attention and encoder cross-attention read two separate block tables.
* "[V1] Add sliding window support to Flex Attention backend" — encoder-only
  prefill with layers alternating full / window-64 / window-64.

Random draws happen in a fixed order per workload (context lengths, block
permutation, queries, per-token K/V, bias) from ``numpy.random.default_rng``
for everything small, and from a seeded ``torch.Generator`` on the target
device for the multi-GB token arrays of the large decode workloads.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

# dtype codes of the C ABI (pka_dtype) and of the oracle: 0 = f32, 1 = f16, 2 = bf16
F32, F16, BF16 = 0, 1, 2
DTYPE_NAMES = {F32: "f32", F16: "f16", BF16: "bf16"}
ELT_BYTES = {F32: 4, F16: 2, BF16: 2}
NP_STORAGE = {F32: np.float32, F16: np.float16, BF16: np.uint16}

T5_MAX_DISTANCE = 128  # distances beyond this reuse the last table entry


# --------------------------------------------------------------------------
# storage encodings (fp32 draws -> stored bytes)
# --------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round to nearest, ties to even) and return the raw
    16-bit patterns.  NaN stays NaN (quiet)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        r = r.copy()
        r[nan] = (((u[nan] >> 16) | 0x40).astype(np.uint16))
    return r


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def encode(x: np.ndarray, dtype: int) -> np.ndarray:
    """fp32 values -> the array that holds their stored representation."""
    if dtype == F32:
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == F16:
        return np.ascontiguousarray(x.astype(np.float16))
    if dtype == BF16:
        return f32_to_bf16_bits(x)
    raise ValueError(dtype)


def decode_to_f32(a: np.ndarray, dtype: int) -> np.ndarray:
    """Stored representation -> fp32 values (exact for every dtype here)."""
    if dtype == F32:
        return np.asarray(a, dtype=np.float32)
    if dtype == F16:
        return np.asarray(a, dtype=np.float16).astype(np.float32)
    if dtype == BF16:
        return bf16_bits_to_f32(a)
    raise ValueError(dtype)


def log_uniform_int(rng: np.random.Generator, lo: int, hi: int, n: int) -> np.ndarray:
    """floor(exp(U(ln lo, ln(hi+1)))) clipped to [lo, hi]."""
    v = np.floor(np.exp(rng.uniform(math.log(lo), math.log(hi + 1), size=n)))
    return np.clip(v, lo, hi).astype(np.int32)


def t5_bucket(distance: np.ndarray) -> np.ndarray:
    """Table column for a T5-style relative distance: distances beyond the
    maximum reuse the last column."""
    return np.minimum(distance, T5_MAX_DISTANCE)


# --------------------------------------------------------------------------
# decode workloads
# --------------------------------------------------------------------------
@dataclasses.dataclass
class DecodeCase:
    """One paged decode call's inputs, with host copies of everything.

    Token arrays ``key``/``value`` are [T, H, D] in storage encoding, token t of
    sequence s at position j sitting at row ``tok_offsets[s] + j``; the cache is
    meant to be filled from them through ``slot_mapping`` (one slot per token).
    ``q`` is [S, H, D]; ``bias`` is fp32 [S, H, bias_row_stride] or None.
    """
    name: str
    dtype: int
    num_seqs: int
    num_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    context_lens: np.ndarray            # int32 [S]
    block_tables: np.ndarray            # int32 [S, max_blocks_per_seq]
    slot_mapping: np.ndarray            # int64 [T]
    tok_offsets: np.ndarray             # int64 [S+1]
    q: np.ndarray                       # storage [S, H, D]
    key: Optional[np.ndarray]           # storage [T, H, D] (None when generated on device)
    value: Optional[np.ndarray]
    bias: Optional[np.ndarray]          # f32 [S, H, stride] or None
    window: int
    scale: float
    device_kv: object = None            # (key, value) torch tensors when drawn on device
    bias_table: Optional[np.ndarray] = None  # f32 [H, 129] when the bias is T5-style

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    @property
    def bias_row_stride(self) -> int:
        return int(self.bias.shape[2]) if self.bias is not None else 0

    @property
    def num_tokens(self) -> int:
        return int(self.tok_offsets[-1])

    def visible(self) -> np.ndarray:
        """Number of keys each sequence attends to (window applied)."""
        c = self.context_lens.astype(np.int64)
        return np.minimum(c, self.window) if self.window > 0 else c


def _paged_layout(rng, context_lens, block_size, pool_blocks=None, max_blocks_per_seq=None):
    """Random physical placement: every sequence's logical blocks take the next
    entries of one seeded permutation of the pool.  Unused table entries = -1."""
    S = len(context_lens)
    nblk = (context_lens.astype(np.int64) + block_size - 1) // block_size
    need = int(nblk.sum())
    pool = need if pool_blocks is None else pool_blocks
    assert pool >= need, (pool, need)
    perm = rng.permutation(pool).astype(np.int32)
    mbps = max_blocks_per_seq or max(1, int(nblk.max()) if S else 1)
    bt = np.full((S, mbps), -1, dtype=np.int32)
    pos = 0
    for s in range(S):
        n = int(nblk[s])
        bt[s, :n] = perm[pos:pos + n]
        pos += n
    tok_off = np.zeros(S + 1, dtype=np.int64)
    tok_off[1:] = np.cumsum(context_lens.astype(np.int64))
    T = int(tok_off[-1])
    slot = np.empty(T, dtype=np.int64)
    for s in range(S):
        j = np.arange(int(context_lens[s]), dtype=np.int64)
        slot[tok_off[s]:tok_off[s + 1]] = bt[s, j // block_size].astype(np.int64) * block_size + j % block_size
    return pool, bt, slot, tok_off


def t5_bias(table: np.ndarray, context_lens: np.ndarray, stride: int, pad_value: float = 0.0) -> np.ndarray:
    """Materialise A[s, h, j] = table[h, bucket(ctx_s - 1 - j)] for j < ctx_s,
    ``pad_value`` past the context."""
    H = table.shape[0]
    S = len(context_lens)
    A = np.full((S, H, stride), pad_value, dtype=np.float32)
    for s in range(S):
        c = int(context_lens[s])
        d = (c - 1) - np.arange(c)
        A[s, :, :c] = table[:, t5_bucket(d)]
    return A


def make_decode_case(name: str, seed: int, dtype: int, num_seqs: int, num_heads: int, head_dim: int,
                     context_lens: np.ndarray = None, ctx_range=(1, 64), log_uniform=False,
                     block_size: int = 16, pool_blocks: Optional[int] = None,
                     bias: str = "none", bias_stride: Optional[int] = None, bias_std: float = 1.0,
                     bias_pad: float = 0.0, window: int = -1, scale: Optional[float] = None,
                     device: Optional[str] = None, max_blocks_per_seq: Optional[int] = None,
                     rng: Optional[np.random.Generator] = None) -> DecodeCase:
    """Draw one decode case.  Draw order: context lengths, block permutation,
    q, per-token K and V, bias.  ``bias`` is "none", "gauss" (N(0, bias_std^2)
    per entry) or "t5" (materialised from a N(0,1) table [H, 129]).
    ``device``: None draws K/V with numpy on the host; "cuda" draws them with a
    seeded torch generator on the GPU and keeps them there (host copies None)."""
    rng = rng or np.random.default_rng(seed)
    S, H, D = num_seqs, num_heads, head_dim
    if context_lens is None:
        lo, hi = ctx_range
        context_lens = (log_uniform_int(rng, lo, hi, S) if log_uniform
                        else rng.integers(lo, hi + 1, size=S).astype(np.int32))
    context_lens = np.asarray(context_lens, dtype=np.int32)
    pool, bt, slot, tok_off = _paged_layout(rng, context_lens, block_size, pool_blocks, max_blocks_per_seq)
    T = int(tok_off[-1])
    q = encode(rng.standard_normal((S, H, D), dtype=np.float32), dtype)
    key = value = None
    device_kv = None
    if device is None:
        key = encode(rng.standard_normal((T, H, D), dtype=np.float32), dtype)
        value = encode(rng.standard_normal((T, H, D), dtype=np.float32), dtype)
    else:
        device_kv = draw_device_tokens(seed, T, H, D, dtype, device)
    stride = bias_stride if bias_stride is not None else (int(context_lens.max()) if S else 0)
    A = None
    table = None
    if bias == "gauss":
        A = (rng.standard_normal((S, H, stride), dtype=np.float32) * np.float32(bias_std)).astype(np.float32)
        for s in range(S):
            A[s, :, int(context_lens[s]):] = bias_pad
    elif bias == "t5":
        table = rng.standard_normal((H, T5_MAX_DISTANCE + 1), dtype=np.float32)
        A = t5_bias(table, context_lens, stride, bias_pad)
    elif bias != "none":
        raise ValueError(bias)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    return DecodeCase(name, dtype, S, H, D, block_size, pool, context_lens, bt, slot, tok_off,
                      q, key, value, A, window, float(scale), device_kv, table)


def draw_device_tokens(seed: int, T: int, H: int, D: int, dtype: int, device: str):
    """Per-token K and V drawn N(0,1) on ``device`` with a seeded torch
    generator, rounded once to the storage dtype."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed * 7919 + 17)
    tdt = {F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}[dtype]
    # chunked draw keeps the fp32 temporaries small
    step = max(1, (1 << 26) // max(1, H * D))
    kk = torch.empty((T, H, D), dtype=tdt, device=device)
    vv = torch.empty((T, H, D), dtype=tdt, device=device)
    for t0 in range(0, T, step):
        t1 = min(T, t0 + step)
        kk[t0:t1] = torch.randn((t1 - t0, H, D), generator=g, device=device, dtype=torch.float32).to(tdt)
        vv[t0:t1] = torch.randn((t1 - t0, H, D), generator=g, device=device, dtype=torch.float32).to(tdt)
    return kk, vv


# --------------------------------------------------------------------------
# named decode workloads
# --------------------------------------------------------------------------
def decode_workload(n: int, device: Optional[str] = None, bias_on: bool = True,
                    num_seqs: Optional[int] = None) -> DecodeCase:
    """The decode workloads by number.

    1: tiny fp32, 4 seqs x 2 heads x 64, ctx U[1,64], 32-block permuted pool,
       Gaussian bias [4,2,64] zero-padded, scale 1/8.
    2: T5-small-shaped decoder self-attention, bf16, 64 seqs x 8 heads x 64,
       ctx U[1,512], T5 bias from a [8,129] table padded to 512, scale 1/8.
    3: T5-large-shaped decoder self-attention, bf16, 256 x 16 x 64, ctx U[1,2048],
       T5 bias [16,129] padded to 2048 (the cross-attention half is
       ``cross_workload``).
    5: long-context fp16, 512 x 16 x 128, ctx log-U[16,8192], causal window
       4096, Gaussian bias N(0, 0.5^2) [512,16,8192] with NaN padding,
       shared permuted pool, scale 1/sqrt(128).
    """
    seed = 1000 + n
    S = num_seqs
    if n == 1:
        return make_decode_case("tiny-f32-decode", seed, F32, S or 4, 2, 64, ctx_range=(1, 64), pool_blocks=32,
                                bias="gauss" if bias_on else "none", bias_stride=64, scale=1 / 8,
                                device=device)
    if n == 2:
        return make_decode_case("t5-small-self-decode", seed, BF16, S or 64, 8, 64, ctx_range=(1, 512),
                                bias="t5" if bias_on else "none", bias_stride=512, scale=1 / 8, device=device)
    if n == 3:
        return make_decode_case("t5-large-self-decode", seed, BF16, S or 256, 16, 64, ctx_range=(1, 2048),
                                bias="t5" if bias_on else "none", bias_stride=2048, scale=1 / 8, device=device)
    if n == 5:
        return make_decode_case("long-ctx-f16-window-decode", seed, F16, S or 512, 16, 128, ctx_range=(16, 8192),
                                log_uniform=True, bias="gauss" if bias_on else "none", bias_stride=8192,
                                bias_std=0.5, bias_pad=float("nan"), window=4096,
                                scale=1 / math.sqrt(128), device=device)
    raise ValueError(n)


def cross_workload(device: Optional[str] = None, num_seqs: Optional[int] = None) -> DecodeCase:
    """Encoder cross-attention decode of the T5-large-shaped step: 256 seqs x
    16 heads x 64, every encoder length 512, its own block table and pool, no
    bias, no window."""
    seed = 1000 + 3 + 100
    S = num_seqs or 256
    return make_decode_case("t5-large-cross-decode", seed, BF16, S, 16, 64,
                            context_lens=np.full(S, 512, dtype=np.int32), bias="none",
                            scale=1 / 8, device=device)


# --------------------------------------------------------------------------
# prefill workloads
# --------------------------------------------------------------------------
@dataclasses.dataclass
class PrefillCase:
    name: str
    dtype: int
    num_heads: int
    head_dim: int
    cu_seqlens: np.ndarray              # int32 [num_seqs+1]
    q: Optional[np.ndarray]             # storage [T, H, D]
    k: Optional[np.ndarray]
    v: Optional[np.ndarray]
    window: int
    causal: int
    scale: float
    device_qkv: object = None
    chunk: int = 0                      # > 0: chunked local attention (window must be -1)
    rel_bias: Optional[np.ndarray] = None   # f32 [H, 2B-1] signed relative-position bias, or None

    @property
    def num_seqs(self) -> int:
        return len(self.cu_seqlens) - 1

    @property
    def num_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def max_seqlen(self) -> int:
        return int(np.diff(self.cu_seqlens).max()) if self.num_seqs else 0

    def visible_pairs(self) -> int:
        """Number of (query, key) pairs the mask keeps, summed over sequences."""
        tot = 0
        W = self.window
        for L in np.diff(self.cu_seqlens).astype(np.int64):
            L = int(L)
            if self.chunk > 0:
                for a in range(0, L, self.chunk):
                    c = min(self.chunk, L - a)
                    tot += c * (c + 1) // 2 if self.causal else c * c
                continue
            if W <= 0:
                tot += L * (L + 1) // 2 if self.causal else L * L
            else:
                w = min(W, L)
                causal_pairs = w * L - w * (w - 1) // 2       # 0 <= i-j < W
                tot += causal_pairs if self.causal else 2 * causal_pairs - L
        return tot


def make_prefill_case(name: str, seed: int, seqlens, num_heads: int, head_dim: int, window: int,
                      causal: int, dtype: int = BF16, scale: Optional[float] = None,
                      device: Optional[str] = None) -> PrefillCase:
    seqlens = np.asarray(seqlens, dtype=np.int64)
    cu = np.zeros(len(seqlens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(seqlens)
    T = int(cu[-1])
    H, D = num_heads, head_dim
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if device is None:
        rng = np.random.default_rng(seed)
        q = encode(rng.standard_normal((T, H, D), dtype=np.float32), dtype)
        k = encode(rng.standard_normal((T, H, D), dtype=np.float32), dtype)
        v = encode(rng.standard_normal((T, H, D), dtype=np.float32), dtype)
        return PrefillCase(name, dtype, H, D, cu, q, k, v, window, causal, float(scale))
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed * 7919 + 29)
    tdt = {F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}[dtype]
    qkv = tuple(torch.randn((T, H, D), generator=g, device=device, dtype=torch.float32).to(tdt)
                for _ in range(3))
    return PrefillCase(name, dtype, H, D, cu, None, None, None, window, causal, float(scale), qkv)


ENCODER_LAYER_WINDOWS = (-1, 64, 64)   # full, sliding 64, sliding 64 (repeating)


def prefill_seqlens(seed: int = 1004, num_seqs: int = 32, lo: int = 128, hi: int = 8192) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi + 1, size=num_seqs).astype(np.int64)


def prefill_workload(layer: int, device: Optional[str] = None, seqlens=None, head_dim: int = 64) -> PrefillCase:
    """Encoder-only bidirectional prefill, bf16, 12 heads x 64, 32 sequences
    with lengths U[128,8192] packed by cu_seqlens.  ``layer`` 0, 1, 2 selects
    the window of the alternating pattern (full, 64, 64) and its own seeded
    q/k/v.  ``head_dim`` 128 gives the same shapes at head dim 128 (scale
    1/sqrt(128))."""
    if seqlens is None:
        seqlens = prefill_seqlens()
    W = ENCODER_LAYER_WINDOWS[layer % 3]
    name = f"encoder-prefill-layer{layer}-w{W}" + ("" if head_dim == 64 else f"-d{head_dim}")
    return make_prefill_case(name, 1004 * 10 + layer, seqlens, 12, head_dim, W, 0, BF16, 1 / math.sqrt(head_dim),
                             device)


CHUNKED_PREFILL_CHUNK = 1024


def chunked_prefill_workload(device: Optional[str] = None, seqlens=None) -> PrefillCase:
    """Chunked local attention (decoder-style, causal within each chunk of
    1024 positions) over the same 32 packed sequences, 12 heads x 64, bf16."""
    if seqlens is None:
        seqlens = prefill_seqlens()
    c = make_prefill_case("chunked-prefill-c1024", 1004 * 10 + 9, seqlens, 12, 64, -1, 1, BF16, 1 / 8, device)
    c.chunk = CHUNKED_PREFILL_CHUNK
    return c


# --------------------------------------------------------------------------
# relative-position bias and prefill against the paged cache
# --------------------------------------------------------------------------
def rel_bias_table(seed: int, num_heads: int, buckets: int = T5_MAX_DISTANCE + 1) -> np.ndarray:
    """A seeded N(0,1) signed relative-position table [H, 2*buckets - 1]:
    column buckets-1+d holds the bias of a query d positions after its key."""
    rng = np.random.default_rng(seed * 131 + 3)
    return rng.standard_normal((num_heads, 2 * buckets - 1), dtype=np.float32)


@dataclasses.dataclass
class PagedPrefillCase:
    """Prefill of each sequence's newest query tokens against its keys in the
    paged cache.  ``cache`` holds the keys/values of all ctx_s positions (token
    arrays, slot mapping, block tables); the queries are the last Lq_s
    positions, packed [Tq, H, D] by ``cu_seqlens_q``."""
    name: str
    cache: DecodeCase
    cu_seqlens_q: np.ndarray            # int32 [S+1]
    q: Optional[np.ndarray]             # storage [Tq, H, D] (None when drawn on device)
    window: int
    causal: int
    scale: float
    rel_bias: Optional[np.ndarray] = None
    device_q: object = None

    @property
    def dtype(self) -> int:
        return self.cache.dtype

    @property
    def num_heads(self) -> int:
        return self.cache.num_heads

    @property
    def head_dim(self) -> int:
        return self.cache.head_dim

    @property
    def num_seqs(self) -> int:
        return len(self.cu_seqlens_q) - 1

    @property
    def num_tokens(self) -> int:
        return int(self.cu_seqlens_q[-1])

    @property
    def query_lens(self) -> np.ndarray:
        return np.diff(self.cu_seqlens_q).astype(np.int64)

    @property
    def max_query_len(self) -> int:
        return int(self.query_lens.max()) if self.num_seqs else 0

    def kept_pairs(self) -> int:
        """(query, key) pairs the mask keeps, summed over sequences."""
        total = 0
        for Lq, ctx in zip(self.query_lens, self.cache.context_lens.astype(np.int64)):
            if Lq == 0 or ctx == 0:
                continue
            p = ctx - Lq + np.arange(Lq)
            lo = np.zeros(Lq, dtype=np.int64)
            hi = np.full(Lq, ctx, dtype=np.int64)
            if self.window > 0:
                lo = np.maximum(lo, p - self.window + 1)
                if not self.causal:
                    hi = np.minimum(hi, p + self.window)
            if self.causal:
                hi = np.minimum(hi, p + 1)
            total += int(np.maximum(hi - lo, 0).sum())
        return total


def make_paged_prefill_case(name: str, seed: int, dtype: int, context_lens, query_lens, num_heads: int,
                            head_dim: int, window: int = -1, causal: int = 1, rel_buckets: int = 0,
                            scale: Optional[float] = None, pool_blocks: Optional[int] = None,
                            max_blocks_per_seq: Optional[int] = None, device: Optional[str] = None,
                            cache: Optional[DecodeCase] = None) -> PagedPrefillCase:
    """Draw the paged keys (or take ``cache``), then the queries of the last
    query_lens[s] positions of each sequence, then the bias table."""
    context_lens = np.asarray(context_lens, dtype=np.int32)
    query_lens = np.asarray(query_lens, dtype=np.int64)
    H, D = num_heads, head_dim
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if cache is None:
        cache = make_decode_case(name, seed, dtype, len(context_lens), H, D, context_lens=context_lens,
                                 pool_blocks=pool_blocks, window=window, scale=scale, device=device,
                                 max_blocks_per_seq=max_blocks_per_seq)
    cu = np.zeros(len(query_lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(query_lens)
    Tq = int(cu[-1])
    q = dq = None
    if device is None:
        q = encode(np.random.default_rng(seed * 31 + 5).standard_normal((Tq, H, D), dtype=np.float32), dtype)
    else:
        import torch
        g = torch.Generator(device=device)
        g.manual_seed(seed * 7919 + 41)
        tdt = {F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}[dtype]
        dq = torch.randn((Tq, H, D), generator=g, device=device, dtype=torch.float32).to(tdt)
    rel = rel_bias_table(seed, H, rel_buckets) if rel_buckets > 0 else None
    return PagedPrefillCase(name, cache, cu, q, window, causal, float(scale), rel, dq)


def t5_encoder_prefill_workload(device: Optional[str] = None, num_seqs: int = 256,
                                enc_len: int = 512) -> PrefillCase:
    """T5-large-shaped encoder self-attention: 256 sequences x 512 tokens
    (the encoder length of the cross-attention decode workload), 16 heads x
    64, bf16, bidirectional, T5 relative-position bias [16, 257] (distance
    capped at 128 either way), scale 1/8."""
    c = make_prefill_case("t5-encoder-prefill", 1004 * 10 + 21, np.full(num_seqs, enc_len), 16, 64, -1, 0, BF16,
                          1 / 8, device)
    c.rel_bias = rel_bias_table(1004 * 10 + 21, 16)
    return c


def t5_paged_prefill_workload(device: Optional[str] = None, num_seqs: Optional[int] = None):
    """A prompt chunk of each sequence of the T5-large-shaped decode workload
    through its block tables: the last Lq_s = min(ctx_s, U[1,256]) positions
    query (a) the decoder self-attention cache (contexts U[1,2048], causal,
    the T5 bias table's non-negative half) and (b) the encoder cross-attention
    cache (encoder length 512, no bias, no mask).  Returns (self, cross)."""
    sc = decode_workload(3, device=device, num_seqs=num_seqs)
    cc = cross_workload(device=device, num_seqs=num_seqs)
    rng = np.random.default_rng(1004 * 10 + 22)
    ql = np.minimum(sc.context_lens, rng.integers(1, 257, size=sc.num_seqs)).astype(np.int64)
    self_case = make_paged_prefill_case("t5-large-paged-prefill-self", 1004 * 10 + 22, BF16, sc.context_lens, ql,
                                        16, 64, -1, 1, T5_MAX_DISTANCE + 1, 1 / 8, device=device, cache=sc)
    cross_case = make_paged_prefill_case("t5-large-paged-prefill-cross", 1004 * 10 + 23, BF16, cc.context_lens,
                                         ql, 16, 64, -1, 0, 0, 1 / 8, device=device, cache=cc)
    # the cross-attention queries are the same prompt tokens
    cross_case.q, cross_case.device_q = self_case.q, self_case.device_q
    return self_case, cross_case
