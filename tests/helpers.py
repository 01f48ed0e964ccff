"""Shared test plumbing: move seeded synthetic cases to the GPU, run them
through the library, and run the same bytes through the oracle."""
from __future__ import annotations

import numpy as np

import synth
from synth import BF16, F16, F32

TOL = {F32: 1e-5, F16: 2e-2, BF16: 2e-2}      # max abs error vs the fp64 oracle


def torch_dtype(code):
    import torch
    return {F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}[code]


def to_dev(arr, code, device="cuda"):
    """Storage array (numpy) -> device tensor of the matching torch dtype."""
    import torch
    a = np.ascontiguousarray(arr)
    if code == BF16:
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(a).to(device)


def to_host_storage(t, code):
    """Device tensor -> numpy storage array (bf16 as uint16 bits)."""
    import torch
    t = t.detach().contiguous().cpu()
    if code == BF16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def to_f64(t, code):
    return synth.decode_to_f32(to_host_storage(t, code), code).astype(np.float64)


class GpuDecode:
    """A DecodeCase resident on the GPU, caches filled by the library's
    reshape_and_cache from the token arrays."""

    def __init__(self, case, pka, device="cuda"):
        import torch
        self.case = case
        self.pka = pka
        H, D, bs = case.num_heads, case.head_dim, case.block_size
        tdt = torch_dtype(case.dtype)
        if case.device_kv is not None:
            self.key, self.value = case.device_kv
        else:
            self.key = to_dev(case.key, case.dtype, device)
            self.value = to_dev(case.value, case.dtype, device)
        self.k_cache = torch.zeros((case.num_blocks, H, bs, D), dtype=tdt, device=device)
        self.v_cache = torch.zeros_like(self.k_cache)
        self.slots = torch.from_numpy(case.slot_mapping).to(device)
        pka.reshape_and_cache(self.key, self.value, self.k_cache, self.v_cache, self.slots)
        self.q = to_dev(case.q, case.dtype, device)
        self.block_tables = torch.from_numpy(np.ascontiguousarray(case.block_tables)).to(device)
        self.context_lens = torch.from_numpy(case.context_lens).to(device)
        self.bias = torch.from_numpy(case.bias).to(device) if case.bias is not None else None
        self.out = torch.empty((case.num_seqs, H, D), dtype=tdt, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def run_t5(self, workspace=None):
        """Decode with the bias computed in the kernel from the case's T5 table."""
        import torch
        c = self.case
        tab = torch.from_numpy(c.bias_table).to(self.q.device)
        self.pka.paged_attn_decode_t5bias(self.out, self.q, self.k_cache, self.v_cache, self.block_tables,
                                          self.context_lens, tab, c.window, c.scale,
                                          max_context_len=c.max_context_len, workspace=workspace,
                                          status=self.status)
        return self.out

    def problem(self, mode="bias", workspace=None):
        """This case as one problem of paged_attn_decode_multi; mode is
        "bias" (materialised A), "t5" (in-kernel table) or "none"."""
        import torch
        c = self.case
        pr = dict(out=self.out, q=self.q, k_cache=self.k_cache, v_cache=self.v_cache, block_tables=self.block_tables,
                  context_lens=self.context_lens, sliding_window=c.window, scale=c.scale,
                  max_context_len=c.max_context_len, workspace=workspace)
        if mode == "bias":
            pr["attn_bias"] = self.bias
        elif mode == "t5":
            pr["bias_table"] = torch.from_numpy(c.bias_table).to(self.q.device)
        return pr

    def run(self, bias=True, window=None, workspace=None):
        c = self.case
        self.pka.paged_attn_decode(self.out, self.q, self.k_cache, self.v_cache, self.block_tables,
                                   self.context_lens, self.bias if bias else None,
                                   c.window if window is None else window, c.scale,
                                   max_context_len=c.max_context_len, workspace=workspace, status=self.status)
        return self.out


def oracle_decode_t5(case, pairs=None):
    import oracle
    H, D, bs = case.num_heads, case.head_dim, case.block_size
    shape = (case.num_blocks, H, bs, D)
    kc = np.zeros(shape, dtype=case.key.dtype)
    vc = np.zeros(shape, dtype=case.key.dtype)
    oracle.reshape_and_cache(kc, vc, case.key, case.value, case.slot_mapping, bs)
    return oracle.paged_decode_t5(case.q, kc, vc, case.block_tables, case.context_lens, case.bias_table,
                                  case.window, case.scale, bs, case.dtype, pairs=pairs)


def oracle_decode(case, bias=True, window=None, pairs=None):
    import oracle
    H, D, bs = case.num_heads, case.head_dim, case.block_size
    shape = (case.num_blocks, H, bs, D)
    kc = np.zeros(shape, dtype=case.key.dtype)
    vc = np.zeros(shape, dtype=case.key.dtype)
    oracle.reshape_and_cache(kc, vc, case.key, case.value, case.slot_mapping, bs)
    return oracle.paged_decode(case.q, kc, vc, case.block_tables, case.context_lens,
                               case.bias if bias else None, case.window if window is None else window,
                               case.scale, bs, case.dtype, pairs=pairs)


def max_err(got, ref):
    d = np.abs(got - ref)
    return float(np.nanmax(d)) if d.size else 0.0
