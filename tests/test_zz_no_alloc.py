"""pka_paged_attn_decode_noalloc: the decode entry point for callers that
cannot allocate device memory (a host framework that owns all device memory
through its own pool, or a latency-critical loop where cudaMalloc could stall
the device).  It takes no workspace and uses one fixed scratch array inside
the library instead.

The GPU test calls it through the C ABI twice in a row and checks each result
against pka_paged_attn_decode given its own workspace: the same kernel runs
with the same split of the work, so the outputs must be identical bit for
bit (and so within the tolerance the other decode tests use).  This file is
named to be collected last, so a run that stops at the first failure has run
every other test before it."""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_attention_23_gb300 as pka
import synth
from helpers import TOL, GpuDecode, max_err, to_f64

NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024     # PKA_NOALLOC_SCRATCH_BYTES in include/pka.h


def _noalloc(lib):
    f = lib.pka_paged_attn_decode_noalloc
    P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    f.argtypes = [P, P, P, P, P, P, P, I, F, I, I, I, I, I, I, I, I, I, P, P]
    f.restype = I
    return f


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call_noalloc(lib, g, out):
    c = g.case
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return _noalloc(lib)(_ptr(out), _ptr(g.q), _ptr(g.k_cache), _ptr(g.v_cache), _ptr(g.block_tables),
                         _ptr(g.context_lens), _ptr(g.bias), c.window, c.scale, c.block_size, c.num_seqs,
                         c.num_heads, c.head_dim, c.max_blocks_per_seq, c.bias_row_stride, c.num_blocks,
                         c.max_context_len, c.dtype, _ptr(g.status), stream)


@pytest.mark.gpu
def test_noalloc_decode_matches_workspace_decode_on_two_calls(cuda_lib):
    lib = cuda_lib.load()
    # T5-small-shaped (bias, up to 8 partitions) and T5-large-shaped (bias,
    # up to 16 partitions, ~17 MiB of scratch): both fit the fixed array
    for n in (2, 3):
        case = synth.decode_workload(n)
        need = cuda_lib.paged_attn_decode_workspace_size(case.num_seqs, case.num_heads, case.head_dim,
                                                         case.max_context_len, case.window)
        assert need <= NOALLOC_SCRATCH_BYTES
        g = GpuDecode(case, cuda_lib)
        ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
        ref_t = g.run(workspace=ws).clone()
        ref = to_f64(ref_t, case.dtype)
        for call in range(2):
            out = torch.full_like(g.out, float("nan"))
            assert _call_noalloc(lib, g, out) == cuda_lib.PKA_OK
            torch.cuda.synchronize()
            got = to_f64(out, case.dtype)
            assert np.isfinite(got).all(), f"workload {n} call {call}"
            err = max_err(got, ref)
            assert err <= TOL[case.dtype], f"workload {n} call {call}: max abs diff {err:.3g}"
            assert torch.equal(out.view(torch.uint8), ref_t.view(torch.uint8)), f"workload {n} call {call}"
        assert int(g.status.item()) == 0


def test_noalloc_rejects_a_call_larger_than_its_scratch():
    """A long-context shape needs more scratch than the fixed array holds: the
    call is refused on the host before anything is enqueued (no GPU needed;
    the pointers are never dereferenced)."""
    pka.build()
    lib = pka.load()
    need = lib.pka_paged_attn_decode_workspace_size(512, 16, 128, 8192, -1)
    assert need > NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(1 << 20)
    rc = _noalloc(lib)(fake, fake, fake, fake, fake, fake, None, -1, 0.088, 16, 512, 16, 128, 512, 0, 1000,
                       8192, 1, None, None)
    assert rc == pka.PKA_ERR_WORKSPACE
    # argument errors answer as the workspace entry point does
    rc = _noalloc(lib)(fake, fake, fake, fake, fake, fake, None, 0, 0.088, 16, 2, 16, 128, 512, 0, 1000, 8192, 1,
                       None, None)
    assert rc == pka.PKA_ERR_INVALID_ARG
