"""GPU parity of swa_prefill against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest

import oracle
import synth
from helpers import TOL, max_err, to_dev, to_f64, to_host_storage
from synth import BF16

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


def _check(got, ref, what):
    assert np.isfinite(got).all(), what
    err = max_err(got, ref)
    assert err <= TOL[BF16], f"{what}: max abs err {err:.3g}"


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


@pytest.mark.parametrize("layer", [0, 1])
def test_prefill_encoder_workload_sampled(cuda_lib, layer):
    """The encoder workload (32 sequences, lengths U[128, 8192], 12 heads,
    head_dim 64) at full size: layer 0 is full attention, layer 1 window 64;
    the oracle checks every sequence's first/last rows, the rows at the
    128-row tile edge and a seeded random sample."""
    case = synth.prefill_workload(layer, device="cuda")
    got = run_gpu_prefill(cuda_lib, case)
    q, k, v = (to_host_storage(t, BF16) for t in case.device_qkv)
    rows = _sample_rows(case, np.random.default_rng(400 + layer), per_seq=48 if layer == 0 else 400)
    ref = oracle.prefill(q, k, v, case.cu_seqlens, case.window, case.causal, case.scale, BF16, rows=rows)
    _check(to_f64(got[rows], BF16), ref, f"encoder layer {layer}")


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
