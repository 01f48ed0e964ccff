"""The C ABI library loads and exports every symbol include/pka.h declares;
host-side argument checks answer without touching a GPU.  No GPU needed."""
import ctypes
import os
import re

import pytest

import paged_kv_attention_23_gb300 as pka

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    pka.build()
    return pka.load()


def declared_symbols():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            names |= set(re.findall(r"PKA_API\s+[\w\s\*]+?\b(pka_\w+)\s*\(", src))
    return names


def test_header_declares_the_binding_symbols():
    assert declared_symbols() == set(pka.EXPORTED_SYMBOLS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert lib.pka_status_string(0) == b"PKA_OK"
    assert lib.pka_status_string(1) == b"PKA_ERR_INVALID_ARG"
    assert lib.pka_status_string(99) == b"PKA_ERR_UNKNOWN"
    assert lib.pka_version() >= 100


def test_workspace_size_grows_with_work(lib):
    f = lib.pka_paged_attn_decode_workspace_size
    a = f(64, 8, 64, 512, -1)
    assert a > 0
    assert f(128, 8, 64, 512, -1) > a
    assert f(64, 8, 128, 512, -1) > a
    assert f(64, 8, 64, 512, 16) < a          # a window bounds the partitions
    assert f(0, 8, 64, 512, -1) == 0


NULL = None


def _decode(lib, **kw):
    a = dict(out=NULL, q=NULL, kc=NULL, vc=NULL, bt=NULL, cl=NULL, bias=NULL, window=-1, scale=0.125, bs=16,
             S=0, H=2, D=64, mbps=4, stride=0, nb=8, maxctx=64, dt=0, ws=NULL, wsb=0, st=NULL, stream=NULL)
    a.update(kw)
    return lib.pka_paged_attn_decode(a["out"], a["q"], a["kc"], a["vc"], a["bt"], a["cl"], a["bias"], a["window"],
                                     a["scale"], a["bs"], a["S"], a["H"], a["D"], a["mbps"], a["stride"], a["nb"],
                                     a["maxctx"], a["dt"], a["ws"], a["wsb"], a["st"], a["stream"])


def test_decode_argument_checks_need_no_gpu(lib):
    assert _decode(lib) == pka.PKA_OK                               # zero sequences: nothing to do
    assert _decode(lib, window=0) == pka.PKA_ERR_INVALID_ARG
    assert _decode(lib, window=-2) == pka.PKA_ERR_INVALID_ARG
    assert _decode(lib, D=96) == pka.PKA_ERR_UNSUPPORTED
    assert _decode(lib, bs=32) == pka.PKA_ERR_UNSUPPORTED
    assert _decode(lib, dt=7) == pka.PKA_ERR_INVALID_ARG
    assert _decode(lib, maxctx=65) == pka.PKA_ERR_INVALID_ARG      # > mbps * bs
    assert _decode(lib, scale=float("nan")) == pka.PKA_ERR_INVALID_ARG
    fake = ctypes.c_void_p(4096)                                   # never dereferenced: checks fail first
    assert _decode(lib, bias=fake, stride=10) == pka.PKA_ERR_INVALID_ARG   # stride < max_context_len
    assert _decode(lib, S=1) == pka.PKA_ERR_INVALID_ARG            # NULL buffers
    assert _decode(lib, S=1, out=fake, q=fake, kc=fake, vc=fake, bt=fake, cl=fake,
                   ws=NULL) == pka.PKA_ERR_WORKSPACE
    assert _decode(lib, S=1, out=ctypes.c_void_p(4100), q=fake, kc=fake, vc=fake, bt=fake,
                   cl=fake) == pka.PKA_ERR_INVALID_ARG             # misaligned out


def test_reshape_and_prefill_argument_checks_need_no_gpu(lib):
    f = lib.pka_reshape_and_cache
    assert f(NULL, NULL, NULL, NULL, NULL, 0, 2, 64, 16, 8, 2, NULL, NULL) == pka.PKA_OK
    assert f(NULL, NULL, NULL, NULL, NULL, 3, 2, 64, 16, 8, 2, NULL, NULL) == pka.PKA_ERR_INVALID_ARG
    assert f(NULL, NULL, NULL, NULL, NULL, 3, 2, 80, 16, 8, 2, NULL, NULL) == pka.PKA_ERR_UNSUPPORTED
    p = lib.pka_swa_prefill
    assert p(NULL, NULL, NULL, NULL, NULL, 0, 0, 0, 12, 64, -1, 0, 0.125, 2, NULL, NULL) == pka.PKA_OK
    assert p(NULL, NULL, NULL, NULL, NULL, 1, 5, 5, 12, 64, 0, 0, 0.125, 2, NULL, NULL) == pka.PKA_ERR_INVALID_ARG
    assert p(NULL, NULL, NULL, NULL, NULL, 1, 5, 5, 12, 64, -1, 2, 0.125, 2, NULL, NULL) == pka.PKA_ERR_INVALID_ARG
    assert p(NULL, NULL, NULL, NULL, NULL, 1, 5, 5, 12, 64, -1, 0, 0.125, 0, NULL, NULL) == pka.PKA_ERR_UNSUPPORTED
    assert p(NULL, NULL, NULL, NULL, NULL, 1, 5, 5, 12, 64, -1, 0, 0.125, 1, NULL, NULL) == pka.PKA_ERR_INVALID_ARG
    assert p(NULL, NULL, NULL, NULL, NULL, 1, 5, 5, 12, 64, -1, 0, 0.125, 2, NULL, NULL) == pka.PKA_ERR_INVALID_ARG
    # head dim 128 is taken by the packed prefill (NULL buffers: an argument error), 96 is not
    assert p(NULL, NULL, NULL, NULL, NULL, 1, 5, 5, 12, 128, -1, 0, 0.125, 2, NULL, NULL) == pka.PKA_ERR_INVALID_ARG
    assert p(NULL, NULL, NULL, NULL, NULL, 1, 5, 5, 12, 96, -1, 0, 0.125, 2, NULL, NULL) == pka.PKA_ERR_UNSUPPORTED
    c = lib.pka_chunked_prefill
    assert c(NULL, NULL, NULL, NULL, NULL, 1, 5, 5, 12, 128, 64, 0, 0.125, 2, NULL, NULL) == pka.PKA_ERR_INVALID_ARG
    assert c(NULL, NULL, NULL, NULL, NULL, 1, 5, 5, 12, 96, 64, 0, 0.125, 2, NULL, NULL) == pka.PKA_ERR_UNSUPPORTED


def test_product_path_refuses_to_run_without_the_library(monkeypatch, tmp_path):
    """No silent fallback: with the library missing, load() raises."""
    monkeypatch.setattr(pka, "_lib", None)
    monkeypatch.setattr(pka, "lib_path", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError):
        pka.load()


def test_product_package_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "paged_kv_attention_23_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", src, re.M), f
                assert "oracle.c" not in src and "liboracle" not in src, f


def test_decode_problem_struct_matches_the_header(tmp_path):
    """The binding's ctypes mirror of pka_decode_problem has the C layout:
    compile a probe against include/pka.h with the host compiler."""
    import subprocess
    fields = [f[0] for f in pka.DecodeProblem._fields_]
    src = tmp_path / "layout.c"
    body = "".join(f'  printf("%zu ", offsetof(pka_decode_problem, {f}));\n' for f in fields)
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "pka.h"\nint main(void) {\n' + body +
                   '  printf("%zu\\n", sizeof(pka_decode_problem));\n  return 0;\n}\n')
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    got = [int(x) for x in subprocess.check_output([str(exe)]).split()]
    want = [getattr(pka.DecodeProblem, f).offset for f in fields] + [ctypes.sizeof(pka.DecodeProblem)]
    assert got == want


def test_multi_decode_argument_checks_need_no_gpu(lib):
    f = lib.pka_paged_attn_decode_multi
    P = pka.DecodeProblem

    def prob(**kw):
        d = dict(num_seqs=0, sliding_window=-1, scale=0.125, max_blocks_per_seq=4, num_blocks=8, max_context_len=64)
        d.update(kw)
        return P(**d)

    arr = lambda *ps: (P * len(ps))(*ps)
    assert f(None, 1, 16, 2, 64, 2, NULL, NULL) == pka.PKA_ERR_INVALID_ARG
    assert f(arr(prob()), 0, 16, 2, 64, 2, NULL, NULL) == pka.PKA_ERR_INVALID_ARG
    assert f(arr(prob(), prob(), prob()), 3, 16, 2, 64, 2, NULL, NULL) == pka.PKA_ERR_UNSUPPORTED
    assert f(arr(prob(), prob()), 2, 16, 2, 64, 2, NULL, NULL) == pka.PKA_OK        # nothing to do
    assert f(arr(prob(), prob(sliding_window=0)), 2, 16, 2, 64, 2, NULL, NULL) == pka.PKA_ERR_INVALID_ARG
    assert f(arr(prob()), 1, 16, 2, 96, 2, NULL, NULL) == pka.PKA_ERR_UNSUPPORTED
    fake = 4096
    both = dict(attn_bias=fake, bias_row_stride=64, bias_table=fake, num_buckets=4)
    assert f(arr(prob(**both)), 1, 16, 2, 64, 2, NULL, NULL) == pka.PKA_ERR_INVALID_ARG   # bias and table
    assert f(arr(prob(bias_table=fake, num_buckets=2000)), 1, 16, 2, 64, 2, NULL, NULL) == pka.PKA_ERR_UNSUPPORTED
    bufs = dict(out=fake, q=fake, k_cache=fake, v_cache=fake, block_tables=fake, context_lens=fake)
    assert f(arr(prob(num_seqs=1, **bufs)), 1, 16, 2, 64, 2, NULL, NULL) == pka.PKA_ERR_WORKSPACE
    ws, wsb = 1 << 20, 1 << 16
    two = arr(prob(num_seqs=1, workspace=ws, workspace_bytes=wsb, **bufs),
              prob(num_seqs=1, workspace=ws + 512, workspace_bytes=wsb, **dict(bufs, out=fake * 2)))
    assert f(two, 2, 16, 2, 64, 2, NULL, NULL) == pka.PKA_ERR_WORKSPACE                   # workspaces overlap
    two = arr(prob(num_seqs=1, workspace=ws, workspace_bytes=wsb, **bufs),
              prob(num_seqs=1, workspace=ws * 2, workspace_bytes=wsb, **bufs))
    assert f(two, 2, 16, 2, 64, 2, NULL, NULL) == pka.PKA_ERR_INVALID_ARG                 # outputs overlap
    two = arr(prob(num_seqs=1, workspace=ws, workspace_bytes=wsb, bias_table=fake, num_buckets=4, **bufs),
              prob(num_seqs=1, workspace=ws * 2, workspace_bytes=wsb, bias_table=fake * 4, num_buckets=4,
                   **dict(bufs, out=fake * 2)))
    assert f(two, 2, 16, 2, 64, 2, NULL, NULL) == pka.PKA_ERR_UNSUPPORTED                 # two tables


def test_biased_and_paged_prefill_argument_checks_need_no_gpu(lib):
    fake = 4096
    b = lib.pka_prefill_biased
    #        out   q     k     v     cu    S  T  Lmax H   D   W   c  rel  B  scale  dt
    assert b(NULL, NULL, NULL, NULL, NULL, 0, 0, 0, 12, 64, -1, 0, fake, 4, 0.125, 2, NULL, NULL) == pka.PKA_OK
    assert b(NULL, NULL, NULL, NULL, NULL, 0, 0, 0, 12, 64, -1, 0, NULL, 4, 0.125, 2, NULL, NULL) == \
        pka.PKA_ERR_INVALID_ARG                                                    # no table
    assert b(NULL, NULL, NULL, NULL, NULL, 0, 0, 0, 12, 64, -1, 0, fake, 0, 0.125, 2, NULL, NULL) == \
        pka.PKA_ERR_INVALID_ARG                                                    # no buckets
    assert b(NULL, NULL, NULL, NULL, NULL, 1, 5, 5, 12, 64, -1, 0, fake, 4, 0.125, 0, NULL, NULL) == \
        pka.PKA_ERR_UNSUPPORTED                                                    # f32
    assert b(NULL, NULL, NULL, NULL, NULL, 1, 5, 5, 12, 64, -1, 0, fake, 4, 0.125, 1, NULL, NULL) == \
        pka.PKA_ERR_INVALID_ARG                                                    # f16 accepted; NULL buffers
    assert b(NULL, NULL, NULL, NULL, NULL, 1, 5, 5, 12, 64, -1, 0, fake, 4, 0.125, 2, NULL, NULL) == \
        pka.PKA_ERR_INVALID_ARG                                                    # NULL buffers
    assert b(NULL, NULL, NULL, NULL, NULL, 1, 5, 5, 12, 128, -1, 0, fake, 4, 0.125, 2, NULL, NULL) == \
        pka.PKA_ERR_UNSUPPORTED                                                    # head dim 128: bias not built
    p = lib.pka_paged_prefill

    def paged(**kw):
        a = dict(out=NULL, q=NULL, kc=NULL, vc=NULL, bt=NULL, cu=NULL, cl=NULL, S=0, T=0, Lq=0, H=16, D=64, bs=16,
                 mbps=8, nb=32, W=-1, causal=1, rel=NULL, B=0, scale=0.125, dt=2)
        a.update(kw)
        return p(a["out"], a["q"], a["kc"], a["vc"], a["bt"], a["cu"], a["cl"], a["S"], a["T"], a["Lq"], a["H"],
                 a["D"], a["bs"], a["mbps"], a["nb"], a["W"], a["causal"], a["rel"], a["B"], a["scale"], a["dt"],
                 NULL, NULL)

    assert paged() == pka.PKA_OK
    assert paged(bs=32) == pka.PKA_ERR_UNSUPPORTED
    assert paged(D=128) == pka.PKA_ERR_UNSUPPORTED
    assert paged(mbps=0) == pka.PKA_ERR_INVALID_ARG
    assert paged(rel=fake, B=0) == pka.PKA_ERR_INVALID_ARG
    assert paged(W=0) == pka.PKA_ERR_INVALID_ARG
    bufs = dict(out=fake, q=fake, kc=fake, vc=fake, cu=fake, S=1, T=4, Lq=4)
    assert paged(**bufs) == pka.PKA_ERR_INVALID_ARG                                 # no block table
    assert paged(**dict(bufs, bt=fake, cl=fake + 2)) == pka.PKA_ERR_INVALID_ARG     # misaligned lengths


def test_multi_decode_append_needs_both_rows(lib):
    f = lib.pka_paged_attn_decode_multi
    P = pka.DecodeProblem
    fake = 4096
    bufs = dict(out=fake, q=fake, k_cache=fake, v_cache=fake, block_tables=fake, context_lens=fake, num_seqs=1,
                sliding_window=-1, scale=0.125, max_blocks_per_seq=4, num_blocks=8, max_context_len=64)
    one = (P * 1)(P(key_new=fake, **bufs))
    assert f(one, 1, 16, 2, 64, 2, NULL, NULL) == pka.PKA_ERR_INVALID_ARG            # value_new missing
    one = (P * 1)(P(key_new=fake + 8, value_new=fake, **bufs))
    assert f(one, 1, 16, 2, 64, 2, NULL, NULL) == pka.PKA_ERR_INVALID_ARG            # misaligned
