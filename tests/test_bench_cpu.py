"""bench.py's CPU legs, run as a user runs them (no GPU): the reference arm's
JSON line and the oracle leg that the GPU arm starts as a child process."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*argv):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *argv], capture_output=True, text=True,
                       timeout=300, env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert r.returncode == 0, r.stderr[-2000:]
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_reference_arm_line():
    d = _run("--impl", "reference", "--workload", "tiny-decode", "--steps", "2", "--warmup", "3",
             "--ref-seconds", "1")
    assert d["impl"] == "reference"
    assert d["unit"] == "GB/s" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["config"] == {"workload": "tiny-decode"}
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_oracle_leg_line():
    d = _run("--oracle-leg", "--workload", "t5-small-decode", "--cpu-seconds", "1")
    assert d["unit"] == "GB/s" and d["value"] > 0 and d["kind"] == "oracle"
    assert "drawn on the host" in d["sample"]


def _bench():
    sys.path.insert(0, ROOT)
    import bench
    return bench


def test_paged_prefill_bytes_count_the_keys_each_sequence_sees():
    """bench.py's algorithmic bytes of a paged prefill call: the visible key
    rows of every sequence and head (brute force: the union of the keys each
    query row keeps), the cache blocks that hold them, q and out, the index
    arrays and the bias table."""
    import numpy as np
    import synth
    bench = _bench()
    rng = np.random.default_rng(5)
    for window in (-1, 3, 40):
        for causal in (0, 1):
            ctx = rng.integers(0, 90, size=9)
            ql = np.minimum(ctx, rng.integers(0, 30, size=9))
            pc = synth.make_paged_prefill_case("bytes", 11, synth.BF16, ctx.tolist(), ql.tolist(), 2, 64, window,
                                               causal, 5, scale=1 / 8)
            keys = blocks = 0
            for c, lq in zip(ctx.tolist(), ql.tolist()):
                seen = set()
                for r in range(lq):
                    pos = c - lq + r
                    lo, hi = 0, c
                    if window > 0:
                        lo = max(0, pos - window + 1)
                        if not causal:
                            hi = min(c, pos + window)
                    if causal:
                        hi = min(hi, pos + 1)
                    seen.update(range(lo, hi))
                keys += len(seen)
                blocks += len({k // 16 for k in seen})
            H, D, S = 2, 64, len(ctx)
            want = keys * H * D * 2 * 2 + 2 * int(ql.sum()) * H * D * 2 + blocks * 4 + 4 * S + 4 * (S + 1) \
                + pc.rel_bias.size * 4
            assert bench.paged_prefill_bytes(pc) == want, (window, causal)


def test_prefill_bound_picks_the_longer_of_flops_and_bytes():
    bench = _bench()
    peaks = {"bf16_tflops": 2000.0, "hbm_gbs": 8000.0}          # ridge: 250 FLOP per byte
    b = bench.prefill_bound(2.0e12, 1.0e9, 2.0, peaks)           # 2000 FLOP/B: tensor-bound
    assert b["bound"] == "tensor" and b["frac_roofline"] == b["frac_bf16"] == 0.5
    assert b["frac_hbm"] == 0.0625 and b["intensity_flop_per_byte"] == 2000.0
    b = bench.prefill_bound(1.0e11, 1.0e9, 0.25, peaks)          # 100 FLOP/B: HBM-bound
    assert b["bound"] == "hbm" and b["frac_roofline"] == b["frac_hbm"] == 0.5
    assert b["frac_bf16"] == 0.2


def test_head_dim_128_encoder_workload():
    """--head-dim 128 gives the encoder workload's shapes at head dim 128 (its
    oracle leg runs on them), and is refused for any other workload."""
    sys.path.insert(0, ROOT)
    import synth
    c64, c128 = synth.prefill_workload(0), synth.prefill_workload(0, head_dim=128)
    assert (c64.head_dim, c128.head_dim) == (64, 128)
    assert c64.scale == 1 / 8 and abs(c128.scale - 128 ** -0.5) < 1e-12
    assert (c64.cu_seqlens == c128.cu_seqlens).all() and c64.num_heads == c128.num_heads
    assert c128.q.shape[-1] == 128
    d = _run("--oracle-leg", "--workload", "encoder-prefill", "--head-dim", "128", "--cpu-seconds", "1")
    assert d["unit"] == "TFLOP/s" and d["value"] > 0
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--workload", "tiny-decode",
                        "--head-dim", "128"], capture_output=True, text=True, timeout=120,
                       env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert r.returncode != 0 and "--head-dim" in r.stderr


def test_kernel_source_hash_ignores_comments_only(tmp_path, monkeypatch):
    """The recorded DRAM traffic is keyed by a hash of the kernel's code: a
    comment or blank-line edit keeps the key, a code edit changes it."""
    bench = _bench()
    csrc = tmp_path / "paged_kv_attention_23_gb300" / "csrc"
    csrc.mkdir(parents=True)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    f = csrc / "k.cu"
    f.write_text("// header\nint a = 1;  // trailing\n/* block\n comment */\nint b = 2;\n")
    h0 = bench.kernel_source_hash("k.cu")
    f.write_text("// another header\n\nint a = 1;\n/* other */ int b = 2;\n")
    assert bench.kernel_source_hash("k.cu") == h0
    f.write_text("int a = 1;\nint b = 3;\n")
    assert bench.kernel_source_hash("k.cu") != h0
