"""The benchmark's command line on CPU: the reference arm (the oracle timed on the host cores)
prints one JSON line with the contract's keys, and the defaults keep at least 3 warm-up
steps."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_the_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["value"] > 0 and d["steps"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["e2e"]["value"] == d["value"]


def test_defaults_warm_up_at_least_three_steps(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    a = bench.parse()
    assert a.gpus == 1 and a.warmup >= 3 and a.steps >= 1 and a.impl == "ours"


def test_peak_basis_follows_the_timed_region():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.bf16_peak_basis(0.13) == ("bf16_tflops", "burst")
    assert bench.bf16_peak_basis(2.5) == ("bf16_tflops_sustained", "sustained")


def test_error_stats_of_bf16_bits():
    import numpy as np
    sys.path.insert(0, ROOT)
    import bench
    ref = np.array([0x3F80, 0x4000, 0xBF80, 0x0000], dtype=np.uint16)     # 1, 2, -1, 0
    got = np.array([0x3F81, 0x4000, 0xBF80, 0x0000], dtype=np.uint16)     # 1 + 2^-7
    st = bench.error_stats(np, got, ref, "four values")
    assert st["max_abs"] == 2.0 ** -7 and st["max_ulp"] == 1 and st["mismatch_bits"] == 1
    assert abs(st["frob_rel"] - 2.0 ** -7 / 6 ** 0.5) < 1e-12
