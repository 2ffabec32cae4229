"""bench.py's JSON line and the seeded input recipes, on CPU.

The reference arm (the fp64 oracle on host cores) runs a small sample and must print
one JSON line with the contract's keys; the input generators must be deterministic
and hold the documented recipes (seeded lengths that sum to the total, weight scale).
"""
import json
import os
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_the_contract_line():
    res = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                          "--warmup", "3", "--cpu-seconds", "0.3"],
                         cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["steps"] == 1 and d["warmup"] == 3
    assert d["value"] > 0 and d["unit"] == "tokens/s" and d["higher_is_better"] is True
    assert d["config"]["workload"] == "prefill_8k"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_bench_defaults_and_warmup_floor():
    sys.path.insert(0, ROOT)
    import bench
    a = bench.parse_args([])
    assert a.gpus == 1 and a.warmup >= 3 and a.steps >= 1 and a.impl == "ours"
    assert bench.parse_args(["--warmup", "0"]).warmup == 3


def test_varlen_lengths_recipe():
    from linear_attention_hybrid_fwd_b300.inputs import varlen_lengths
    a = varlen_lengths(65536, 1, 8192, 6)
    assert a == varlen_lengths(65536, 1, 8192, 6)           # seeded
    assert sum(a) == 65536 and all(1 <= n <= 8192 for n in a)
    assert len(a) == 15 and sum(1 for n in a if n % 128) == 15  # every end mid-chunk


def test_projection_inputs_recipe():
    import torch
    from linear_attention_hybrid_fwd_b300.inputs import make_projection_inputs
    x, w = make_projection_inputs(64, 512, 2, 128, 3, "cpu")
    x2, w2 = make_projection_inputs(64, 512, 2, 128, 3, "cpu")
    assert torch.equal(x, x2) and torch.equal(w, w2)
    assert x.dtype == torch.bfloat16 and tuple(w.shape) == (4 * 2 * 128, 512)
    # w ~ N(0, 1) * 0.5 / sqrt(hidden): the projected features are about N(0, 0.25)
    std = float(w.float().std())
    assert abs(std - 0.5 / np.sqrt(512)) < 0.05 * 0.5 / np.sqrt(512)
