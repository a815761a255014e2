"""The benchmark's JSON line on a GPU: one line with the contract's keys, the
roofline block, the end-to-end block and a positive launch count."""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("extra", [[], ["--kv", "fp8"], ["--qlen", "2"]])
def test_bench_prints_one_contract_line(extra):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--steps", "20", "--warmup", "3",
           "--no-clocks", "--no-cpu-baseline"] + extra
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "e2e", "gpu_launches"):
        assert key in d, key
    assert d["n_gpus"] == 1 and d["steps"] == 20 and d["warmup"] == 3
    assert d["value"] > 0 and d["higher_is_better"] is True and d["scaling"] == "weak"
    assert "workload" in d["config"]
    rl = d["roofline"]
    assert rl["bound"] == "hbm" and rl["unit"] == "GB/s" and rl["peak"] > 0
    assert abs(rl["frac"] - rl["achieved"] / rl["peak"]) < 1e-3
    # one launch per step: the kernel's average launch duration is the step time,
    # so achieved equals the headline value; single launches timed alone take longer
    assert abs(rl["achieved"] - d["value"]) <= 1e-3 * d["value"]
    assert abs(rl["kernel_us"] - d["us_per_step"]) <= 0.02
    assert 0 < rl["frac_isolated"] <= rl["frac"] * 1.02
    e2e = d["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] >= 20
