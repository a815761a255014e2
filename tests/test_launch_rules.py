"""The bench's count of kernel launches per step (its `gpu_launches` claim)
follows the library's own grid rule: bench.ctas_per_sm must agree with the
kernel's ctas_per_sm (csrc/decode_kernel.cuh) for every head_dim, page size,
group size and cache format.  The kernel's rule is evaluated by a small host
program compiled with nvcc; no GPU is needed."""
import os
import shutil
import subprocess

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "paged_kv_gqa_decode_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include "decode_kernel.cuh"
int main() {
  for (int D : {64, 128, 256})
    for (int BS : {16, 32})
      for (int g16 = 0; g16 < 2; ++g16)
        for (int fp8 = 0; fp8 < 2; ++fp8)
          std::printf("%d %d %d %d %d\n", D, BS, g16, fp8,
                      pagedattn::ctas_per_sm(D, g16 != 0, BS, fp8 != 0));
  return 0;
}
"""


def test_bench_grid_rule_matches_the_kernel(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    src = tmp_path / "rule.cu"
    src.write_text(PROGRAM)
    exe = tmp_path / "rule"
    subprocess.run([nvcc, "-std=c++17", "--expt-relaxed-constexpr", "-I", CSRC,
                    "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    rows = [list(map(int, line.split())) for line in out.split("\n") if line.strip()]
    assert len(rows) == 3 * 2 * 2 * 2
    for D, BS, g16, fp8, ctas in rows:
        if fp8 and D == 64:
            continue  # no FP8 kernel at head_dim 64
        G = 16 if g16 else 8
        assert bench.ctas_per_sm(D, BS, G, bool(fp8)) == ctas, (D, BS, g16, fp8, ctas)
        # a group of 1..8 heads uses the 8-row pieces
        assert bench.ctas_per_sm(D, BS, 4 if not g16 else 12, bool(fp8)) == ctas
