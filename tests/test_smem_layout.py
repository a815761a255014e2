"""Host-only check of the decode kernel's shared-memory layout.

The layout header is plain C++; this test compiles a small program against it
with the host compiler and checks, for every supported head_dim / block_size,
every ring depth the planner can choose, every group size and a spread of batch
sizes, that each region starts where its accesses need it to (1024 bytes for the
TMA-filled ring, 8 for mbarriers, 16 or more for the float4 merge buffer) and
that the regions are in order without overlap.  A misaligned merge buffer is a
misaligned-address fault on the GPU, so this runs before any kernel does.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "paged_kv_gqa_decode_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <initializer_list>
#include "smem_layout.h"
using namespace pagedattn;

static int bad = 0;
#define CHECK(c, ...) do { if (!(c)) { if (bad < 20) std::printf(__VA_ARGS__); ++bad; } } while (0)

template <int D, int BS, bool FP8 = false>
void run() {
  using L = SmemLayout<D, BS, FP8>;
  const int ns[] = {1, 2, 3, 5, 7, 31, 32, 33, 255, 256, 257, 1000, 4095, 4096};
  for (int st = 4; st <= 16; ++st)
    for (int G = 1; G <= 16; ++G)
      for (int n : ns)
      for (int qo : {0, n + 1})
      for (int walks : {1, 3}) {
        const L l{st, G, n, qo, walks};
        CHECK(l.bars() % 1024 == 0, "bars D%d BS%d st%d\n", D, BS, st);
        CHECK(L::kStageBytes % 1024 == 0, "stage size D%d BS%d\n", D, BS);
        CHECK(l.merge_m() >= l.bars() + (2 * st + 1) * 8, "barrier overlap\n");
        CHECK(l.scales() >= l.bars() + (2 * st + 1) * 8, "scales overlap\n");
        CHECK(l.merge_m() >= l.scales() + st * L::kScaleBytes, "scale ring size\n");
        const int starts[] = {l.scales(), l.merge_m(), l.merge_l(), l.final_ml(), l.flag(),
                              l.merge_o(), l.qtile(), l.prefix(), l.wprefix(), l.lens()};
        for (int x : starts)
          CHECK(x % 128 == 0, "region at %d D%d BS%d st%d G%d n%d\n", x, D, BS, st, G, n);
        CHECK(l.merge_l() - l.merge_m() >= kConsumerWarps * 16 * 4, "merge_m size\n");
        CHECK(l.final_ml() - l.merge_l() >= kConsumerWarps * 16 * 4, "merge_l size\n");
        CHECK(l.flag() - l.final_ml() >= 32 * 4, "final size\n");
        CHECK(l.merge_o() - l.flag() >= 4 * 4, "flag size\n");
        CHECK(l.qtile() - l.merge_o() >= kConsumerWarps * G * L::kRowStride * 4, "merge_o size\n");
        CHECK(l.prefix() - l.qtile() >= kQSlots * ((G > 8 ? 16 : 8) * D * 2 + 4 * D + 4),
              "qtile size\n");
        if (FP8) {
          CHECK(l.q_extra_bytes() >= (G > 8 ? 16 : 8) * (2 * D + 32), "q16 size\n");
          CHECK(L::kQ16Stride % 32 == 0, "q16 stride\n");
          CHECK(L::kPageBytes == BS * D, "fp8 page\n");
        }
        CHECK(l.q_slot_bytes() % 128 == 0, "q slot\n");
        CHECK(l.q_tile_bytes() % 128 == 0, "qtile bytes\n");
        CHECK((L::kRowStride * 4) % 16 == 0, "row stride\n");
        CHECK(l.wprefix() - l.prefix() >= (walks * n + 1) * 4, "prefix size\n");
        CHECK(l.lens() - l.wprefix() >= (walks * n + 1) * 4, "wprefix size\n");
        CHECK(l.qo() - l.lens() >= n * 4, "lens size\n");
        CHECK(l.qo() % 16 == 0, "qo alignment\n");
        CHECK(l.total() - l.qo() >= qo * 4, "qo size\n");
      }
}

int main() {
  run<64, 16>(); run<64, 32>(); run<128, 16>(); run<128, 32>(); run<256, 16>(); run<256, 32>();
  run<128, 16, true>(); run<128, 32, true>(); run<256, 16, true>(); run<256, 32, true>();
  std::printf(bad ? "FAIL %d\n" : "OK\n", bad);
  return bad ? 1 : 0;
}
"""


def test_shared_memory_regions_aligned_and_disjoint(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    src = tmp_path / "layout_check.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "layout_check"
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip().endswith("OK"), r.stdout
