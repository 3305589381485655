"""Host test of the binning workspace layout (csrc/binsort_layout.h), no GPU.

The header is plain C++, so a small program compiled with g++ walks many
(n, capacity, tiles) triples and checks the invariants the kernels rely on:
  * the depth sort's buffers (keys A, keys B, values B) are pairwise disjoint and
    disjoint from the persistent depth-sorted values A;
  * the tile sort's buffers (keys A, keys B, the other values buffer) are pairwise
    disjoint;
  * the emission reads the depth-sorted ids from values B (when the last depth pass
    is the identity and skips its copy) while it writes tile keys A and the other
    values buffer: values B overlaps neither;
  * every buffer lies inside the workspace and starts on a 256-byte boundary.
"""
import os
import shutil
import subprocess
import tempfile

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "..", "gaussian_splatting_differentiable_project_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include <cstdint>
#include "binsort_layout.h"
using namespace gs;

struct Buf { size_t off, len; };
static bool disjoint(Buf a, Buf b) { return a.off + a.len <= b.off || b.off + b.len <= a.off; }

int main() {
  uint64_t s = 12345;
  auto rnd = [&](uint64_t m) { s = s * 6364136223846793005ull + 1442695040888963407ull; return (s >> 17) % m; };
  long checked = 0;
  for (int it = 0; it < 20000; ++it) {
    const int64_t n = 1 + int64_t(rnd(it % 3 == 0 ? 100 : (it % 3 == 1 ? 70000 : 5000000)));
    const uint32_t cap = 1u + uint32_t(rnd(it % 4 == 0 ? 50 : (it % 4 == 1 ? 3 * uint64_t(n) : 40000000)));
    const int64_t tiles = 1 + int64_t(rnd(70000));
    const SortLayout L = sort_layout(n, cap, tiles);
    const size_t vn = size_t(n) * 4, vk = size_t(cap) * 4;
    const Buf dvA{L.dvA, vn}, dkA{L.dkA(), vn}, dkB{L.dkB(), vn}, dvB{L.dvB(), vn};
    const Buf tkA{L.tkA(), vk}, tkB{L.tkB(), vk}, tvAlt{L.tvAlt(), vk};
    const Buf all[] = {dvA, dkA, dkB, dvB, tkA, tkB, tvAlt};
    for (const Buf& b : all) {
      if (b.off % 256 != 0 || b.off + b.len > L.total) { printf("bounds n=%lld cap=%u\n", (long long)n, cap); return 1; }
    }
    const Buf depth[] = {dvA, dkA, dkB, dvB};
    for (int i = 0; i < 4; ++i)
      for (int j = i + 1; j < 4; ++j)
        if (!disjoint(depth[i], depth[j])) { printf("depth overlap n=%lld cap=%u\n", (long long)n, cap); return 1; }
    const Buf tile[] = {tkA, tkB, tvAlt};
    for (int i = 0; i < 3; ++i)
      for (int j = i + 1; j < 3; ++j)
        if (!disjoint(tile[i], tile[j])) { printf("tile overlap n=%lld cap=%u\n", (long long)n, cap); return 1; }
    if (!disjoint(dvB, tkA) || !disjoint(dvB, tvAlt) || !disjoint(dvA, tkA) || !disjoint(dvA, tvAlt)) {
      printf("emission overlap n=%lld cap=%u\n", (long long)n, cap);
      return 1;
    }
    ++checked;
  }
  printf("ok %ld\n", checked);
  return 0;
}
"""


def test_sort_workspace_slots():
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "layout_check.cpp")
        exe = os.path.join(d, "layout_check")
        with open(src, "w") as f:
            f.write(PROGRAM)
        subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, src, "-o", exe], check=True)
        out = subprocess.run([exe], capture_output=True, text=True)
        assert out.returncode == 0, out.stdout + out.stderr
        assert out.stdout.startswith("ok 20000")
