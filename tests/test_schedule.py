"""The causal work split of the persistent kernels, checked on the CPU.

``causal_unit`` (in the forward kernel header, shared by every forward kernel and both
backward kernels) deals a CTA its k-th causal unit: whole pairs of blocks b and n-1-b for
all rounds of the grid but the last, then the remaining units sorted by cost and dealt in
snake order.  A unit dealt twice or never would corrupt or leave out part of O or of a
gradient, so every grid size, head count, block count and cost direction here must deal
each (head, block) exactly once.  The function is compiled for the host from the header
itself (its device qualifiers defined away), so the test checks the kernels' own code.
"""
import os
import re
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
HEADER = os.path.join(HERE, "..", "transformer_attention_flashattention_gb300", "csrc", "fa_fwd_kernel.cuh")

DRIVER = r"""
#include <algorithm>
#include <cstdio>
#include <vector>
using std::max;
using std::min;
#define __device__
#define __noinline__
#define __forceinline__ inline
@FUNCTION@
int main() {
  const int grids[] = {1, 2, 3, 7, 16, 151, 152, 304};
  const int heads[] = {1, 2, 3, 5, 16, 32, 64, 256};
  const int blocks[] = {1, 2, 3, 4, 5, 8, 15, 16, 17, 64, 256};
  long bad = 0, configs = 0;
  for (int G : grids) for (int BH : heads) for (int n : blocks) for (int cg = 0; cg < 2; ++cg) {
    if ((long)BH * n > 70000) continue;
    std::vector<int> seen((size_t)BH * n, 0);
    std::vector<long> load(G, 0);
    for (int c = 0; c < G; ++c) {
      int bh, blk;
      for (int k = 0; causal_unit(G, c, BH, n, k, cg != 0, bh, blk); ++k) {
        if (bh < 0 || bh >= BH || blk < 0 || blk >= n) { ++bad; break; }
        ++seen[(size_t)bh * n + blk];
        load[c] += cg ? blk + 1 : n - blk;
      }
    }
    for (int x : seen) if (x != 1) ++bad;
    ++configs;
    // the load balance the split is for, at two shapes of the benchmarks
    if (G == 152 && n == 16 && BH == 256) {
      long mx = 0, sum = 0;
      for (long l : load) { mx = std::max(mx, l); sum += l; }
      printf("balance %d %d %d %.4f\n", BH, n, cg, (double)mx * G / sum);
    }
  }
  printf("configs %ld bad %ld\n", configs, bad);
  return bad != 0;
}
"""


def _extract():
    src = open(HEADER).read()
    m = re.search(r"static __device__ __noinline__ bool causal_unit\(.*?\n}\n", src, re.S)
    assert m, "causal_unit not found in the forward kernel header"
    return m.group(0).replace("static ", "", 1)


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs a host C++ compiler")
def test_causal_unit_deals_every_unit_once(tmp_path):
    cpp = tmp_path / "sched.cpp"
    cpp.write_text(DRIVER.replace("@FUNCTION@", _extract()))
    exe = tmp_path / "sched"
    r = subprocess.run(["g++", "-O2", "-std=c++17", str(cpp), "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "bad 0" in r.stdout
    # 16x16x2048 backward: 256 heads of 16 tiles on 152 CTAs; whole pairs alone would leave
    # the most loaded CTA at 1.039 x the mean
    for line in r.stdout.splitlines():
        if line.startswith("balance"):
            assert float(line.split()[-1]) <= 1.02, line
