"""The decode's automatic split count, checked on the CPU.

``decode_split`` (in the C-ABI source) picks how many key chunks each head's decode is cut
into when the caller passes num_splits = 0.  Its contract, which fa_decode_noalloc's static
scratch relies on: every automatic choice needs at most 4 MiB of split scratch, chunks hold
at least 256 keys (a whole number of 64-key tiles) unless the cache is shorter, the chunks
cover the cache exactly once, and an explicit request is honoured.  The function and its
scratch-size helper are compiled for the host from the source itself, so the test checks
the library's own code.
"""
import os
import re
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "..", "transformer_attention_flashattention_gb300", "csrc", "fa_api.cu")

DRIVER = r"""
#include <cstdio>
@FUNCTIONS@
int main() {
  const int heads[] = {1, 3, 16, 64, 152, 256, 304, 1024, 4096};
  const int nqs[] = {1, 2, 4, 5, 16};
  const int nks[] = {1, 63, 64, 256, 300, 1000, 4096, 32768, 131072};
  const int ds[] = {64, 128};
  long bad = 0, configs = 0;
  for (int BH : heads) for (int Nq : nqs) for (int Nk : nks) for (int d : ds) {
    if (Nq > Nk) continue;
    int splits = 0, chunk = 0;
    decode_split(BH, Nq, Nk, d, 0, 152, &splits, &chunk);
    ++configs;
    const bool covers = splits >= 1 && chunk % 64 == 0 && (long)(splits - 1) * chunk < Nk &&
                        (long)splits * chunk >= Nk;
    const bool fits = decode_workspace(BH, Nq, d, splits) <= (4ull << 20);
    const bool big_enough = splits == 1 || chunk >= 256;
    if (!covers || !fits || !big_enough) {
      ++bad;
      printf("bad BH=%d Nq=%d Nk=%d d=%d -> splits %d chunk %d\n", BH, Nq, Nk, d, splits, chunk);
    }
    // an explicit request: that many chunks, or fewer when 64-key rounding merges some
    int s2 = 0, c2 = 0;
    decode_split(BH, Nq, Nk, d, 7, 152, &s2, &c2);
    if (s2 < 1 || s2 > 7 || (long)(s2 - 1) * c2 >= Nk || (long)s2 * c2 < Nk) ++bad;
  }
  int s = 0, c = 0;
  decode_split(256, 1, 32768, 128, 0, 152, &s, &c);
  printf("bench %d %d\n", s, c);
  printf("configs %ld bad %ld\n", configs, bad);
  return bad != 0;
}
"""


def _extract():
    src = open(SOURCE).read()
    out = []
    for pat in (r"unsigned long long decode_workspace\(int BH.*?\n}\n",
                r"constexpr unsigned long long kAutoSplitScratch = .*?;\n",
                r"void decode_split\(int BH.*?\n}\n"):
        m = re.search(pat, src, re.S)
        assert m, f"{pat} not found in the C-ABI source"
        out.append(m.group(0))
    return "\n".join(out)


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs a host C++ compiler")
def test_automatic_split_count_keeps_its_contract(tmp_path):
    cpp = tmp_path / "split.cpp"
    cpp.write_text(DRIVER.replace("@FUNCTIONS@", _extract()))
    exe = tmp_path / "split"
    r = subprocess.run(["g++", "-O2", "-std=c++17", str(cpp), "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "bad 0" in r.stdout
    # the benchmark's decode workload (8 x 32 heads, one query row, 32768 keys, d = 128):
    # two CTAs per SM, 7 chunks of 4736 keys (1792 CTAs, 5.9 waves of 304)
    assert "bench 7 4736" in r.stdout, r.stdout
