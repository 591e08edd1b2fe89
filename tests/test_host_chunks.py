"""The host pipeline's chunking of heads, checked on the CPU.

``chunk_sizes`` (in the host-pipeline source) cuts a call's B*H heads into the chunks whose
copies and computations fa_fwd_host and fa_fwd_fp8_host overlap.  Every head must land in
exactly one chunk, every chunk must hold a head, and there are at most 32 of them (the
per-device event arrays).  With chunks = 0 the sizes ramp 1, 2, 4, ... up to B*H/8 and back
down, so the link carries only a small chunk while nothing computes.  The function is
compiled for the host from the source itself.
"""
import os
import re
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "..", "transformer_attention_flashattention_gb300", "csrc", "fa_host.cu")

DRIVER = r"""
#include <cstdio>
@CONSTANTS@
@FUNCTION@
int main() {
  long bad = 0, configs = 0;
  const int requests[] = {0, 1, 2, 3, 8, 31, 32, 64};
  for (long long BH = 1; BH <= 3000; ++BH) for (int ch : requests) {
    long long size[kMaxChunks];
    const int n = chunk_sizes(BH, ch, size);
    long long sum = 0;
    bool ok = n >= 1 && n <= kMaxChunks;
    for (int i = 0; ok && i < n; ++i) { ok = size[i] >= 1; sum += size[i]; }
    ok = ok && sum == BH;
    if (ch > 0) ok = ok && n <= ch;
    if (!ok) { ++bad; printf("bad BH=%lld chunks=%d n=%d\n", BH, ch, n); }
    ++configs;
  }
  long long size[kMaxChunks];
  const int n = chunk_sizes(32, 0, size);
  printf("ramp32");
  for (int i = 0; i < n; ++i) printf(" %lld", size[i]);
  printf("\nconfigs %ld bad %ld\n", configs, bad);
  return bad != 0;
}
"""


def _extract():
    src = open(SOURCE).read()
    consts = re.findall(r"constexpr int (?:kMaxChunks|kAutoChunks) = \d+;", src)
    assert len(consts) == 2, "chunk constants not found"
    m = re.search(r"int chunk_sizes\(long long BH.*?\n}\n", src, re.S)
    assert m, "chunk_sizes not found in the host-pipeline source"
    return "\n".join(consts), m.group(0)


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs a host C++ compiler")
def test_chunk_sizes_cover_every_head_once(tmp_path):
    consts, fn = _extract()
    cpp = tmp_path / "chunks.cpp"
    cpp.write_text(DRIVER.replace("@CONSTANTS@", consts).replace("@FUNCTION@", fn))
    exe = tmp_path / "chunks"
    r = subprocess.run(["g++", "-O2", "-std=c++17", str(cpp), "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "bad 0" in r.stdout
    # the long-context workload's 32 heads: 1, 2, then chunks of B*H/8 = 4, then back down
    assert "ramp32 1 2 4 4 4 4 4 4 2 2 1" in r.stdout, r.stdout
