"""The decode split's host arithmetic (csrc/fa_internal.h, csrc/fa_api.cu),
compiled as host code with nvcc (no GPU).

fa_decode sizes its workspace for decode_splits(BH, Nk) key ranges, a
figure that does not depend on the GPU, and launches decode_splits_run(BH,
Nk, SMs) ranges, rounded to 64-key chunks.  Checked over a grid of shapes and
SM counts: the launch never uses more ranges than the workspace holds, every
chunk is a whole number of 64-key tiles, no range is empty, and the ranges
cover the cache.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_io_aware_16_gb300", "csrc")

PROGRAM = r"""
#include <cstdio>
#include "fa_internal.h"
int main() {
  const long long bhs[] = {1, 2, 3, 7, 16, 32, 64, 100, 152, 304, 607, 608, 609, 1024, 4096,
                           65536, 1 << 20};
  const int nks[] = {1, 2, 63, 64, 65, 255, 256, 257, 1000, 4096, 8191, 32768, 100000,
                     1 << 20, (1 << 24) + 3};
  const int sms[] = {1, 2, 132, 148, 152, 160, 1024};
  long long checked = 0;
  for (long long bh : bhs)
    for (int nk : nks)
      for (int sm : sms) {
        const int ws = fa::decode_splits(bh, nk);
        int s = fa::decode_splits_run(bh, nk, sm);
        if (s < 1 || s > ws) { std::printf("bad run splits %lld %d %d: %d of %d\n", bh, nk, sm, s, ws); return 1; }
        const int chunk = ((nk + s - 1) / s + 63) / 64 * 64;
        const int s2 = (nk + chunk - 1) / chunk;
        if (chunk % 64 != 0 || s2 < 1 || s2 > s || (long long)(s2 - 1) * chunk >= nk ||
            (long long)s2 * chunk < nk) {
          std::printf("bad chunks %lld %d %d: chunk %d ranges %d of %d\n", bh, nk, sm, chunk, s2, s);
          return 1;
        }
        ++checked;
      }
  std::printf("ok %lld\n", checked);
  return 0;
}
"""


def test_decode_launch_fits_its_workspace(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    src = tmp_path / "splits.cu"
    src.write_text(PROGRAM)
    exe = tmp_path / "splits"
    subprocess.run([nvcc, "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe)],
                   check=True, capture_output=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.startswith("ok"), out.stdout
