"""The generator's shared-counter-word forms against the oracle's Philox4x32-10.

The dropout kernels form the products that depend only on the counter words a
row shares (query row, head, offset; or key group, head, offset) once per
item, and each call then runs the remaining rounds (`philox_row_call`,
`philox_col_call` in csrc/philox.cuh).  Both must give the generator's own
output, bit for bit ("Parallel random numbers: as easy as 1, 2, 3", Salmon et
al., SC 2011: ten rounds of the two multiplies and the key schedule).  The
header is compiled here as host code with nvcc (no GPU) and checked against
the oracle's generator on seeded random counters and keys, with the extreme
word values included.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_io_aware_16_gb300", "csrc")

PROGRAM = r"""
#include <cuda_runtime.h>
#include <cstdio>
#include "philox.cuh"
int main() {
  unsigned c0, c1, c2, c3, k0, k1;
  while (std::scanf("%u %u %u %u %u %u", &c0, &c1, &c2, &c3, &k0, &k1) == 6) {
    fa::DropArgs dr;
    dr.set_seed(k0, k1);
    dr.offset = c3;
    const uint4 a = fa::philox_row_call(dr, fa::philox_row_init(dr, c1, c2), c0);
    const uint4 b = fa::philox_col_call(dr, fa::philox_col_init(dr, c0, c2), c1);
    std::printf("%u %u %u %u %u %u %u %u\n", a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w);
  }
  return 0;
}
"""


def nvcc():
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        pytest.skip("nvcc not found")
    return path


def test_shared_word_forms_equal_the_generator(tmp_path):
    src = tmp_path / "philox_forms.cu"
    src.write_text(PROGRAM)
    exe = tmp_path / "philox_forms"
    subprocess.run([nvcc(), "-std=c++17", "-O2", "-I", CSRC, str(src), "-o", str(exe)],
                   check=True, capture_output=True)
    rng = np.random.default_rng(20261203)
    words = rng.integers(0, 2**32, size=(2000, 6), dtype=np.uint64)
    edge = [0, 1, 0x7FFFFFFF, 0x80000000, 0xFFFFFFFF]
    for r, v in enumerate(edge):  # extreme values in every word position
        words[r, :] = v
        words[len(edge) + r, r % 6] = v
    lines = "\n".join(" ".join(str(int(x)) for x in row) for row in words) + "\n"
    out = subprocess.run([str(exe)], input=lines, capture_output=True, text=True, check=True)
    got = [list(map(int, line.split())) for line in out.stdout.splitlines()]
    assert len(got) == len(words)
    o = oracle.default()
    for row, g in zip(words, got):
        c0, c1, c2, c3, k0, k1 = (int(x) for x in row)
        want = o.philox([c0, c1, c2, c3], [k0, k1])
        assert g[:4] == want, f"row form differs at counter {row.tolist()}"
        assert g[4:] == want, f"column form differs at counter {row.tolist()}"
