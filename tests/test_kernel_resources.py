"""Register and spill budget of every attention kernel, read from the
compiler's own report (`ptxas -v`) of the sources as built (no GPU).

- The forward, dQ and dK/dV kernels run 10 warps (320 threads) and allocate
  all 512 tensor-memory columns.  At most 168 registers a thread lets three
  of those warps share one SM sub-partition's 16,384 registers.  More than
  102 means two CTAs never fit the SM's 65,536 registers, so no CTA's
  tensor-memory allocation waits for another CTA of the same kernel.  (Their
  dynamic shared memory, above half the SM's, guarantees the same, but the
  compiler does not report it.)
- The plain and e4m3 forwards, every dQ kernel, the dK/dV kernels without
  dropout and the D pre-pass spill nothing.  The block-sparse and dropout
  forwards and the dropout dK/dV kernels spill a few dozen bytes each (the
  keep bits and the tile list's state), bounded here so that a change which
  spills the softmax loop shows up.
"""
import os
import re
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

import pytest

from exact_io_aware_16_gb300 import build as fabuild

SOURCES = ("fa_fwd.cu", "fa_bwd.cu")
# a kernel's mangled name: <length>fa_..._kernel I Li<D>E Lb<flag>E ... E
MANGLED = re.compile(r"\d(fa_[a-z0-9_]+?_kernel)ILi(\d+)E((?:Lb[01]E)*)E")
# template flags after D, in declaration order
FLAGS = {"fa_fwd_kernel": ("CAUSAL", "SPARSE", "DROPOUT", "FP8", "PERSIST"),
         "fa_bwd_dkdv_kernel": ("CAUSAL", "SPARSE", "DROPOUT", "PERSIST"),
         "fa_bwd_dq_kernel": ("CAUSAL", "SPARSE", "DROPOUT", "PERSIST")}


def ptxas_report(tmp_path):
    if not (shutil.which("nvcc") or os.path.exists("/usr/local/cuda/bin/nvcc")):
        pytest.skip("nvcc not found")
    cc = fabuild.nvcc()

    def one(src):
        cmd = [cc, *fabuild.ARCH, *fabuild.FLAGS, "-Xptxas", "-v", "-c",
               os.path.join(fabuild.CSRC, src), "-o", str(tmp_path / (src + ".o"))]
        r = subprocess.run(cmd, capture_output=True, text=True)
        assert r.returncode == 0, r.stderr[-2000:]
        return r.stdout + r.stderr

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        return "\n".join(ex.map(one, SOURCES))


def parse(report):
    """{mangled entry: {"regs", "stack", "spill_st", "spill_ld"}}"""
    out, cur = {}, None
    for line in report.splitlines():
        m = re.search(r"Compiling entry function '(\S+)'", line)
        if m:
            cur = out.setdefault(m.group(1), {})
            continue
        m = re.search(r"Function properties for (\S+)", line)
        if m:
            cur = out.setdefault(m.group(1), {})
            continue
        m = re.search(r"(\d+) bytes stack frame, (\d+) bytes spill stores, (\d+) bytes spill loads",
                      line)
        if m and cur is not None:
            cur["stack"], cur["spill_st"], cur["spill_ld"] = (int(x) for x in m.groups())
            continue
        m = re.search(r"Used (\d+) registers", line)
        if m and cur is not None:
            cur["regs"] = int(m.group(1))
    return out


def kernels(tmp_path):
    res = []
    for name, st in parse(ptxas_report(tmp_path)).items():
        m = MANGLED.search(name)
        if "regs" not in st:
            continue
        if m:
            kname, d = m.group(1), int(m.group(2))
            bits = [b == "1" for b in re.findall(r"Lb([01])E", m.group(3))]
            flags = dict(zip(FLAGS.get(kname, ()), bits))
        elif "fa_bwd_pre_kernel" in name:
            kname, d, flags = "fa_bwd_pre_kernel", None, {}
        else:
            continue
        res.append((kname, d, flags, st))
    return res


def test_register_and_spill_budget(tmp_path):
    ks = kernels(tmp_path)
    seen = {(k, d) for k, d, _, _ in ks}
    for k in FLAGS:
        assert {(k, 64), (k, 128)} <= seen, f"{k}: both head sizes must be instantiated"
    assert any(k == "fa_bwd_pre_kernel" for k, *_ in ks)
    for k, d, flags, st in ks:
        tag = f"{k}<{d}, {flags}>"
        if k in FLAGS:
            assert 103 <= st["regs"] <= 168, f"{tag}: {st['regs']} registers"
        spill_free = (k == "fa_bwd_pre_kernel" or k == "fa_bwd_dq_kernel"
                      or (k == "fa_bwd_dkdv_kernel" and not flags["DROPOUT"])
                      or (k == "fa_fwd_kernel" and not flags["SPARSE"] and not flags["DROPOUT"]))
        if spill_free:
            assert st["spill_st"] == 0 and st["spill_ld"] == 0, f"{tag} spills: {st}"
        else:
            assert st["spill_st"] <= 96 and st["spill_ld"] <= 160, f"{tag} spills: {st}"
