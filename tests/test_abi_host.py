"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point declared in include/fa.h, and rejects bad arguments with
the documented status codes before touching the device."""
import ctypes
import os
import re

import pytest

import exact_io_aware_16_gb300 as fa
from exact_io_aware_16_gb300 import build as fabuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    fabuild.build()
    return fa.library()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            txt = open(os.path.join(ROOT, "include", fn)).read()
            txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
            names |= set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", txt))
    return sorted(names)


def test_header_declares_entry_points():
    names = declared_functions()
    for must in ("fa_forward", "fa_backward", "fa_backward_workspace_size",
                 "fa_get_device_error", "fa_status_string"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation returns first


def fwd(lib, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=1, N=128, d=64, scale=0.125,
        causal=0):
    return lib.fa_forward(q, k, v, o, lse, B, H, N, d, scale, causal, None)


def test_forward_validation(lib):
    assert fwd(lib, q=None) == -1
    assert fwd(lib, lse=None) == -1
    assert fwd(lib, N=0) == -2
    assert fwd(lib, B=0) == -2
    assert fwd(lib, H=-1) == -2
    assert fwd(lib, d=96) == -3
    assert fwd(lib, d=256) == -3
    assert fwd(lib, scale=0.0) == -2
    assert fwd(lib, scale=-1.0) == -2
    assert fwd(lib, scale=float("inf")) == -2
    assert fwd(lib, B=1 << 16, H=1 << 15, N=4, d=64) == -2  # B*H >= 2^31
    assert fwd(lib, q=FAKE + 8) == -4
    assert fwd(lib, o=FAKE + 2) == -4
    assert fwd(lib, lse=FAKE + 4) == -4


def bwd(lib, ws=FAKE * 16, ws_bytes=1 << 20, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, dO=FAKE, lse=FAKE, dq=FAKE, dk=FAKE, dv=FAKE,
             B=1, H=1, N=128, d=64, scale=0.125, causal=0)
    a.update(kw)
    return lib.fa_backward(a["q"], a["k"], a["v"], a["o"], a["dO"], a["lse"], a["dq"], a["dk"],
                           a["dv"], a["B"], a["H"], a["N"], a["d"], a["scale"], a["causal"],
                           ws, ws_bytes, None)


def test_backward_validation(lib):
    assert bwd(lib, dO=None) == -1
    assert bwd(lib, dv=None) == -1
    assert bwd(lib, N=0) == -2
    assert bwd(lib, d=32) == -3
    assert bwd(lib, ws=None) == -6
    assert bwd(lib, ws_bytes=100) == -6
    assert bwd(lib, ws=FAKE * 16 + 16) == -6  # workspace must be 256-byte aligned
    assert bwd(lib, dk=FAKE + 4) == -4


def test_shapes_beyond_2_31_elements(lib):
    """B*H*N*d is not limited to 32 bits; B*H and the work items of a launch
    (B*H*ceil(N/128)) are.  Each call below passes the shape check and then
    fails the alignment check that follows it (FA_ERR_ALIGN), so nothing is
    launched on any machine."""
    # 2^36 elements: B*H = 2^20, N = 512, d = 128
    big = dict(B=1 << 10, H=1 << 10, N=512, d=128)
    assert fwd(lib, q=FAKE + 8, **big) == -4
    assert bwd(lib, dq=FAKE + 8, ws_bytes=1 << 40, **big) == -4
    n = 4 * (1 << 20) * 512
    assert lib.fa_backward_workspace_size(1 << 10, 1 << 10, 512, 128) == n
    # largest allowed item count: B*H*ceil(N/128) = 2^31 - 1
    assert fwd(lib, q=FAKE + 8, B=1, H=(1 << 31) - 1, N=128, d=64) == -4
    # one more item, or B*H = 2^31, is refused
    assert fwd(lib, q=FAKE + 8, B=1, H=(1 << 30), N=257, d=64) == -2
    assert fwd(lib, q=FAKE + 8, B=2, H=1 << 30, N=1, d=64) == -2
    assert lib.fa_backward_workspace_size(2, 1 << 30, 1, 64) == 0
    # decode: a 2^33-element cache is accepted by the shape check
    assert lib.fa_decode(FAKE + 8, FAKE, FAKE, FAKE, FAKE, 1, 64, 4, 1 << 20, 128, 0.125, 0,
                         FAKE * 16, 1 << 40, None) == -4
    assert lib.fa_decode_workspace_size(1, 64, 4, 1 << 20, 128) > 0


def test_blocksparse_validation(lib):
    f = lib.fa_forward_blocksparse
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 256, 64, 0.125, 0, None, 0, None) == -1
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 256, 64, 0.125, 0, FAKE, -5, None) == -2
    # more than 1024 tiles along N
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 128 * 1024 + 1, 64, 0.125, 0, FAKE, 0,
             None) == -2
    g = lib.fa_backward_blocksparse
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 256, 64, 0.125, 0,
             None, 0, FAKE * 16, 1 << 20, None) == -1


def test_dropout_validation(lib):
    f = lib.fa_forward_dropout
    g = lib.fa_backward_dropout

    def fw(p=0.1, q=FAKE, mask=None, stride=0, N=256):
        return f(q, FAKE, FAKE, FAKE, FAKE, 1, 1, N, 64, 0.125, 0, p, 7, 0, mask, stride, None)

    for p in (-0.01, 1.0, 2.0, float("nan"), float("inf")):
        assert fw(p=p) == -2
    assert fw(q=None) == -1
    assert fw(mask=FAKE, stride=-1) == -2
    assert fw(mask=FAKE, N=128 * 1024 + 1) == -2

    def bw(p=0.1, q=FAKE, w=FAKE * 16):
        return g(q, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 256, 64, 0.125, 0, p,
                 7, 0, None, 0, w, 1 << 20, None)

    assert bw(p=1.5) == -2
    assert bw(q=None) == -1
    assert bw(w=None) == -6


def test_fp8_validation(lib):
    f = lib.fa_forward_fp8

    def fw(N=256, d=128, qd=1.0, q=FAKE, scale=0.125):
        return f(q, FAKE, FAKE, qd, 1.0, 1.0, FAKE, FAKE, 1, 2, N, d, scale, 0, None)

    assert fw(q=None) == -1
    assert fw(d=64) == -3
    assert fw(N=100) == -2  # not a multiple of 16
    assert fw(qd=0.0) == -2
    assert fw(qd=float("nan")) == -2
    assert fw(scale=-1.0) == -2
    assert fw(qd=1e30, scale=1e30) == -2  # folded score scale overflows


def test_host_plan_validation(lib):
    h = ctypes.c_void_p()
    f = lib.fa_host_plan_create
    assert f(1, 1, 128, 64, 0.125, 0, None) == -1
    assert f(0, 1, 128, 64, 0.125, 0, ctypes.byref(h)) == -2
    assert f(1, 1, 128, 96, 0.125, 0, ctypes.byref(h)) == -3
    assert f(1, 1, 128, 64, float("nan"), 0, ctypes.byref(h)) == -2
    assert h.value is None  # nothing was created
    assert lib.fa_host_step(None, *([FAKE] * 9)) == -1
    assert lib.fa_host_wait(None) == -1
    assert lib.fa_host_plan_destroy(None) == 0


def test_decode_validation(lib):
    ws = lib.fa_decode_workspace_size(2, 4, 8, 1000, 128)
    assert ws > 0 and ws % 256 == 0
    assert lib.fa_decode_workspace_size(1, 1, 17, 1000, 128) == 0  # Nq > 16
    assert lib.fa_decode_workspace_size(1, 1, 4, 1000, 96) == 0

    def dec(Nq=4, Nk=100, d=64, causal=0, w=FAKE * 16, wb=1 << 24, q=FAKE):
        return lib.fa_decode(q, FAKE, FAKE, FAKE, FAKE, 1, 2, Nq, Nk, d, 0.125, causal, w, wb,
                             None)

    assert dec(q=None) == -1
    assert dec(Nq=17) == -2
    assert dec(Nq=8, Nk=4, causal=1) == -2  # causal needs Nk >= Nq
    assert dec(d=32) == -3
    assert dec(w=None) == -6
    assert dec(wb=16) == -6


def test_split_backward_validation(lib):
    """The backward's three kernels called one at a time reject bad arguments
    with the documented codes before anything is launched."""
    pre = lib.fa_backward_preprocess
    assert pre(None, FAKE, FAKE, 1, 1, 128, 64, None) == -1
    assert pre(FAKE, FAKE, None, 1, 1, 128, 64, None) == -1
    assert pre(FAKE, FAKE, FAKE, 1, 1, 0, 64, None) == -2
    assert pre(FAKE, FAKE, FAKE, 1, 1, 128, 96, None) == -3
    assert pre(FAKE, FAKE, FAKE + 4, 1, 1, 128, 64, None) == -4

    def dq(D=FAKE, out=FAKE, d=64, scale=0.125, N=128):
        return lib.fa_backward_dq(FAKE, FAKE, FAKE, FAKE, FAKE, D, out, 1, 2, N, d, scale, 1,
                                  None)

    assert dq(D=None) == -1
    assert dq(out=None) == -1
    assert dq(N=-3) == -2
    assert dq(d=80) == -3
    assert dq(scale=float("nan")) == -2
    assert dq(out=FAKE + 2) == -4

    def dkdv(dk=FAKE, dv=FAKE, D=FAKE, d=128, scale=0.125):
        return lib.fa_backward_dkdv(FAKE, FAKE, FAKE, FAKE, FAKE, D, dk, dv, 1, 2, 256, d, scale,
                                    0, None)

    assert dkdv(dk=None) == -1
    assert dkdv(dv=None) == -1
    assert dkdv(D=None) == -1
    assert dkdv(d=256) == -3
    assert dkdv(scale=0.0) == -2
    assert dkdv(dv=FAKE + 8) == -4


def test_noalloc_validation(lib):
    """fa_backward_noalloc refuses problems its built-in workspace cannot
    hold (more than FA_NOALLOC_MAX_ROWS rows) and bad shapes before it does
    anything else; its remaining checks are fa_backward's."""
    max_rows = 2097152  # FA_NOALLOC_MAX_ROWS in include/fa.h
    hdr = open(os.path.join(ROOT, "include", "fa.h")).read()
    assert f"#define FA_NOALLOC_MAX_ROWS {max_rows}" in hdr

    def na(q=FAKE, B=1, H=2, N=128, d=64):
        return lib.fa_backward_noalloc(q, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, B, H,
                                       N, d, 0.125, 0, None)

    assert na(q=None) == -1
    assert na(B=0) == -2
    assert na(N=-1) == -2
    assert na(d=96) == -3
    assert na(B=1, H=16, N=max_rows // 16 + 1) == -6  # one row too many
    assert na(B=2, H=1 << 10, N=1 << 20) == -6  # rows beyond 2^31


def test_workspace_size_is_linear_in_n(lib):
    f = lib.fa_backward_workspace_size
    assert f(1, 1, 0, 64) == 0
    assert f(1, 1, 128, 96) == 0
    for N in (1000, 4096, 8192, 16384):
        assert f(2, 16, N, 128) == ((2 * 16 * N * 4 + 255) // 256) * 256
    assert f(2, 16, 16384, 128) == 2 * f(2, 16, 8192, 128)


def test_tile_count(lib):
    for N in (1, 127, 128, 129, 1000, 8192):
        nt = -(-N // 128)
        assert fa.fa_forward_tile_count(N, False) == nt * nt
        assert fa.fa_forward_tile_count(N, True) == sum(i + 1 for i in range(nt))


def test_status_strings(lib):
    for s in range(-8, 1):
        assert fa.fa_status_string(s) not in ("", "unknown status")
    assert fa.fa_status_string(-99) == "unknown status"


def test_binding_has_no_fallback(monkeypatch, tmp_path):
    # With the library path pointing nowhere, the binding raises instead of
    # computing anything on another path.
    from exact_io_aware_16_gb300 import _binding
    monkeypatch.setattr(_binding, "_lib", None)
    monkeypatch.setattr(_binding, "_LIB", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        _binding.library()
