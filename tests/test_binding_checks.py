"""Host-side checks of the Python binding (no GPU): every wrapper that takes
caller-owned output tensors validates their dtype, shape and contiguity before
anything reaches the library, so a too-small output can never be written past
its end by a kernel.

The binding's device test is replaced by one that accepts CPU tensors, and the
library by a stub that records every call; a rejected call must leave the stub
untouched, an accepted one must reach it (so the checks are not vacuous).
"""
import pytest
import torch

from exact_io_aware_16_gb300 import _binding as bd


class StubLib:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        if not name.startswith("fa_"):
            raise AttributeError(name)

        def fn(*args):
            self.calls.append(name)
            if name.endswith("workspace_size"):
                B, H, N = args[0], args[1], args[2]
                return 4 * B * H * N
            return 0

        return fn


@pytest.fixture
def stub(monkeypatch):
    lib = StubLib()
    monkeypatch.setattr(bd, "library", lambda: lib)
    monkeypatch.setattr(bd, "_on_device", lambda t: True)
    return lib


SHAPE = (1, 2, 130, 64)


def inputs():
    q, k, v, o, dO = (torch.zeros(SHAPE, dtype=torch.bfloat16) for _ in range(5))
    lse = torch.zeros(SHAPE[:3], dtype=torch.float32)
    return q, k, v, o, dO, lse


def bad_outputs():
    """(keyword, tensor) pairs that must each be rejected."""
    short = torch.zeros((1, 2, 129, 64), dtype=torch.bfloat16)
    wrong_dtype = torch.zeros(SHAPE, dtype=torch.float32)
    strided = torch.zeros((1, 2, 64, 130), dtype=torch.bfloat16).transpose(-1, -2)
    return [("short", short), ("dtype", wrong_dtype), ("strided", strided)]


def test_fa_backward_rejects_bad_outputs(stub):
    q, k, v, o, dO, lse = inputs()
    ws = torch.zeros(4096, dtype=torch.uint8)
    for name in ("dq", "dk", "dv"):
        for why, bad in bad_outputs():
            with pytest.raises((TypeError, ValueError)):
                bd.fa_backward(q, k, v, o, dO, lse, workspace=ws, **{name: bad}, stream=0)
    assert [c for c in stub.calls if c == "fa_backward"] == []
    bd.fa_backward(q, k, v, o, dO, lse, workspace=ws, stream=0)
    assert stub.calls[-1] == "fa_backward"


def test_noalloc_rejects_bad_outputs(stub):
    q, k, v, o, dO, lse = inputs()
    for name in ("dq", "dk", "dv"):
        for why, bad in bad_outputs():
            with pytest.raises((TypeError, ValueError)):
                bd.fa_backward_noalloc(q, k, v, o, dO, lse, **{name: bad}, stream=0)
    assert stub.calls == []
    bd.fa_backward_noalloc(q, k, v, o, dO, lse, stream=0)
    assert stub.calls == ["fa_backward_noalloc"]


def test_blocksparse_rejects_bad_outputs(stub):
    q, k, v, o, dO, lse = inputs()
    mask = torch.ones((2, 2), dtype=torch.uint8)
    ws = torch.zeros(4096, dtype=torch.uint8)
    for name in ("dq", "dk", "dv"):
        for why, bad in bad_outputs():
            with pytest.raises((TypeError, ValueError)):
                bd.fa_backward_blocksparse(q, k, v, o, dO, lse, mask, workspace=ws,
                                           stream=0, **{name: bad})
    for why, bad in bad_outputs():
        with pytest.raises((TypeError, ValueError)):
            bd.fa_forward_blocksparse(q, k, v, mask, o=bad, stream=0)
    assert [c for c in stub.calls if not c.endswith("workspace_size")] == []
    bd.fa_backward_blocksparse(q, k, v, o, dO, lse, mask, workspace=ws, stream=0)
    assert stub.calls[-1] == "fa_backward_blocksparse"


def test_split_backward_rejects_bad_outputs(stub):
    q, k, v, o, dO, lse = inputs()
    D = torch.zeros(SHAPE[:3], dtype=torch.float32)
    for why, bad in bad_outputs():
        with pytest.raises((TypeError, ValueError)):
            bd.fa_backward_dq(q, k, v, dO, lse, D, dq=bad, stream=0)
        with pytest.raises((TypeError, ValueError)):
            bd.fa_backward_dkdv(q, k, v, dO, lse, D, dk=bad, stream=0)
        with pytest.raises((TypeError, ValueError)):
            bd.fa_backward_dkdv(q, k, v, dO, lse, D, dv=bad, stream=0)
    assert stub.calls == []
    bd.fa_backward_dq(q, k, v, dO, lse, D, stream=0)
    bd.fa_backward_dkdv(q, k, v, dO, lse, D, stream=0)
    assert stub.calls == ["fa_backward_dq", "fa_backward_dkdv"]


def test_dropout_backward_rejects_bad_outputs(stub):
    q, k, v, o, dO, lse = inputs()
    ws = torch.zeros(4096, dtype=torch.uint8)
    for name in ("dq", "dk", "dv"):
        for why, bad in bad_outputs():
            with pytest.raises((TypeError, ValueError)):
                bd.fa_backward_dropout(q, k, v, o, dO, lse, 0.1, 1, workspace=ws, **{name: bad}, stream=0)
    with pytest.raises(TypeError):
        bd.fa_backward_dropout(q, k, v, o, dO, lse, 0.1, 1,
                               workspace=torch.zeros(4096, dtype=torch.float32), stream=0)
    assert [c for c in stub.calls if c == "fa_backward_dropout"] == []
