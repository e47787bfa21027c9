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


def every_call(q, k, v, o, dO, lse):
    """One accepted call of every launching wrapper: (library function, thunk)."""
    D = torch.zeros(SHAPE[:3], dtype=torch.float32)
    ws = torch.zeros(4096, dtype=torch.uint8)
    mask = torch.ones((2, 2), dtype=torch.uint8)
    B, H, N, d = SHAPE
    q8, k8 = (torch.zeros((B, H, 128, 128), dtype=torch.uint8) for _ in range(2))
    vt8 = torch.zeros((B, H, 128, 128), dtype=torch.uint8)
    qd = torch.zeros((B, H, 4, d), dtype=torch.bfloat16)
    return [
        ("fa_forward", lambda: bd.fa_forward(q, k, v, stream=0)),
        ("fa_forward_blocksparse", lambda: bd.fa_forward_blocksparse(q, k, v, mask, stream=0)),
        ("fa_forward_dropout", lambda: bd.fa_forward_dropout(q, k, v, 0.1, 7, stream=0)),
        ("fa_forward_fp8", lambda: bd.fa_forward_fp8(q8, k8, vt8, 1.0, 1.0, 1.0, stream=0)),
        ("fa_decode", lambda: bd.fa_decode(qd, k, v, workspace=ws, stream=0)),
        ("fa_backward_preprocess", lambda: bd.fa_backward_preprocess(o, dO, stream=0)),
        ("fa_backward", lambda: bd.fa_backward(q, k, v, o, dO, lse, workspace=ws, stream=0)),
        ("fa_backward_blocksparse",
         lambda: bd.fa_backward_blocksparse(q, k, v, o, dO, lse, mask, workspace=ws, stream=0)),
        ("fa_backward_dropout",
         lambda: bd.fa_backward_dropout(q, k, v, o, dO, lse, 0.1, 7, workspace=ws, stream=0)),
        ("fa_backward_noalloc", lambda: bd.fa_backward_noalloc(q, k, v, o, dO, lse, stream=0)),
        ("fa_backward_dq", lambda: bd.fa_backward_dq(q, k, v, dO, lse, D, stream=0)),
        ("fa_backward_dkdv", lambda: bd.fa_backward_dkdv(q, k, v, dO, lse, D, stream=0)),
    ]


def test_every_wrapper_reaches_its_library_function(stub):
    """Each wrapper marshals its arguments all the way to the C function of
    the same name (a typo in any wrapper shows here, not first on a GPU)."""
    for name, call in every_call(*inputs()):
        call()
        assert [c for c in stub.calls if not c.endswith("workspace_size")][-1] == name


def test_tensors_on_another_gpu_are_rejected(stub, monkeypatch):
    """A tensor on a GPU other than q's is refused before the library is
    called, for every wrapper and every tensor argument it passes on."""
    q, k, v, o, dO, lse = inputs()
    for other in (k, v, o, dO, lse):
        # -1 (a CPU tensor's index) for the rest: accepted calls switch no device
        monkeypatch.setattr(bd, "_device_index", lambda t: 1 if t is other else -1)
        rejected = set()
        for name, call in every_call(q, k, v, o, dO, lse):
            before = list(stub.calls)
            try:
                call()
            except ValueError as e:
                assert "device" in str(e)
                assert [c for c in stub.calls if c == name] == \
                    [c for c in before if c == name], name
                rejected.add(name)
            else:  # the wrapper does not take `other` (e.g. the forward and o, dO)
                assert stub.calls[-1] == name
        assert "fa_backward" in rejected  # it takes every one of them


def test_call_runs_with_the_tensors_device_current(stub, monkeypatch):
    """The library launches on the current device: a call whose tensors are
    on device 1 while device 0 is current runs with device 1 made current,
    and a call on the current device switches nothing."""
    current = {"dev": 0}
    seen = []

    class SwitchTo:
        def __init__(self, dev):
            self.dev = dev

        def __enter__(self):
            self.prev, current["dev"] = current["dev"], self.dev

        def __exit__(self, *exc):
            current["dev"] = self.prev

    monkeypatch.setattr(bd.torch.cuda, "current_device", lambda: current["dev"])
    monkeypatch.setattr(bd.torch.cuda, "device", SwitchTo)
    real_fn = StubLib.__getattr__

    def recording(self, name):
        fn = real_fn(self, name)
        return lambda *a: (seen.append((name, current["dev"])), fn(*a))[1]

    monkeypatch.setattr(StubLib, "__getattr__", recording)
    for dev in (1, 0):
        monkeypatch.setattr(bd, "_device_index", lambda t, dev=dev: dev)
        for name, call in every_call(*inputs()):
            seen.clear()
            call()
            assert (name, dev) in seen, (name, dev, seen)
            assert current["dev"] == 0
