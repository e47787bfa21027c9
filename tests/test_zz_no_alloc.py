"""fa_backward_noalloc: the backward pass for callers that cannot allocate
device memory (a runtime that owns all device memory through its own pool, a
plugin interface that passes only tensors and a stream, or a loop that cannot
take cudaMalloc's implicit device synchronisation).  Its workspace is a fixed
array inside the library instead of caller memory.

Checked through the C ABI against fa_backward (caller workspace) on the same
inputs, within the parity tolerances, on two calls in a row (the second call
finds the first call's contents in the shared array).  This file sorts last so
that a run stopping at its first failure has already run every other test.
"""
import ctypes
import math

import pytest
import torch

from fa_inputs import make_inputs
from parity import check_bf16, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_io_aware_16_gb300 as m
    from exact_io_aware_16_gb300 import build

    build.build()
    m.library()
    return m


def call_noalloc(lib, q, k, v, o, dO, lse, dq, dk, dv, causal, scale, stream):
    B, H, N, d = q.shape
    return lib.fa_backward_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dO.data_ptr(), lse.data_ptr(),
        dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d, ctypes.c_float(scale),
        int(causal), ctypes.c_void_p(stream))


@pytest.mark.parametrize("B,H,N,d,causal", [(2, 4, 1000, 128, True), (1, 8, 640, 64, False)])
def test_noalloc_matches_fa_backward(fa, B, H, N, d, causal):
    dev = torch.device("cuda")
    lib = fa.library()
    scale = 1.0 / math.sqrt(d)
    stream = torch.cuda.current_stream().cuda_stream
    q, k, v, dO = (t.to(dev) for t in make_inputs(B, H, N, d, seed=11))
    o, lse = fa.fa_forward(q, k, v, causal=causal, scale=scale)
    ref = fa.fa_backward(q, k, v, o, dO, lse, causal=causal, scale=scale)
    torch.cuda.synchronize()
    for call in range(2):
        dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
        before = torch.cuda.memory_allocated()
        st = call_noalloc(lib, q, k, v, o, dO, lse, dq, dk, dv, causal, scale, stream)
        assert st == 0, fa.fa_status_string(st)
        assert torch.cuda.memory_allocated() == before
        torch.cuda.synchronize()
        assert fa.fa_get_device_error()[0] == 0
        for name, got, want in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
            check_bf16(f"{name} call {call + 1}", got, to_np(want))


def test_noalloc_rejects_oversize(fa):
    lib = fa.library()
    dev = torch.device("cuda")
    t = torch.zeros(16, dtype=torch.bfloat16, device=dev)
    p = t.data_ptr()
    # B*H*N = 2,097,153 rows is one past the built-in limit
    st = lib.fa_backward_noalloc(p, p, p, p, p, p, p, p, p, 1, 3, 699051, 64,
                                 ctypes.c_float(0.125), 0, None)
    assert st == -6  # FA_ERR_WORKSPACE, nothing launched
    assert fa.fa_get_device_error()[0] == 0
