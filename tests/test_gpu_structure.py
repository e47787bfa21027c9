"""GPU structural checks of the C ABI path: no writes outside the outputs
(guard bands around every output), bitwise determinism, argument errors on a
real device, clean device error word, and device memory linear in N."""
import math

import pytest
import torch

from fa_inputs import make_inputs

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes of canary on each side of every output


@pytest.fixture(scope="module")
def fa():
    import exact_io_aware_16_gb300 as m
    from exact_io_aware_16_gb300 import build

    build.build()
    m.library()
    return m


def guarded(shape, dtype, dev):
    """A tensor view inside a larger byte buffer whose margins hold a pattern."""
    n = math.prod(shape) * torch.tensor([], dtype=dtype).element_size()
    buf = torch.full((GUARD + n + GUARD,), 0xA5, dtype=torch.uint8, device=dev)
    view = buf[GUARD:GUARD + n].view(dtype).view(shape)
    return buf, view


def intact(buf):
    return bool((buf[:GUARD] == 0xA5).all()) and bool((buf[-GUARD:] == 0xA5).all())


@pytest.mark.parametrize("N,d,causal", [(1, 64, False), (130, 64, True), (300, 128, False),
                                        (257, 128, True)])
def test_outputs_stay_in_bounds(fa, N, d, causal):
    dev = torch.device("cuda")
    B, H = 1, 3
    q, k, v, dO = (t.to(dev) for t in make_inputs(B, H, N, d, seed=5))
    ob, o = guarded((B, H, N, d), torch.bfloat16, dev)
    lb, lse = guarded((B, H, N), torch.float32, dev)
    fa.fa_forward(q, k, v, causal=causal, o=o, lse=lse)
    Db, D = guarded((B, H, N), torch.float32, dev)
    fa.fa_backward_preprocess(o, dO, D)
    kb, dk = guarded((B, H, N, d), torch.bfloat16, dev)
    vb, dv = guarded((B, H, N, d), torch.bfloat16, dev)
    qb, dq = guarded((B, H, N, d), torch.bfloat16, dev)
    fa.fa_backward_dq(q, k, v, dO, lse, D, causal=causal, dq=dq)
    fa.fa_backward_dkdv(q, k, v, dO, lse, D, causal=causal, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error()[0] == 0
    for name, b in (("o", ob), ("lse", lb), ("D", Db), ("dk", kb), ("dv", vb), ("dq", qb)):
        assert intact(b), f"{name}: write outside the tensor"


def test_wait_timeout_is_reported_then_cleared(fa):
    """A kernel waiting on a barrier nothing arrives on gives up after the
    bounded wait's limit (2 s) instead of hanging; the error comes back once
    through fa_get_device_error and the context keeps working."""
    import time

    assert fa.fa_get_device_error()[0] == 0
    t0 = time.time()
    fa.fa_selftest_wait_timeout()
    st, detail = fa.fa_get_device_error()
    waited = time.time() - t0
    assert st == -8 and detail == 0x800007E0, (st, hex(detail))
    assert 1.0 < waited < 60.0
    assert fa.fa_get_device_error() == (0, 0)
    dev = torch.device("cuda")
    q, k, v, dO = (t.to(dev) for t in make_inputs(1, 2, 300, 64, seed=4))
    o, lse = fa.fa_forward(q, k, v, causal=True)
    fa.fa_backward(q, k, v, o, dO, lse, causal=True)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error()[0] == 0


def test_deterministic(fa):
    dev = torch.device("cuda")
    q, k, v, dO = (t.to(dev) for t in make_inputs(2, 4, 1000, 128, seed=9))
    outs = []
    for _ in range(2):
        o, lse = fa.fa_forward(q, k, v, causal=True)
        dq, dk, dv = fa.fa_backward(q, k, v, o, dO, lse, causal=True)
        torch.cuda.synchronize()
        outs.append([t.clone() for t in (o, lse, dq, dk, dv)])
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_errors_on_device(fa):
    dev = torch.device("cuda")
    q = torch.zeros((1, 1, 128, 96), dtype=torch.bfloat16, device=dev)
    with pytest.raises(fa.FaError) as e:
        fa.fa_forward(q, q, q)
    assert e.value.status == -3
    q = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16, device=dev)
    lib = fa.library()
    # N = 0 (empty input) is rejected, nothing is launched
    assert lib.fa_forward(q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(), q.data_ptr(),
                          1, 1, 0, 64, 0.125, 0, None) == -2
    # misaligned view
    flat = torch.zeros(128 * 64 + 8, dtype=torch.bfloat16, device=dev)
    mis = flat[1:1 + 128 * 64].view(1, 1, 128, 64)
    with pytest.raises(fa.FaError) as e:
        fa.fa_forward(mis, q, q)
    assert e.value.status == -4
    assert fa.fa_get_device_error()[0] == 0


def test_memory_linear_in_n(fa):
    """Beyond inputs and outputs, the backward needs only its fp32 [B,H,N]
    workspace, so device memory grows linearly with N; the library itself
    allocates nothing.  Measured two ways: PyTorch's allocator statistics
    (nothing allocated through PyTorch) and the device's free memory from
    cudaMemGetInfo, which would also show a cudaMalloc made inside libfa.so.
    Each size runs once untimed first, so that the first launch of each kernel
    (module loading) is not counted."""
    dev = torch.device("cuda")
    extra = []
    for N in (2048, 4096, 8192):
        q, k, v, dO = (t.to(dev) for t in make_inputs(1, 4, N, 128, seed=1))
        o = torch.empty_like(q)
        lse = torch.empty((1, 4, N), dtype=torch.float32, device=dev)
        dq, dk, dv = (torch.empty_like(q) for _ in range(3))
        ws = torch.empty(fa.fa_backward_workspace_size(1, 4, N, 128), dtype=torch.uint8,
                         device=dev)

        def step():
            fa.fa_forward(q, k, v, causal=True, o=o, lse=lse)
            fa.fa_backward(q, k, v, o, dO, lse, causal=True, dq=dq, dk=dk, dv=dv, workspace=ws)

        step()
        torch.cuda.synchronize()
        torch.cuda.reset_peak_memory_stats()
        base = torch.cuda.memory_allocated()
        free_before = torch.cuda.mem_get_info(dev)[0]
        step()
        torch.cuda.synchronize()
        free_after = torch.cuda.mem_get_info(dev)[0]
        extra.append(torch.cuda.max_memory_allocated() - base)
        assert free_after == free_before, (N, free_before - free_after)
        assert ws.numel() == 4 * 4 * N
    # the library itself allocates nothing
    assert extra == [0, 0, 0]
