"""GPU check of a problem larger than 2^31 elements per tensor.

B=1, H=16400, N=1024, d=128: 2,149,580,800 elements (4.3 GB) per tensor, so
the last head starts past element 2^31 and past byte 2^32.  Every head holds
the same seeded inputs (heads are independent problems), so every head's
outputs must equal head 0's bit for bit (the kernels are deterministic), and
the last head is checked in full against the fp64 oracle.  About 36 GB of
device memory.
"""
import math

import pytest
import torch

import oracle
from fa_inputs import make_inputs
from parity import check_bf16, check_lse

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

B, H, N, D = 1, 16400, 1024, 128


@pytest.fixture(scope="module")
def fa():
    import exact_io_aware_16_gb300 as m
    from exact_io_aware_16_gb300 import build

    build.build()
    m.library()
    return m


def all_heads_equal(t):
    flat = t.view(B * H, -1)
    return bool((flat == flat[:1]).all())


def test_beyond_2_31_elements(fa):
    assert B * H * N * D > 2 ** 31 and (B * H - 1) * N * D > 2 ** 31
    dev = torch.device("cuda")
    scale = 1.0 / math.sqrt(D)
    head = make_inputs(1, 1, N, D, seed=21)
    q, k, v, dO = (t.to(dev).expand(B, H, N, D).contiguous() for t in head)
    o, lse = fa.fa_forward(q, k, v, causal=True, scale=scale)
    dq, dk, dv = fa.fa_backward(q, k, v, o, dO, lse, causal=True, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error()[0] == 0
    del q, k, v, dO
    for name, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
        assert all_heads_equal(t), f"{name}: heads differ"
    last = {n: t[0, H - 1].cpu() for n, t in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk),
                                               ("dv", dv))}
    q1, k1, v1, dO1 = head
    o_ref, lse_ref = oracle.forward(q1, k1, v1, scale, True)
    dq_ref, dk_ref, dv_ref, _ = oracle.backward(q1, k1, v1, dO1, scale, True)
    report = []
    check_bf16("O[last head]", last["o"], o_ref.reshape(N, D), report)
    check_lse("lse[last head]", last["lse"], lse_ref.reshape(N), report)
    check_bf16("dQ[last head]", last["dq"], dq_ref.reshape(N, D), report)
    check_bf16("dK[last head]", last["dk"], dk_ref.reshape(N, D), report)
    check_bf16("dV[last head]", last["dv"], dv_ref.reshape(N, D), report)
    print("b1h16400n1024d128 causal;", "; ".join(report))
