"""GPU parity of block-sparse attention (fa_forward_blocksparse /
fa_backward_blocksparse) against the fp64 oracle with the same block mask:
random per-head and shared masks with fully dropped query tiles and key tiles
nobody keeps, causal and not, ragged N; and an all-ones mask, which must give
the dense path's results bit for bit."""
import math

import numpy as np
import pytest
import torch

import oracle
from fa_inputs import make_inputs
from parity import check_bf16, check_lse

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_io_aware_16_gb300 as m
    from exact_io_aware_16_gb300 import build

    build.build()
    m.library()
    return m


def random_mask(rng, heads, nt, density):
    m = (rng.random((heads, nt, nt)) < density).astype(np.uint8)
    if nt > 2:
        m[:, 1, :] = 0  # a query tile with no key tile at all
        m[:, :, nt - 1] = 0  # a key tile no query tile keeps
    return m


CASES = [(1, 2, 600, 64, 0.5, True), (1, 2, 1000, 128, 0.4, False), (2, 1, 777, 128, 0.6, True),
         (1, 1, 300, 64, 0.7, False)]


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("B,H,N,d,density,per_head", CASES,
                         ids=[f"b{c[0]}h{c[1]}n{c[2]}d{c[3]}" for c in CASES])
def test_blocksparse_matches_oracle(fa, B, H, N, d, density, per_head, causal):
    rng = np.random.default_rng(N + d)
    nt = -(-N // 128)
    mask = random_mask(rng, B * H if per_head else 1, nt, density)
    q, k, v, dO = make_inputs(B, H, N, d, seed=N)
    scale = 1.0 / math.sqrt(d)
    dev = torch.device("cuda")
    qd, kd, vd, dOd = (t.to(dev) for t in (q, k, v, dO))
    md = torch.from_numpy(mask if per_head else mask[0]).to(dev)
    o, lse = fa.fa_forward_blocksparse(qd, kd, vd, md, causal=causal, scale=scale)
    dq, dk, dv = fa.fa_backward_blocksparse(qd, kd, vd, o, dOd, lse, md, causal=causal,
                                            scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error()[0] == 0
    o_ref, lse_ref = oracle.forward(q, k, v, scale, causal, mask=mask, block=(128, 128))
    dq_ref, dk_ref, dv_ref, _ = oracle.backward(q, k, v, dO, scale, causal, mask=mask,
                                                block=(128, 128))
    shape = (B, H, N, d)
    check_bf16("O", o.cpu(), o_ref.reshape(shape))
    check_lse("lse", lse.cpu(), lse_ref.reshape(shape[:3]))
    check_bf16("dQ", dq.cpu(), dq_ref.reshape(shape))
    check_bf16("dK", dk.cpu(), dk_ref.reshape(shape))
    check_bf16("dV", dv.cpu(), dv_ref.reshape(shape))


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_all_ones_mask_equals_dense(fa, causal):
    B, H, N, d = 1, 3, 900, 128
    dev = torch.device("cuda")
    q, k, v, dO = (t.to(dev) for t in make_inputs(B, H, N, d, seed=3))
    nt = -(-N // 128)
    ones = torch.ones((nt, nt), dtype=torch.uint8, device=dev)
    o1, l1 = fa.fa_forward(q, k, v, causal=causal)
    o2, l2 = fa.fa_forward_blocksparse(q, k, v, ones, causal=causal)
    g1 = fa.fa_backward(q, k, v, o1, dO, l1, causal=causal)
    g2 = fa.fa_backward_blocksparse(q, k, v, o1, dO, l1, ones, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    for a, b in zip(g1, g2):
        assert torch.equal(a, b)


def test_blocksparse_argument_errors(fa):
    dev = torch.device("cuda")
    q = torch.zeros((1, 1, 256, 64), dtype=torch.bfloat16, device=dev)
    with pytest.raises(ValueError):
        fa.fa_forward_blocksparse(q, q, q, torch.ones((3, 3), dtype=torch.uint8, device=dev))
    lib = fa.library()
    p = q.data_ptr()
    assert lib.fa_forward_blocksparse(p, p, p, p, p, 1, 1, 256, 64, 0.125, 0, None, 0, None) == -1
    assert lib.fa_forward_blocksparse(p, p, p, p, p, 1, 1, 256, 64, 0.125, 0, p, -1, None) == -2
