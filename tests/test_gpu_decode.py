"""GPU parity of the decode step (fa_decode: a few query rows against a long
key/value cache, split over the key axis and merged by the online-softmax
update) against the fp64 oracle's decode definition."""
import math

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


CASES = [
    (2, 4, 1, 1000, 128, False),
    (2, 4, 1, 1000, 128, True),
    (1, 8, 16, 4097, 64, True),
    (1, 2, 7, 300, 128, False),
    (1, 2, 7, 300, 128, True),
    (1, 1, 16, 16, 128, True),
    (3, 1, 3, 1, 64, False),
    (1, 4, 8, 20000, 128, True),
    (1, 3, 4, 1000, 128, True),     # the first query count on the tensor core
    (2, 2, 5, 1000, 64, False),
    (1, 2, 16, 129, 128, True),     # a 64-key tile with one key in it
    (4, 80, 6, 3000, 128, True),    # more heads than CTA slots: one range per head
    (1, 1, 12, 65536, 64, True),
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", CASES,
                         ids=[f"b{c[0]}h{c[1]}q{c[2]}k{c[3]}d{c[4]}{'c' if c[5] else ''}"
                              for c in CASES])
def test_decode_matches_oracle(fa, B, H, Nq, Nk, d, causal):
    q, _, _, _ = make_inputs(B, H, Nq, d, seed=Nk + Nq, with_dO=False)
    _, k, v, _ = make_inputs(B, H, Nk, d, seed=Nk, with_dO=False)
    scale = 1.0 / math.sqrt(d)
    dev = torch.device("cuda")
    o, lse = fa.fa_decode(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error()[0] == 0
    o_ref, lse_ref = oracle.decode(q, k, v, scale, causal)
    check_bf16("O", o.cpu(), o_ref.reshape(B, H, Nq, d))
    check_lse("lse", lse.cpu(), lse_ref.reshape(B, H, Nq))


def test_decode_equals_forward_last_rows(fa):
    """The decode of the last Nq rows equals those rows of the causal forward."""
    B, H, N, d, Nq = 1, 2, 700, 128, 9
    dev = torch.device("cuda")
    q, k, v, _ = (t.to(dev) if t is not None else None
                  for t in make_inputs(B, H, N, d, seed=4, with_dO=False))
    o, lse = fa.fa_forward(q, k, v, causal=True)
    od, lsed = fa.fa_decode(q[:, :, N - Nq:].contiguous(), k, v, causal=True)
    torch.cuda.synchronize()
    ref = o[:, :, N - Nq:].float()
    assert (od.float() - ref).abs().max().item() < 2e-2
    assert (lsed - lse[:, :, N - Nq:]).abs().max().item() < 1e-4
