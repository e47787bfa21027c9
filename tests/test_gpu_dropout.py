"""GPU parity of dropout on P (fa_forward_dropout / fa_backward_dropout)
against the fp64 oracle replaying the same Philox4x32-10 keep matrix.

* small shapes spanning several tiles and a ragged tail, causal and not,
  several probabilities, seeds and offsets: O, lse, dQ, dK, dV element by
  element (max-abs bound 2e-2 / q, q the keep probability, since every kept
  term carries 1/q before it is rounded; rel-L2 1e-2 and lse 1e-4 as
  without dropout);
* the keep decisions themselves, bit for bit: with V the identity, the zero
  pattern of O is the dropped pattern of Z (an integer result: exact);
* p = 0 gives the plain path's results bit for bit; the same (seed, offset)
  gives the same bits twice, another offset another mask;
* dropout on top of a block mask;
* the benchmark workload (B2 H16 N8192 d128 causal, p = 0.1) on sampled rows
  and key rows.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from fa_inputs import WORKLOADS, make_inputs, sample_indices
from parity import check_bf16, check_lse

from oracle import dropout_params


def _check_all(o, lse, dq, dk, dv, refs, shape, p, report=None):
    """Compare against the oracle; max-abs bounds scaled by 1/q = rs."""
    o_ref, lse_ref, dq_ref, dk_ref, dv_ref = refs
    rs = dropout_params(p)[1]
    check_bf16("O", o.cpu(), o_ref.reshape(shape), report, abs_scale=rs)
    check_lse("lse", lse.cpu(), lse_ref.reshape(shape[:3]), report)
    check_bf16("dQ", dq.cpu(), dq_ref.reshape(shape), report, abs_scale=rs)
    check_bf16("dK", dk.cpu(), dk_ref.reshape(shape), report, abs_scale=rs)
    check_bf16("dV", dv.cpu(), dv_ref.reshape(shape), report, abs_scale=rs)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_io_aware_16_gb300 as m
    from exact_io_aware_16_gb300 import build

    build.build()
    m.library()
    return m


def _dev(*ts):
    dev = torch.device("cuda")
    return [t.to(dev) for t in ts]


CASES = [  # B, H, N, d, p, seed, offset
    (1, 2, 200, 64, 0.1, 1, 0),
    (2, 1, 383, 128, 0.5, 2**40 + 7, 3),
    (1, 2, 640, 64, 0.25, 12345, 1),
    (1, 1, 1000, 128, 0.1, 0xDEADBEEFCAFEF00D, 2**31 + 5),
]


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("B,H,N,d,p,seed,offset", CASES,
                         ids=[f"b{c[0]}h{c[1]}n{c[2]}d{c[3]}p{c[4]}" for c in CASES])
def test_dropout_matches_oracle(fa, B, H, N, d, p, seed, offset, causal):
    q, k, v, dO = make_inputs(B, H, N, d, seed=N + 11)
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd, dOd = _dev(q, k, v, dO)
    o, lse = fa.fa_forward_dropout(qd, kd, vd, p, seed, offset, causal=causal, scale=scale)
    dq, dk, dv = fa.fa_backward_dropout(qd, kd, vd, o, dOd, lse, p, seed, offset, causal=causal,
                                        scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error()[0] == 0
    drop = (p, seed, offset)
    o_ref, lse_ref = oracle.forward(q, k, v, scale, causal, dropout=drop)
    dq_ref, dk_ref, dv_ref, _ = oracle.backward(q, k, v, dO, scale, causal, dropout=drop)
    report = []
    _check_all(o, lse, dq, dk, dv, (o_ref, lse_ref, dq_ref, dk_ref, dv_ref), (B, H, N, d), p,
               report)
    print(B, H, N, d, p, "causal" if causal else "full", "; ".join(report))


@pytest.mark.parametrize("p,seed,offset", [(0.3, 99, 0), (0.9, 2**63 + 1, 77)])
def test_keep_pattern_is_exact(fa, p, seed, offset):
    """V = I (N = d = 128, non-causal): O_ij = P_ij Z_ij / (1 - p) / 1, so O
    is zero exactly where Z drops; compare that pattern bit for bit, for
    every head, with the oracle's Philox replay."""
    B, H, N, d = 1, 3, 128, 128
    q, k, _, _ = make_inputs(B, H, N, d, seed=4)
    q, k = q * 0.25, k * 0.25  # keep every P_ij well above bf16 underflow
    eye = torch.eye(N, dtype=torch.bfloat16).expand(B, H, N, N).contiguous()
    qd, kd, vd = _dev(q.to(torch.bfloat16), k.to(torch.bfloat16), eye)
    o, _ = fa.fa_forward_dropout(qd, kd, vd, p, seed, offset)
    torch.cuda.synchronize()
    got = (o.cpu().reshape(B * H, N, N) != 0).numpy()
    for bh in range(B * H):
        want = oracle.dropout_keep(p, seed, offset, bh, N, N)
        assert np.array_equal(got[bh], want), f"head {bh}: {int((got[bh] != want).sum())} bits"
    assert abs(got.mean() - (1 - p)) < 0.02


def test_p_zero_is_plain_path(fa):
    B, H, N, d = 1, 2, 700, 128
    q, k, v, dO = _dev(*make_inputs(B, H, N, d, seed=5))
    for causal in (False, True):
        o1, l1 = fa.fa_forward(q, k, v, causal=causal)
        o2, l2 = fa.fa_forward_dropout(q, k, v, 0.0, 123, 4, causal=causal)
        g1 = fa.fa_backward(q, k, v, o1, dO, l1, causal=causal)
        g2 = fa.fa_backward_dropout(q, k, v, o1, dO, l1, 0.0, 123, 4, causal=causal)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
        for a, b in zip(g1, g2):
            assert torch.equal(a, b)


def test_replay_and_independence(fa):
    B, H, N, d = 2, 2, 512, 64
    q, k, v, dO = _dev(*make_inputs(B, H, N, d, seed=6))
    runs = []
    for off in (10, 10, 11):
        o, l = fa.fa_forward_dropout(q, k, v, 0.2, 42, off, causal=True)
        g = fa.fa_backward_dropout(q, k, v, o, dO, l, 0.2, 42, off, causal=True)
        torch.cuda.synchronize()
        runs.append([t.clone() for t in (o, l, *g)])
    for a, b in zip(runs[0], runs[1]):
        assert torch.equal(a, b)
    assert torch.equal(runs[0][1], runs[2][1])  # lse does not depend on the mask
    assert not torch.equal(runs[0][0], runs[2][0])


def test_dropout_with_block_mask(fa):
    B, H, N, d, p, seed, off = 1, 2, 600, 64, 0.2, 5, 9
    rng = np.random.default_rng(1)
    nt = -(-N // 128)
    mask = (rng.random((B * H, nt, nt)) < 0.6).astype(np.uint8)
    mask[:, 1, :] = 0
    q, k, v, dO = make_inputs(B, H, N, d, seed=7)
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd, dOd = _dev(q, k, v, dO)
    md = torch.from_numpy(mask).cuda()
    for causal in (False, True):
        o, lse = fa.fa_forward_dropout(qd, kd, vd, p, seed, off, causal=causal, scale=scale,
                                       block_mask=md)
        dq, dk, dv = fa.fa_backward_dropout(qd, kd, vd, o, dOd, lse, p, seed, off,
                                            causal=causal, scale=scale, block_mask=md)
        torch.cuda.synchronize()
        assert fa.fa_get_device_error()[0] == 0
        kw = dict(mask=mask, block=(128, 128), dropout=(p, seed, off))
        o_ref, lse_ref = oracle.forward(q, k, v, scale, causal, **kw)
        dq_ref, dk_ref, dv_ref, _ = oracle.backward(q, k, v, dO, scale, causal, **kw)
        _check_all(o, lse, dq, dk, dv, (o_ref, lse_ref, dq_ref, dk_ref, dv_ref),
                   (B, H, N, d), p)


def test_bad_probability_rejected(fa):
    q, k, v, _ = _dev(*make_inputs(1, 1, 128, 64, seed=1))
    for p in (-0.1, 1.0, float("nan")):
        with pytest.raises(fa.FaError) as e:
            fa.fa_forward_dropout(q, k, v, p, 1, 0)
        assert e.value.status == -2


@pytest.mark.slow
def test_workload_causal_b2h16n8192d128_dropout(fa):
    """The benchmark workload with p = 0.1, on sampled rows (O, lse, dQ) of
    every head and sampled key rows (dK, dV) of two heads."""
    w = WORKLOADS["causal_b2h16n8192d128"]
    p, seed, off = 0.1, 2024, 0
    drop = (p, seed, off)
    q, k, v, dO = make_inputs(w.B, w.H, w.N, w.d, w.seed, w.qk_mult)
    qd, kd, vd, dOd = _dev(q, k, v, dO)
    o, lse = fa.fa_forward_dropout(qd, kd, vd, p, seed, off, causal=True, scale=w.scale)
    dq, dk, dv = fa.fa_backward_dropout(qd, kd, vd, o, dOd, lse, p, seed, off, causal=True,
                                        scale=w.scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error()[0] == 0
    o, lse, dq, dk, dv = (t.cpu() for t in (o, lse, dq, dk, dv))
    BH, N, d = w.BH, w.N, w.d
    must = (0, 127, 128, N - 1)
    rows = []
    for h in range(BH):
        rows += [h * N + i for i in sample_indices(N, 32, seed=1 + h, must=must)]
    rows = np.array(rows, dtype=np.int64)
    report = []
    rs = dropout_params(p)[1]
    o_ref, lse_ref = oracle.forward(q, k, v, w.scale, True, rows=rows, dropout=drop)
    check_bf16("O[sampled rows]", o.reshape(-1, d)[rows], o_ref, report, abs_scale=rs)
    check_lse("lse[sampled rows]", lse.reshape(-1)[rows], lse_ref, report)
    dq_ref, *_ = oracle.backward_rows(q, k, v, dO, w.scale, True, rows=rows, dropout=drop)
    check_bf16("dQ[sampled rows]", dq.reshape(-1, d)[rows], dq_ref, report, abs_scale=rs)
    heads = sample_indices(BH, 2, seed=2)
    m_all, l_all, D_all = (np.full(BH * N, np.nan) for _ in range(3))
    cols = []
    for h in heads:
        hr = np.arange(h * N, (h + 1) * N, dtype=np.int64)
        _, m, l, D, _ = oracle.backward_rows(q, k, v, dO, w.scale, True, rows=hr, dropout=drop)
        m_all[hr], l_all[hr], D_all[hr] = m, l, D
        cols += [h * N + j for j in sample_indices(N, 96, seed=3 + h, must=must)]
    cols = np.array(cols, dtype=np.int64)
    dk_ref, dv_ref = oracle.backward_cols(q, k, v, dO, m_all, l_all, D_all, w.scale, True,
                                          cols=cols, dropout=drop)
    check_bf16("dK[sampled keys]", dk.reshape(-1, d)[cols], dk_ref, report, abs_scale=rs)
    check_bf16("dV[sampled keys]", dv.reshape(-1, d)[cols], dv_ref, report, abs_scale=rs)
    print(w.name, "dropout", "; ".join(report))
