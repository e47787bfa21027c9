"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded bf16 inputs, element by element.

Small shapes that span several 128-row tiles and a ragged tail are checked in
full, forward and backward, causal and not.  The benchmark workloads are
checked in full (the 8K workload too, in about 100 s of oracle time), except
the 32K one, which is checked on seeded samples of rows (O, lse, dQ) and key
rows (dK, dV) computed one by one by the oracle.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from fa_inputs import WORKLOADS, make_inputs, sample_indices
from parity import check_bf16, check_lse

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_io_aware_16_gb300 as m
    from exact_io_aware_16_gb300 import build

    build.build()
    m.library()
    return m


def run_gpu(fa, q, k, v, dO, causal, scale, backward=True):
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o, lse = fa.fa_forward(qd, kd, vd, causal=causal, scale=scale)
    out = {"o": o, "lse": lse}
    if backward:
        dOd = dO.to(dev)
        dq, dk, dv = fa.fa_backward(qd, kd, vd, o, dOd, lse, causal=causal, scale=scale)
        out.update(dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    st, detail = fa.fa_get_device_error()
    assert st == 0, f"device error {st} detail {detail:#x}"
    return {k_: t.cpu() for k_, t in out.items()}


SMALL = [
    (1, 1, 1, 64),
    (1, 2, 17, 64),
    (2, 1, 129, 128),
    (1, 1, 200, 64),
    (1, 2, 256, 128),
    (1, 1, 383, 128),
    (2, 2, 640, 64),
    (1, 1, 1000, 128),
]


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("B,H,N,d", SMALL, ids=[f"b{b}h{h}n{n}d{d}" for b, h, n, d in SMALL])
def test_small_shapes_full(fa, B, H, N, d, causal):
    q, k, v, dO = make_inputs(B, H, N, d, seed=N * 7 + d)
    scale = 1.0 / math.sqrt(d)
    g = run_gpu(fa, q, k, v, dO, causal, scale)
    o_ref, lse_ref = oracle.forward(q, k, v, scale, causal)
    dq_ref, dk_ref, dv_ref, _ = oracle.backward(q, k, v, dO, scale, causal)
    check_bf16("O", g["o"], o_ref.reshape(B, H, N, d))
    check_lse("lse", g["lse"], lse_ref.reshape(B, H, N))
    check_bf16("dQ", g["dq"], dq_ref.reshape(B, H, N, d))
    check_bf16("dK", g["dk"], dk_ref.reshape(B, H, N, d))
    check_bf16("dV", g["dv"], dv_ref.reshape(B, H, N, d))


def full_check(fa, w, causal):
    q, k, v, dO = make_inputs(w.B, w.H, w.N, w.d, w.seed, w.qk_mult, with_dO=w.backward)
    g = run_gpu(fa, q, k, v, dO, causal, w.scale, backward=w.backward)
    shape = (w.B, w.H, w.N, w.d)
    report = []
    o_ref, lse_ref = oracle.forward(q, k, v, w.scale, causal)
    check_bf16("O", g["o"], o_ref.reshape(shape), report)
    check_lse("lse", g["lse"], lse_ref.reshape(shape[:3]), report)
    if w.backward:
        dq_ref, dk_ref, dv_ref, _ = oracle.backward(q, k, v, dO, w.scale, causal)
        check_bf16("dQ", g["dq"], dq_ref.reshape(shape), report)
        check_bf16("dK", g["dk"], dk_ref.reshape(shape), report)
        check_bf16("dV", g["dv"], dv_ref.reshape(shape), report)
    print(w.name, "causal" if causal else "full", "; ".join(report))


def test_workload_fwd_b1h2n256d64(fa):
    full_check(fa, WORKLOADS["fwd_b1h2n256d64"], False)


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_workload_b4h16n2048d64(fa, causal):
    full_check(fa, WORKLOADS["b4h16n2048d64"], causal)


def test_workload_short_b64h12n512d64(fa):
    full_check(fa, WORKLOADS["short_b64h12n512d64"], False)


def sampled_check(fa, w, causal, rows_per_head, dkdv_heads, keys_per_head):
    q, k, v, dO = make_inputs(w.B, w.H, w.N, w.d, w.seed, w.qk_mult)
    g = run_gpu(fa, q, k, v, dO, causal, w.scale)
    BH, N, d = w.BH, w.N, w.d
    report = []
    must = (0, 127, 128, N - 1)
    rows = []
    for h in range(BH):
        rows += [h * N + i for i in sample_indices(N, rows_per_head, seed=1 + h, must=must)]
    rows = np.array(rows, dtype=np.int64)
    o_ref, lse_ref = oracle.forward(q, k, v, w.scale, causal, rows=rows)
    check_bf16("O[sampled rows]", g["o"].reshape(-1, d)[rows], o_ref, report)
    check_lse("lse[sampled rows]", g["lse"].reshape(-1)[rows], lse_ref, report)
    dq_ref, *_ = oracle.backward_rows(q, k, v, dO, w.scale, causal, rows=rows)
    check_bf16("dQ[sampled rows]", g["dq"].reshape(-1, d)[rows], dq_ref, report)
    # dK / dV of sampled key rows need m, l, D of every row of their head
    heads = sample_indices(BH, dkdv_heads, seed=2)
    m_all = np.full(BH * N, np.nan)
    l_all = np.full(BH * N, np.nan)
    D_all = np.full(BH * N, np.nan)
    cols = []
    for h in heads:
        hr = np.arange(h * N, (h + 1) * N, dtype=np.int64)
        _, m, l, D, _ = oracle.backward_rows(q, k, v, dO, w.scale, causal, rows=hr)
        m_all[hr], l_all[hr], D_all[hr] = m, l, D
        cols += [h * N + j for j in sample_indices(N, keys_per_head, seed=3 + h, must=must)]
    cols = np.array(cols, dtype=np.int64)
    dk_ref, dv_ref = oracle.backward_cols(q, k, v, dO, m_all, l_all, D_all, w.scale, causal,
                                          cols=cols)
    check_bf16("dK[sampled keys]", g["dk"].reshape(-1, d)[cols], dk_ref, report)
    check_bf16("dV[sampled keys]", g["dv"].reshape(-1, d)[cols], dv_ref, report)
    print(w.name, "; ".join(report))


@pytest.mark.slow
def test_workload_causal_b2h16n8192d128(fa):
    """The long-context workload in full: every row of O, lse and dQ and every
    key of dK and dV of all 32 heads against the fp64 oracle (about 10^12
    fp64 operations, some 100 s on 16 host cores)."""
    full_check(fa, WORKLOADS["causal_b2h16n8192d128"], True)


@pytest.mark.slow
def test_workload_causal_b1h32n32768d128_qk2(fa):
    sampled_check(fa, WORKLOADS["causal_b1h32n32768d128_qk2"], True, rows_per_head=256,
                  dkdv_heads=4, keys_per_head=256)
