"""GPU parity of the e4m3 forward (fa_forward_fp8) against the fp64 oracle run
on the dequantised inputs (the exact attention the FP8 path approximates).

Tolerance, derived from the arithmetic of the path.  With e4m3 inputs the
score products are exact in fp32 and the softmax statistics are kept in
fp32; the one approximation is the rounding of each unnormalised probability
P~_j (<= 2^8, relative to the running max) to e4m3 before the P V product:
|err| <= 2^-4 P~_j for normal values and <= 2^-10 below 2^-6.  Carried
through O = sum_j P^_j v_j / L with L >= l (the row sum against the true
max, itself >= 1):

    |O_ic - ref_ic| <= 2^-4 (P|V|)_ic + 2^-10 sum_{j visible} |v_jc| / l_i
                       + half a bf16 ulp of ref_ic + 1e-3

(P|V| is the oracle's attention with |v| in place of v; l_i its row sum;
1e-3 covers fp32 accumulation and exp2).  lse comes from fp32 scores of
exact products: 1e-4 as for bf16 inputs.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from fa_inputs import dequantize, make_fp8_inputs, sample_indices
from parity import bf16_ulp, check_lse, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_io_aware_16_gb300 as m
    from exact_io_aware_16_gb300 import build

    build.build()
    m.library()
    return m


def run_fp8(fa, q8, k8, vt8, ds, causal, scale):
    dev = torch.device("cuda")
    qd, kd, vtd = (t.view(torch.uint8).to(dev) for t in (q8, k8, vt8))
    o, lse = fa.fa_forward_fp8(qd, kd, vtd, *ds, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_get_device_error()[0] == 0
    return o.cpu(), lse.cpu()


def fp8_bound(q, k, v, scale, causal, rows=None):
    """Per-element bound of the e4m3 path (module docstring) and the
    reference O, lse for the selected rows."""
    BH, N, d = q.shape[0] * q.shape[1], q.shape[2], q.shape[3]
    o_ref, lse_ref = oracle.forward(q, k, v, scale, causal, rows=rows)
    pv_abs, _ = oracle.forward(q, k, v.abs(), scale, causal, rows=rows)
    zero = torch.zeros_like(q)
    _, m, l, _, _ = oracle.backward_rows(q, k, v, zero, scale, causal, rows=rows)
    av = v.abs().reshape(BH, N, d).numpy()
    flat = np.arange(BH * N) if rows is None else np.asarray(rows)
    bh_idx, i_idx = flat // N, flat % N
    if causal:  # keys 0..i are visible to row i
        vis_sum = np.cumsum(av, axis=1)[bh_idx, i_idx]
    else:
        vis_sum = av.sum(axis=1)[bh_idx]
    bound = (2.0 ** -4) * pv_abs + (2.0 ** -10) * vis_sum / l[:, None] \
        + 0.5 * bf16_ulp(o_ref) + 1e-3
    return o_ref, lse_ref, bound


def check_fp8(name, got, ref, bound, report):
    got = to_np(got).reshape(ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite"
    err = np.abs(got - ref)
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-30))
    worst = float(np.max(err / bound))
    line = (f"{name}: max_abs={err.max():.3e} rel_l2={rel:.3e} "
            f"worst err/bound={worst:.3f} mean bound={bound.mean():.3e}")
    report.append(line)
    assert worst <= 1.0, line
    return rel


SHAPES = [(1, 1, 16, 128), (1, 2, 144, 128), (2, 1, 400, 128), (1, 2, 1008, 128)]


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("B,H,N,d", SHAPES, ids=[f"b{b}h{h}n{n}d{d}" for b, h, n, d in SHAPES])
def test_fp8_forward_matches_oracle(fa, B, H, N, d, causal):
    q8, k8, v8, vt8, ds = make_fp8_inputs(B, H, N, d, seed=N + 3)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_fp8(fa, q8, k8, vt8, ds, causal, scale)
    q, k, v = dequantize(q8, ds[0]), dequantize(k8, ds[1]), dequantize(v8, ds[2])
    o_ref, lse_ref, bound = fp8_bound(q, k, v, scale, causal)
    report = []
    rel = check_fp8("O", o.reshape(-1, d), o_ref, bound, report)
    check_lse("lse", lse.reshape(-1), lse_ref, report)
    print(B, H, N, d, "causal" if causal else "full", "; ".join(report))
    assert rel <= 5e-2


def test_fp8_sharp_scores(fa):
    """q, k x2 (sharper softmax, more weight on few keys): the relative term
    dominates the bound."""
    B, H, N, d = 1, 2, 512, 128
    q8, k8, v8, vt8, ds = make_fp8_inputs(B, H, N, d, seed=9, qk_mult=2.0)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_fp8(fa, q8, k8, vt8, ds, True, scale)
    q, k, v = dequantize(q8, ds[0]), dequantize(k8, ds[1]), dequantize(v8, ds[2])
    o_ref, lse_ref, bound = fp8_bound(q, k, v, scale, True)
    report = []
    check_fp8("O", o.reshape(-1, d), o_ref, bound, report)
    check_lse("lse", lse.reshape(-1), lse_ref, report)
    print("sharp", "; ".join(report))


def test_fp8_errors(fa):
    dev = torch.device("cuda")
    q = torch.zeros((1, 1, 128, 64), dtype=torch.uint8, device=dev)
    with pytest.raises(fa.FaError) as e:
        fa.fa_forward_fp8(q, q, q.view(1, 1, 64, 128), 1.0, 1.0, 1.0)
    assert e.value.status == -3
    q = torch.zeros((1, 1, 100, 128), dtype=torch.uint8, device=dev)
    with pytest.raises(fa.FaError) as e:
        fa.fa_forward_fp8(q, q, q.view(1, 1, 128, 100), 1.0, 1.0, 1.0)
    assert e.value.status == -2
    q = torch.zeros((1, 1, 128, 128), dtype=torch.uint8, device=dev)
    with pytest.raises(fa.FaError) as e:
        fa.fa_forward_fp8(q, q, q, 1.0, -1.0, 1.0)
    assert e.value.status == -2


@pytest.mark.slow
def test_fp8_workload_causal_b2h16n8192d128(fa):
    """The benchmark shape in e4m3, on 32 sampled rows of every head."""
    B, H, N, d = 2, 16, 8192, 128
    q8, k8, v8, vt8, ds = make_fp8_inputs(B, H, N, d, seed=0)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_fp8(fa, q8, k8, vt8, ds, True, scale)
    q, k, v = dequantize(q8, ds[0]), dequantize(k8, ds[1]), dequantize(v8, ds[2])
    rows = []
    for h in range(B * H):
        rows += [h * N + i for i in sample_indices(N, 32, seed=1 + h, must=(0, 127, 128, N - 1))]
    rows = np.array(rows, dtype=np.int64)
    o_ref, lse_ref, bound = fp8_bound(q, k, v, scale, True, rows=rows)
    report = []
    check_fp8("O[sampled rows]", o.reshape(-1, d)[rows], o_ref, bound, report)
    check_lse("lse[sampled rows]", lse.reshape(-1)[rows], lse_ref, report)
    print("fp8 causal_b2h16n8192d128", "; ".join(report))
