"""Comparison helpers: CUDA-path results against the fp64 oracle.

Tolerances (bf16 outputs and gradients): max-abs error <= 2e-2 AND relative
L2 error ||x - ref|| / ||ref|| <= 1e-2 per tensor; lse: max-abs <= 1e-4.
With dropout every kept term is multiplied by 1/q (q the keep probability)
before it is rounded, so absolute errors grow by that factor: the max-abs
bound is 2e-2 / q there (abs_scale); rel-L2 stays 1e-2.
Where bf16 storage alone cannot meet 2e-2 (|ref| >= 8, where half an ulp of
bf16 is >= 1/32), the max-abs bound of that element is widened by half a bf16
ulp of the reference, and the report says so; rel-L2 is never widened.
"""
from __future__ import annotations

import numpy as np
import torch

MAX_ABS = 2e-2
REL_L2 = 1e-2
LSE_ABS = 1e-4


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significand bits)."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.maximum(ax, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def to_np(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def check_bf16(name: str, got, ref, report: list | None = None, abs_scale: float = 1.0):
    """abs_scale multiplies the max-abs bound (dropout: the inverse keep
    probability, which every kept term carries before it is rounded)."""
    got = to_np(got).reshape(ref.shape)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = np.abs(got - ref)
    floor = float(np.max(np.abs(to_np(torch.from_numpy(ref).to(torch.bfloat16)) - ref))) \
        if ref.size else 0.0
    bound = np.full(ref.shape, MAX_ABS * abs_scale)
    widened = floor > 1e-2
    if widened:
        bound = bound + 0.5 * bf16_ulp(ref)
    nref = float(np.linalg.norm(ref))
    rel = float(np.linalg.norm(got - ref)) / max(nref, 1e-30)
    max_abs = float(err.max()) if err.size else 0.0
    line = (f"{name}: max_abs={max_abs:.3e} rel_l2={rel:.3e} repr_floor={floor:.3e}"
            + (" (max-abs widened by half a bf16 ulp)" if widened else "")
            + (f" (max-abs bound x{abs_scale:.4g})" if abs_scale != 1.0 else ""))
    if report is not None:
        report.append(line)
    ok_abs = bool(np.all(err <= bound))
    if not ok_abs:
        i = int(np.argmax(err - bound))
        raise AssertionError(f"{line}; worst at flat {i}: got {got.reshape(-1)[i]} "
                             f"ref {ref.reshape(-1)[i]}")
    if nref > 0:
        assert rel <= REL_L2, line
    return max_abs, rel


def check_lse(name: str, got, ref, report: list | None = None):
    got = to_np(got).reshape(ref.shape)
    ref = np.asarray(ref, dtype=np.float64)
    # rows with no visible key (block-sparse) have lse = -inf on both sides
    inf_ref = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), inf_ref), f"{name}: -inf rows differ"
    got = np.where(inf_ref, 0.0, got)
    ref = np.where(inf_ref, 0.0, ref)
    err = np.abs(got - ref)
    max_abs = float(err.max()) if err.size else 0.0
    line = f"{name}: max_abs={max_abs:.3e}"
    if report is not None:
        report.append(line)
    assert np.all(np.isfinite(got)), f"{name}: non-finite"
    assert max_abs <= LSE_ABS, line
    return max_abs
