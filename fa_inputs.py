"""Seeded synthetic inputs for attention workloads.

This module holds no arithmetic of the attention method.  It only draws
random numbers and rounds them to bf16, and it is the one piece shared by the
CUDA path's tests/bench and the CPU oracle.

Recipe: one CPU ``torch.Generator`` seeded with ``seed`` draws, in this order,
full tensors q, k, v and dO of shape [B, H, N, d], each fp32 N(0, 1); q and k
are multiplied by ``qk_mult`` (x2 is exact in bf16) and every tensor is cast
to bf16 with round-to-nearest-even.  ``scale`` defaults to 1/sqrt(d).

e4m3 inputs (``make_fp8_inputs``): the same fp32 draws of q, k, v, each
divided by its per-tensor descale amax / 448 (448 = largest finite e4m3)
and rounded to e4m3 (round to nearest even); V is also given transposed per
head, [B, H, d, N].
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: tuple  # the masking modes this workload is run in
    backward: bool = True
    qk_mult: float = 1.0
    seed: int = 0
    note: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def BH(self) -> int:
        return self.B * self.H


# The five workloads of the exact-attention benchmark suite: short forward-only
# check, mid-size fwd+bwd in both masking modes, two long-context causal runs
# (8K at d=128; 32K at d=128 with a sharpened softmax) and the short-sequence
# regime where tiling overhead matters.
WORKLOADS = {
    "fwd_b1h2n256d64": Workload("fwd_b1h2n256d64", 1, 2, 256, 64, (False,), backward=False),
    "b4h16n2048d64": Workload("b4h16n2048d64", 4, 16, 2048, 64, (True, False)),
    "causal_b2h16n8192d128": Workload("causal_b2h16n8192d128", 2, 16, 8192, 128, (True,)),
    "causal_b1h32n32768d128_qk2": Workload("causal_b1h32n32768d128_qk2", 1, 32, 32768, 128,
                                           (True,), qk_mult=2.0),
    "short_b64h12n512d64": Workload("short_b64h12n512d64", 64, 12, 512, 64, (False,)),
}

# The 8K workload's shape at half and twice the sequence length (same B, H,
# d): the DRAM traffic of every kernel must grow linearly with N.
SCALING_WORKLOADS = {
    "causal_b2h16n4096d128": Workload("causal_b2h16n4096d128", 2, 16, 4096, 128, (True,)),
    "causal_b2h16n16384d128": Workload("causal_b2h16n16384d128", 2, 16, 16384, 128, (True,)),
}


def make_inputs(B: int, H: int, N: int, d: int, seed: int = 0, qk_mult: float = 1.0,
                with_dO: bool = True):
    """bf16 CPU tensors (q, k, v, dO) of shape [B, H, N, d] (dO None if not asked)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    shape = (B, H, N, d)
    q = torch.randn(shape, generator=g, dtype=torch.float32)
    k = torch.randn(shape, generator=g, dtype=torch.float32)
    v = torch.randn(shape, generator=g, dtype=torch.float32)
    dO = torch.randn(shape, generator=g, dtype=torch.float32) if with_dO else None
    if qk_mult != 1.0:
        q.mul_(qk_mult)
        k.mul_(qk_mult)
    q = q.to(torch.bfloat16)
    k = k.to(torch.bfloat16)
    v = v.to(torch.bfloat16)
    dO = dO.to(torch.bfloat16) if dO is not None else None
    return q, k, v, dO


E4M3_MAX = 448.0


def make_fp8_inputs(B: int, H: int, N: int, d: int, seed: int = 0, qk_mult: float = 1.0):
    """e4m3 CPU tensors and their per-tensor descales.

    Returns (q8, k8, v8, vt8, descales): q8, k8, v8 torch.float8_e4m3fn of
    shape [B, H, N, d], vt8 = v8 transposed to [B, H, d, N] (contiguous),
    descales = (q_descale, k_descale, v_descale) as Python floats that are
    exact fp32 values; the real inputs are q8 * q_descale etc.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    shape = (B, H, N, d)
    xs = [torch.randn(shape, generator=g, dtype=torch.float32) for _ in range(3)]
    if qk_mult != 1.0:
        xs[0].mul_(qk_mult)
        xs[1].mul_(qk_mult)
    out, desc = [], []
    for x in xs:
        ds = float(torch.tensor(float(x.abs().max()) / E4M3_MAX, dtype=torch.float32))
        out.append((x / ds).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn))
        desc.append(ds)
    q8, k8, v8 = out
    vt8 = v8.transpose(-1, -2).contiguous()
    return q8, k8, v8, vt8, tuple(desc)


def dequantize(x8, descale: float):
    """The real values of an e4m3 tensor, exactly, as float64."""
    return x8.to(torch.float64) * float(descale)


def sample_indices(n_total: int, n_sample: int, seed: int = 1, must=()):
    """Seeded sample of distinct indices in [0, n_total), always holding `must`."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    must = sorted({int(m) for m in must if 0 <= int(m) < n_total})
    if n_sample >= n_total:
        return list(range(n_total))
    perm = torch.randperm(n_total, generator=g).tolist()
    out = list(must)
    seen = set(out)
    for p in perm:
        if len(out) >= n_sample:
            break
        if p not in seen:
            out.append(p)
            seen.add(p)
    return sorted(out)
