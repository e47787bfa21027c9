"""Host-side logic of bench.py (no GPU): the CPU baseline and the reference
arm time the oracle on bounded samples.  The oracle's timing is replaced by a
fake that reports a fixed cost per sample, so the bounds can be checked
exactly: the baseline takes samples until at least ORACLE_BASELINE_SECONDS of
work and never starts one past ORACLE_BASELINE_MAX_SECONDS; the reference
arm sizes its per-step row sample from a probe so that warm-up and timed steps
together cost about REFERENCE_RUN_SECONDS whatever --steps / --warmup are."""
import argparse
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from fa_inputs import WORKLOADS  # noqa: E402


def fake_sampler(per_pair_s, per_row_s, calls):
    """oracle_sample stand-in: a full pair costs per_pair_s, a row sample
    per_row_s per row; flops 1 per second of work (rate 1e-12 TFLOP/s)."""

    def sample(w, causal, q, k, v, dO, bh_index=0, n_rows=None):
        dt = per_pair_s if (n_rows is None and w.N <= bench.ORACLE_FULL_HEAD_MAX_N) else \
            per_row_s * min(w.N, 256 if n_rows is None else n_rows)
        calls.append((bh_index, n_rows, dt))
        return dt, dt, 16, "fake", None

    return sample


@pytest.mark.parametrize("per_pair", [0.5, 3.0, 9.0, 25.0])
def test_baseline_takes_at_least_the_minimum_and_stops_before_the_maximum(monkeypatch, per_pair):
    calls = []
    monkeypatch.setattr(bench, "oracle_sample", fake_sampler(per_pair, 0.0, calls))
    w = WORKLOADS["causal_b2h16n8192d128"]
    dt, fl, cores, desc, extrap = bench.oracle_baseline(w, True, None, None, None, None)
    n = len(calls)
    assert n >= 1 and dt == pytest.approx(n * per_pair)
    assert [c[0] for c in calls] == list(range(n))  # distinct (batch, head) pairs
    if n < w.B * w.H:
        # it stopped because the minimum was reached, or the next sample would pass the max
        assert dt >= bench.ORACLE_BASELINE_SECONDS or \
            dt + per_pair > bench.ORACLE_BASELINE_MAX_SECONDS
    # no sample started once the minimum was reached
    assert (n - 1) * per_pair < bench.ORACLE_BASELINE_SECONDS
    assert f"{n} sample(s)" in desc


def test_baseline_is_limited_by_the_pairs_of_a_small_workload(monkeypatch):
    calls = []
    monkeypatch.setattr(bench, "oracle_sample", fake_sampler(0.01, 0.0, calls))
    w = WORKLOADS["fwd_b1h2n256d64"]  # two (batch, head) pairs
    bench.oracle_baseline(w, False, None, None, None, None)
    assert len(calls) == w.B * w.H


@pytest.mark.parametrize("steps,warmup", [(3, 3), (50, 10), (200, 10), (1000, 3)])
def test_reference_arm_fits_its_time_budget(monkeypatch, capsys, steps, warmup):
    calls = []
    per_row = 4e-4  # seconds of oracle work per query row
    monkeypatch.setattr(bench, "oracle_sample", fake_sampler(0.0, per_row, calls))
    monkeypatch.setattr(bench, "make_inputs", lambda *a, **k: (None, None, None, None))
    args = argparse.Namespace(workload="causal_b2h16n8192d128", steps=steps, warmup=warmup,
                              gpus=1)
    assert bench.run_reference(args, 1, 0) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == steps
    probe, rest = calls[0], calls[1:]
    assert probe[1] == 64 and len(rest) == steps + warmup
    n_rows = {c[1] for c in rest}
    assert len(n_rows) == 1  # every step samples the same number of rows
    total = sum(c[2] for c in rest)
    # about REFERENCE_RUN_SECONDS of work in all (rows never below 16 nor above N)
    w = WORKLOADS["causal_b2h16n8192d128"]
    rows = n_rows.pop()
    assert 16 <= rows <= w.N
    if 16 < rows < w.N:
        assert total == pytest.approx(bench.REFERENCE_RUN_SECONDS, rel=0.02)
    else:
        assert total <= bench.REFERENCE_RUN_SECONDS * 1.5 or rows == 16


@pytest.mark.parametrize("name", ["causal_b2h16n8192d128", "b4h16n2048d64",
                                  "short_b64h12n512d64"])
@pytest.mark.parametrize("causal", [True, False])
def test_kernel_work_counts_the_method_once(name, causal):
    """The backward kernels' method work sums to the step's 10 N^2 d (S
    recomputed once), the forward's is 4 N^2 d, and the executed work of the
    dQ kernel is its four products (S, dP, B = P K, dQ)."""
    w = WORKLOADS[name]
    kw = bench.kernel_work(w, causal)
    f_fwd, f_bwd = bench.flops(w, causal)
    assert kw["fwd"]["flops"] == f_fwd
    assert kw["bwd_dq"]["flops"] + kw["bwd_dkdv"]["flops"] == f_bwd
    base = w.B * w.H * w.N * w.N * w.d * (0.5 if causal else 1.0)
    assert kw["bwd_dq"]["exec_flops"] == 8 * base and kw["bwd_dkdv"]["exec_flops"] == 8 * base
    t = w.B * w.H * w.N * w.d * 2
    r = w.B * w.H * w.N * 4
    fwd_b, bwd_b = bench.alg_bytes(w)
    assert kw["fwd"]["bytes"] == fwd_b
    # every backward input once (q, k, v, dO, o, lse, D read; dq, dk, dv, D written)
    # is read or written by exactly the kernels that need it
    assert kw["bwd_pre"]["bytes"] == 2 * t + r
    assert kw["bwd_dq"]["bytes"] == 5 * t + 3 * r
    assert kw["bwd_dkdv"]["bytes"] == 6 * t + 2 * r


def test_kernel_table_rates():
    w = WORKLOADS["causal_b2h16n8192d128"]
    per = {"fwd": 4.5, "bwd_pre": 0.25, "bwd_dq": 7.5, "bwd_dkdv": 7.5}  # ms over 10 steps
    tab = bench.kernel_table(w, True, per, 10, 2000.0, 7000.0, 5e12)  # any MUFU peak
    kw = bench.kernel_work(w, True)
    assert tab["bwd_dkdv"]["alg_tflops"] == pytest.approx(kw["bwd_dkdv"]["flops"] / 0.75e-3 / 1e12)
    assert tab["bwd_dq"]["frac_of_peak"] == pytest.approx(tab["bwd_dq"]["alg_tflops"] / 2000.0)
    assert tab["bwd_dq"]["exec_tflops"] == pytest.approx(4 * tab["bwd_dq"]["alg_tflops"])
    assert tab["fwd"]["us_per_launch"] == pytest.approx(450.0)
    assert "alg_tflops" not in tab["bwd_pre"]
    assert sum(k["share"] for k in tab.values()) == pytest.approx(1.0)
    assert tab["fwd"]["exp2_frac_of_mufu"] == pytest.approx(
        w.B * w.H * w.N * w.N * 0.5 / 0.45e-3 / 5e12)


def test_clock_summary_counts_samples_in_the_timed_region():
    """NVML samples (time, MHz, W, reason bits): only those between
    mark_load and mark_done count as under load, and reasons are decoded."""

    class FakeNvml:
        max_mhz = 2070.0

    cs = bench.ClockSampler(0)
    cs.nvml = FakeNvml()
    cs.samples = [(0.0, 1000.0, 100.0, 0x1), (1.0, 2070.0, 900.0, 0x4), (1.5, 2040.0, 950.0, 0x0),
                  (2.0, 2070.0, 1000.0, 0x0), (3.0, 1200.0, 200.0, 0x1)]
    cs.t_load, cs.t_done = 0.9, 2.1
    s = cs._summary_nvml()
    assert s["samples"] == 5 and s["samples_under_load"] == 3
    assert s["sm_mhz"] == 2070.0 and s["sm_mhz_min"] == 2040.0
    assert s["reasons"] == ["sw_power_cap"]
    assert s["power_w_max"] == 1000.0
