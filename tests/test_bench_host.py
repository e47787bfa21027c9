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
