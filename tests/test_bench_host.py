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


class StubRun:
    """The real binding over a stub library that records its calls, CPU
    tensors accepted as device tensors, CUDA events that report 0.5 ms per
    interval, and small stand-ins for the 8K and 32K workloads."""

    def __init__(self, monkeypatch):
        import types

        import torch
        from exact_io_aware_16_gb300 import _binding as bd
        from fa_inputs import Workload

        calls = self.calls = []

        class Stub:
            def __getattr__(self, name):
                def fn(*a):
                    calls.append(name)
                    if name == "fa_backward_workspace_size":
                        return 4 * a[0] * a[1] * a[2]
                    if name == "fa_decode_workspace_size":
                        return 4096
                    return 0
                return fn

        class Event:
            def __init__(self, enable_timing=False):
                pass

            def record(self, stream=None):
                pass

            def elapsed_time(self, other):
                return 0.5

        monkeypatch.setattr(bd, "library", lambda: Stub())
        monkeypatch.setattr(bd, "_on_device", lambda t: True)
        dec_name = bench.NEXT_ROW_DECODE[0]
        self.small = {
            bench.DEFAULT_WORKLOAD: Workload(bench.DEFAULT_WORKLOAD, 1, 2, 1024, 128, (True,)),
            dec_name: Workload(dec_name, 1, 2, 2048, 128, (True,), qk_mult=2.0)}
        monkeypatch.setattr(bench, "WORKLOADS", self.small)
        monkeypatch.setattr(bench.torch.cuda, "Event", Event)
        monkeypatch.setattr(bench.torch.cuda, "synchronize", lambda *a: None)
        monkeypatch.setattr(bench, "ClockSampler", lambda dev: types.SimpleNamespace(
            start=lambda: None, stop=lambda: None, mark_load=lambda: None,
            mark_done=lambda: None))
        fa = types.SimpleNamespace(**{n: getattr(bd, n) for n in dir(bd) if n.startswith("fa_")})
        fa.fa_get_device_error = lambda stream=None: (0, 0)
        self.fa = fa
        self.dev = torch.device("cpu")


def test_next_rows_record_drives_every_widened_row(monkeypatch):
    """The default line's record of the widened rows: every row's entry
    point is launched for its warm-up and timed steps, and the rates follow
    from the FLOP and byte counts."""
    run = StubRun(monkeypatch)
    calls, small, fa = run.calls, run.small, run.fa
    dec_name = bench.NEXT_ROW_DECODE[0]

    peaks = {"bf16_tflops": 2000.0, "hbm_gbs": 7000.0}
    steps = 2
    rec = bench.next_rows_record(fa, None, run.dev, 0, peaks, steps=steps)

    n = 3 + steps
    for name in ("fa_forward_dropout", "fa_backward_dropout", "fa_forward_blocksparse",
                 "fa_backward_blocksparse", "fa_forward_fp8", "fa_decode"):
        assert calls.count(name) == n, (name, calls.count(name))
    w, wd = small[bench.DEFAULT_WORKLOAD], small[dec_name]
    E = 0.5 * w.B * w.H * w.N * w.N
    drop = rec["dropout"]
    assert drop["ms_per_step"] == pytest.approx(1.0)
    assert drop["fwd_tflops"] == pytest.approx(4 * w.d * E / 0.5e-3 / 1e12)
    assert drop["bwd_tflops"] == pytest.approx(10 * w.d * E / 0.5e-3 / 1e12)
    bs = rec["blocksparse"]
    kept = bench.kept_elements(bench.band_mask(bench.NEXT_ROW_BAND, w.N), w.N, False)
    assert bs["kept_fraction"] == pytest.approx(kept / (w.N * w.N))
    assert bs["step_tflops"] == pytest.approx(14 * w.d * kept * w.B * w.H / 1e-3 / 1e12)
    assert rec["fp8_forward"]["ms_per_launch"] == pytest.approx(0.5 / steps)
    assert rec["fp8_forward"]["frac_of_fp8_peak"] == pytest.approx(
        rec["fp8_forward"]["tflops"] / 4000.0)
    dec = rec["decode"]
    # K and V read once, q read and o written (bf16), lse written (fp32)
    nbytes = 2 * (2 * wd.B * wd.H * wd.N * wd.d) + 2 * (2 * wd.B * wd.H * 16 * wd.d) + \
        4 * wd.B * wd.H * 16
    assert dec["us_per_step"] == pytest.approx(1e3 * 0.5 / steps)
    assert dec["hbm_gbs"] == pytest.approx(nbytes / (0.5 / steps * 1e-3) / 1e9)


@pytest.mark.parametrize("flag", ["dropout", "block_mask", "both", "fp8", "decode"])
def test_flag_runners_print_one_line(monkeypatch, capsys, flag):
    """bench.py --dropout / --block-mask / --fp8 / --decode on the stub run:
    each launches its entry points for every warm-up and timed step and
    prints one JSON line whose rate follows from the 0.5 ms intervals."""
    run = StubRun(monkeypatch)
    w = run.small[bench.DEFAULT_WORKLOAD]
    args = argparse.Namespace(steps=3, warmup=2, dropout=None, block_mask=None, decode=None)
    tensors = make_small_inputs(w)
    if flag in ("dropout", "both"):
        args.dropout = 0.1
    if flag in ("block_mask", "both"):
        args.block_mask = "band:2:1"
    if flag == "fp8":
        assert bench.run_fp8(args, 1, 0, 0, run.fa, w, True, 0, run.dev) == 0
        want = {"fa_forward_fp8": 5}
    elif flag == "decode":
        args.decode = 4
        assert bench.run_decode(args, 1, 0, 0, run.fa, w, tensors[:3], 0, run.dev) == 0
        want = {"fa_decode": 5}
    else:
        assert bench.run_variant(args, 1, 0, 0, run.fa, w, True, tensors, 0, run.dev) == 0
        kind = "dropout" if args.dropout else "blocksparse"
        want = {f"fa_forward_{kind}": 5, f"fa_backward_{kind}": 5}
    for name, count in want.items():
        assert run.calls.count(name) == count, (name, run.calls)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["value"] > 0 and line["n_gpus"] == 1 and line["steps"] == 3
    if flag != "decode":  # a few MB of inputs: L2 is flushed, and the line says so
        assert line["config"]["l2"].startswith("L2 flushed before every step")
    if flag == "decode":
        assert line["ms_per_step"] == pytest.approx(0.5 / 3)
    elif flag == "fp8":
        assert line["ms_per_step"] == pytest.approx(0.5)
    else:
        assert line["ms_per_step"] == pytest.approx(1.0)


def make_small_inputs(w):
    from fa_inputs import make_inputs

    return make_inputs(w.B, w.H, w.N, w.d, w.seed, w.qk_mult)


def test_l2_label_follows_the_step_size():
    """The default workload's tensors exceed L2; a workload that fits in L2 is
    timed with a flush and labelled so (the bench flushes exactly when the
    label says it does)."""
    big, small = WORKLOADS["causal_b2h16n8192d128"], WORKLOADS["b4h16n2048d64"]
    assert bench.step_bytes(big) > bench.L2_BYTES
    assert bench.workload_config(big, True)["l2"].startswith("inputs larger than L2")
    assert bench.step_bytes(small) <= bench.L2_BYTES
    assert bench.workload_config(small, True)["l2"].startswith("L2 flushed")
    assert bench.l2_flush_buffer(bench.step_bytes(big), "cpu") is None
    assert bench.l2_flush_buffer(1000, "cpu").numel() == bench.FLUSH_BYTES > bench.L2_BYTES


def test_nccl_ranks_bind_their_gpu_before_the_group_forms(monkeypatch):
    """Under torchrun each rank of the CUDA arm takes its own GPU before the
    NCCL process group forms (no collective has to guess the device); the
    reference arm joins a gloo group and binds no GPU."""
    import torch.distributed as dist

    calls = []
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    monkeypatch.setattr(bench.torch.cuda, "set_device", lambda d: calls.append(("set_device", d)))
    monkeypatch.setattr(dist, "init_process_group",
                        lambda backend, **kw: calls.append(("init", backend)))
    assert bench.dist_setup(argparse.Namespace(impl="ours")) == (2, 1, 1)
    assert calls == [("set_device", 1), ("init", "nccl")]
    calls.clear()
    assert bench.dist_setup(argparse.Namespace(impl="reference")) == (2, 1, 1)
    assert calls == [("init", "gloo")]
