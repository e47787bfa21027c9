#!/usr/bin/env python
"""Benchmark of exact attention fwd+bwd on GB300 through the C ABI of libfa.

One step = one forward pass (fa_forward) and one backward pass (D pre-pass,
dQ kernel, dK/dV kernel) over one batch of seeded synthetic bf16 inputs
already resident in device memory.  The default workload is causal attention
with B=2, H=16, N=8192, d=128, scale 1/sqrt(d) (the long-context case where
the FLOP target applies).

FLOP convention (algorithmic): forward 4*B*H*N^2*d, backward 10*B*H*N^2*d
(five matmuls, the S recompute counted once), halved under the causal mask.

Prints ONE JSON line on rank 0.  ``--impl reference`` times the fp64 CPU
oracle instead (the only other arm this method has), on the host cores.
Under torchrun every rank runs the same per-GPU workload (weak scaling, no
collective on the data path; heads are independent).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from fa_inputs import SCALING_WORKLOADS, WORKLOADS, make_inputs, sample_indices  # noqa: E402

METRIC = "attention fwd/bwd TFLOP/s at 1 GB300 and % of dense BF16 tensor peak"
DEFAULT_WORKLOAD = "causal_b2h16n8192d128"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def captured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` from the committed ncu capture, or None
    when there is none for this workload or the kernel source changed since."""
    import hashlib

    try:
        with open(os.path.join(ROOT, "profiles", "dram_traffic.json")) as f:
            rec = json.load(f).get(kernel)
        if not rec or rec["workload"] != workload:
            return None
        m = hashlib.sha256()
        for src in rec["sources"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                m.update(f.read())
        if m.hexdigest() != rec["source_sha256"]:
            return None
        return rec["read_bytes"] + rec["write_bytes"]
    except Exception:
        return None


def flops(w, causal):
    base = w.B * w.H * w.N * w.N * w.d * (0.5 if causal else 1.0)
    return 4.0 * base, 10.0 * base


def alg_bytes(w):
    """Algorithmic HBM bytes per step: fwd reads q,k,v and writes o,lse; bwd
    reads q,k,v,o,dO,lse,D and writes dq,dk,dv (no N^2 terms)."""
    t = w.B * w.H * w.N * w.d * 2
    r = w.B * w.H * w.N * 4
    return 4 * t + r, 8 * t + 2 * r + r  # fwd; bwd incl. D write + read


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].lower() in ("active", "1")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    """The largest x over all ranks (timings: the job ends with its slowest rank)."""
    if world == 1:
        return x
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(per_rank_work: float, world: int, seconds_max: float) -> float:
    """Whole-job throughput: every rank processes the same per-rank work
    (weak scaling), the job takes as long as its slowest rank."""
    return world * per_rank_work / seconds_max


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


ORACLE_FULL_HEAD_MAX_N = 8192  # above this one head's full fp64 step takes too long


def oracle_sample(w, causal, q, k, v, dO, bh_index=0, n_rows=None):
    """Time the fp64 oracle (as it stands) on a bounded sample of the
    workload.  n_rows None and N <= 8192: the full forward and backward of
    one (batch, head) pair.  Otherwise n_rows (default 256) seeded query rows
    of one pair, forward and the row pass of the backward (dq, m, l, D),
    whose cost per row is what a full run repeats N times per head.  Returns
    (seconds, flops of what was computed, cores, description, extrapolated
    seconds of the full problem at the sampled rate or None)."""
    import oracle

    b, h = divmod(bh_index % (w.B * w.H), w.H)
    qs, ks, vs, ds = (t[b:b + 1, h:h + 1] for t in (q, k, v, dO))
    cores = oracle.default_threads()
    if n_rows is None and w.N <= ORACLE_FULL_HEAD_MAX_N:
        t0 = time.perf_counter()
        oracle.forward(qs, ks, vs, w.scale, causal, nthreads=cores)
        oracle.backward(qs, ks, vs, ds, w.scale, causal, nthreads=cores)
        dt = time.perf_counter() - t0
        base = w.N * w.N * w.d * (0.5 if causal else 1.0)
        desc = (f"full fp64 forward+backward of one (batch, head) pair of {w.B * w.H} "
                f"(flops counted as 14 N^2 d{' x 1/2 causal' if causal else ''} for what the "
                f"oracle computes)")
        return dt, 14.0 * base, cores, desc, None
    n_rows = min(w.N, 256 if n_rows is None else max(1, int(n_rows)))
    rows = sample_indices(w.N, n_rows, seed=1 + bh_index, must=(0, w.N - 1))
    visible = sum((i + 1) if causal else w.N for i in rows)
    t0 = time.perf_counter()
    oracle.forward(qs, ks, vs, w.scale, causal, rows=rows, nthreads=cores)
    oracle.backward_rows(qs, ks, vs, ds, w.scale, causal, rows=rows, nthreads=cores)
    dt = time.perf_counter() - t0
    fl = 12.0 * visible * w.d  # forward 4 n d + row pass 8 n d per row of n visible keys
    full_visible = w.B * w.H * (w.N * (w.N + 1) / 2 if causal else w.N * w.N)
    extrap = dt * full_visible / visible * (14.0 / 12.0)
    desc = (f"{len(rows)} seeded query rows of one (batch, head) pair of {w.B * w.H}, fp64 "
            f"forward + backward row pass ({visible / len(rows):.0f} visible keys per row on "
            f"average; {w.B * w.H * w.N} rows in the problem)")
    return dt, fl, cores, desc, extrap


ORACLE_BASELINE_SECONDS = 10.0  # the CPU baseline samples at least this much oracle work
ORACLE_BASELINE_MAX_SECONDS = 30.0
REFERENCE_RUN_SECONDS = 120.0  # the reference arm's warm-up + timed steps together


def oracle_baseline(w, causal, q, k, v, dO):
    """The oracle on successive (batch, head) pairs (or row samples of them)
    until at least ORACLE_BASELINE_SECONDS of work, never starting a sample
    that would pass ORACLE_BASELINE_MAX_SECONDS.  Returns (seconds, flops,
    cores, description, extrapolated full-problem seconds or None)."""
    tot_t = tot_f = 0.0
    n = 0
    cores, desc, extrap, last = 1, "", None, 0.0
    while n < w.B * w.H and tot_t < ORACLE_BASELINE_SECONDS:
        if n > 0 and tot_t + last > ORACLE_BASELINE_MAX_SECONDS:
            break
        dt, fl, cores, desc, ex = oracle_sample(w, causal, q, k, v, dO, n)
        tot_t += dt
        tot_f += fl
        last = dt
        n += 1
        if ex is not None:
            extrap = ex if extrap is None else extrap
    desc = f"{n} sample(s), {tot_t:.1f} s in all; each: {desc}"
    if extrap is not None:
        extrap = tot_t / tot_f * (14.0 * w.B * w.H * w.N * w.N * w.d * (0.5 if causal else 1.0))
    return tot_t, tot_f, cores, desc, extrap


def run_reference(args, world, rank):
    w = {**WORKLOADS, **SCALING_WORKLOADS}[args.workload]
    causal = w.causal[0]
    if rank != 0:
        return 0
    q, k, v, dO = make_inputs(w.B, w.H, w.N, w.d, w.seed, w.qk_mult)
    # every step is a row sample of one (batch, head) pair, sized from a first
    # 64-row probe so that warm-up and timed steps together take about
    # REFERENCE_RUN_SECONDS
    dt0, _, _, _, _ = oracle_sample(w, causal, q, k, v, dO, 0, n_rows=64)
    per_row = dt0 / min(64, w.N)
    per_step = REFERENCE_RUN_SECONDS / max(args.steps + args.warmup, 1)
    n_rows = int(max(16, min(w.N, per_step / max(per_row, 1e-9))))
    for s in range(args.warmup):
        oracle_sample(w, causal, q, k, v, dO, s, n_rows=n_rows)
    tot_t, tot_f, cores, desc = 0.0, 0.0, 1, ""
    for s in range(args.steps):
        dt, fl, cores, desc, _ = oracle_sample(w, causal, q, k, v, dO, args.warmup + s,
                                               n_rows=n_rows)
        tot_t += dt
        tot_f += fl
    value = tot_f / tot_t / 1e12
    sample = f"each step: {desc}"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_t / max(args.steps, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, causal),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def band_mask(spec: str, N: int):
    """Block mask [nt, nt] from 'band:W[:G]': keep tiles with |i - j| <= W and
    the first G tile rows and columns (local band + global tokens)."""
    parts = spec.split(":")
    if parts[0] != "band" or len(parts) not in (2, 3):
        raise ValueError("block mask spec must be band:W[:G]")
    W = int(parts[1])
    G = int(parts[2]) if len(parts) == 3 else 0
    nt = -(-N // 128)
    i = torch.arange(nt)[:, None]
    j = torch.arange(nt)[None, :]
    return (((i - j).abs() <= W) | (i < G) | (j < G)).to(torch.uint8)


def kept_elements(mask, N: int, causal: bool) -> float:
    """Score elements (query, key) that a block mask and the causal mask keep."""
    nt = mask.shape[0]
    rows = [min(128, N - 128 * t) for t in range(nt)]
    total = 0.0
    for i in range(nt):
        for j in range(nt):
            if not mask[i, j] or (causal and j > i):
                continue
            if causal and j == i:
                total += rows[i] * (rows[i] + 1) / 2
            else:
                total += rows[i] * rows[j]
    return total


def workload_config(w, causal):
    return {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": causal,
            "scale": w.scale, "qk_mult": w.qk_mult, "seed": w.seed,
            "l2": "inputs larger than L2 (q,k,v,o,dO together "
                  f"{5 * w.B * w.H * w.N * w.d * 2 / 1e6:.0f} MB per step > 129 MB)"}


def run_ours(args, world, rank, local):
    import exact_io_aware_16_gb300 as fa
    from exact_io_aware_16_gb300 import build as fabuild

    if rank == 0 or not os.path.exists(fabuild.LIB):
        fabuild.build()
    barrier(world)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = {**WORKLOADS, **SCALING_WORKLOADS}[args.workload]
    causal = w.causal[0] if args.causal is None else bool(args.causal)
    scale = w.scale
    q_h, k_h, v_h, dO_h = make_inputs(w.B, w.H, w.N, w.d, w.seed, w.qk_mult)
    q, k, v, dO = (t.to(dev) for t in (q_h, k_h, v_h, dO_h))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    D = torch.empty_like(lse)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    stream = torch.cuda.current_stream(dev)
    if args.fp8:
        del q, k, v, dO, o, lse, D, dq, dk, dv
        return run_fp8(args, world, rank, local, fa, w, causal, stream, dev)
    if args.block_mask or args.dropout:
        return run_variant(args, world, rank, local, fa, w, causal, (q, k, v, dO), stream, dev)
    if args.decode:
        return run_decode(args, world, rank, local, fa, w, (q, k, v), stream, dev)
    names = ["fwd", "bwd_pre", "bwd_dq", "bwd_dkdv"]

    def step(ev=None):
        fa.fa_forward(q, k, v, causal=causal, scale=scale, o=o, lse=lse, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        fa.fa_backward_preprocess(o, dO, D, stream=stream)
        if ev is not None:
            ev[2].record(stream)
        fa.fa_backward_dq(q, k, v, dO, lse, D, causal=causal, scale=scale, dq=dq, stream=stream)
        if ev is not None:
            ev[3].record(stream)
        fa.fa_backward_dkdv(q, k, v, dO, lse, D, causal=causal, scale=scale, dk=dk, dv=dv,
                            stream=stream)
        if ev is not None:
            ev[4].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    st, detail = fa.fa_get_device_error(stream)
    if st != 0:
        raise RuntimeError(f"device error during warm-up: {st} {detail:#x}")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    h0 = time.perf_counter()
    n_enq = min(args.steps, 8)  # before the launch queue can fill and block the host
    enqueue_us = 0.0
    for s in range(args.steps):
        evs[s][0].record(stream)
        step(evs[s])
        if s + 1 == n_enq:
            enqueue_us = (time.perf_counter() - h0) * 1e6 / n_enq  # host side, per step
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    st, detail = fa.fa_get_device_error(stream)
    if st != 0:
        raise RuntimeError(f"device error in timed region: {st} {detail:#x}")
    total_ms = t_start.elapsed_time(t_end)
    per_kernel = {n: 0.0 for n in names}
    for s in range(args.steps):
        for i, n in enumerate(names):
            per_kernel[n] += evs[s][i].elapsed_time(evs[s][i + 1])
    total_ms_max = max_over_ranks(total_ms, world)
    ms_per_step = total_ms_max / args.steps
    f_fwd, f_bwd = flops(w, causal)
    value = aggregate_rate(f_fwd + f_bwd, world, ms_per_step * 1e-3) / 1e12

    peaks, peak_src = read_peaks()
    long_region = total_ms > 1000.0
    peak = peaks["bf16_tflops_sustained"] if long_region else peaks["bf16_tflops"]
    peak_kind = "sustained" if long_region else "burst"
    fwd_ms = per_kernel["fwd"] / args.steps
    bwd_ms = (per_kernel["bwd_pre"] + per_kernel["bwd_dkdv"] + per_kernel["bwd_dq"]) / args.steps
    fwd_tf = f_fwd / (fwd_ms * 1e-3) / 1e12
    bwd_tf = f_bwd / (bwd_ms * 1e-3) / 1e12
    # diagnostics: HBM share of the algorithmic bytes (the measure that matters
    # for the short, low-intensity workloads), exp2 rate, host enqueue time
    fwd_bytes, bwd_bytes = alg_bytes(w)
    diag = {
        "fwd_hbm_gbs": fwd_bytes / (fwd_ms * 1e-3) / 1e9,
        "fwd_hbm_frac": fwd_bytes / (fwd_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
        "bwd_hbm_gbs": bwd_bytes / (bwd_ms * 1e-3) / 1e9,
        "bwd_hbm_frac": bwd_bytes / (bwd_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
        "fwd_exp2_per_s": w.B * w.H * w.N * w.N * (0.5 if causal else 1.0) / (fwd_ms * 1e-3),
        "host_enqueue_us_per_step": enqueue_us,
        "device_us_per_step": ms_per_step * 1e3,
    }

    # dominant kernel and its roofline (algorithmic work of that kernel alone)
    base = w.B * w.H * w.N * w.N * w.d * (0.5 if causal else 1.0)
    # per-kernel algorithmic FLOPs: the matmuls that kernel's own outputs require
    # (dQ needs S, dP and dS K; dK/dV need S, dP, P^T dO and dS^T Q), so the
    # recomputed S and dP count in both backward kernels
    kflops = {"fwd": 4 * base, "bwd_dkdv": 8 * base, "bwd_dq": 6 * base, "bwd_pre": 0.0}
    tbytes = w.B * w.H * w.N * w.d * 2
    kbytes = {"bwd_pre": 2 * tbytes + w.B * w.H * w.N * 4}
    dom = max(names, key=lambda n: per_kernel[n])
    dom_ms = per_kernel[dom] / args.steps
    if dom == "bwd_pre":
        ach = kbytes[dom] / (dom_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "kernel": dom, "achieved": ach, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": ach / peaks["hbm_gbs"],
                "traffic": captured_traffic(dom, w.name) if causal == w.causal[0] else None}
    else:
        ach = kflops[dom] / (dom_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "kernel": dom, "achieved": ach, "peak": peak,
                "unit": "TFLOP/s", "frac": ach / peak,
                "traffic": captured_traffic(dom, w.name) if causal == w.causal[0] else None,
                "peak_kind": f"{peak_kind} bf16 ({peak_src})"}
    roof["ms_per_launch"] = dom_ms

    kernels = {}
    for n in names:
        ms = per_kernel[n] / args.steps
        kernels[n] = {"ms_per_launch": ms, "share": per_kernel[n] / max(sum(per_kernel.values()),
                                                                         1e-9)}
        if kflops.get(n):
            kernels[n]["alg_tflops"] = kflops[n] / (ms * 1e-3) / 1e12

    # end to end through the C ABI's host-buffer runtime (fa_host_step): every
    # step copies its inputs in from pinned host memory and its outputs
    # (o, lse, dq, dk, dv) back; copies of neighbouring steps overlap the
    # kernels of the current one; host wall clock from the first call to the
    # end of fa_host_wait
    e2e = None
    if not args.no_e2e:
        del o, lse, D, dq, dk, dv  # the plan holds its own device buffers
        torch.cuda.empty_cache()
        sets = []
        for i in range(2):  # two host buffer sets, alternated between steps
            ins = [t.pin_memory() for t in (q_h, k_h, v_h, dO_h)]
            outs = [torch.empty(q_h.shape, dtype=torch.bfloat16).pin_memory() for _ in range(4)]
            outs.append(torch.empty((w.B, w.H, w.N), dtype=torch.float32).pin_memory())
            sets.append((ins, outs))
        plan = fa.HostPlan(w.B, w.H, w.N, w.d, causal=causal, scale=scale, device=dev)

        def e2e_step(i):
            (qh, kh, vh, dOh), (oh, dqh, dkh, dvh, lseh) = sets[i % 2]
            plan.step(qh, kh, vh, dOh, oh, lseh, dqh, dkh, dvh)

        for i in range(max(2, args.warmup // 2)):
            e2e_step(i)
        plan.wait()
        n_e2e = max(4, args.steps // 4)
        torch.cuda.synchronize(dev)
        barrier(world)
        t0 = time.perf_counter()
        for i in range(n_e2e):
            e2e_step(i)
        plan.wait()
        e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3, world) / n_e2e
        plan.close()
        h2d = sum(t.numel() * t.element_size() for t in sets[0][0])
        d2h = sum(t.numel() * t.element_size() for t in sets[0][1])
        e2e = {"value": aggregate_rate(f_fwd + f_bwd, world, e_ms * 1e-3) / 1e12,
               "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
               "steps": n_e2e,
               "how": "fa_host_step (C ABI, pinned host buffers, two-slot copy/compute "
                      "pipeline), host wall clock"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        dt, fl, cores, desc, extrap = oracle_baseline(w, causal, q_h, k_h, v_h, dO_h)
        cpu = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": desc}
        if extrap is not None:
            cpu["extrapolated_full_problem_s"] = extrap

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": workload_config(w, causal),
            "fwd_tflops": fwd_tf, "bwd_tflops": bwd_tf,
            "fwd_frac_of_peak": fwd_tf / peak, "bwd_frac_of_peak": bwd_tf / peak,
            "peak_tflops": peak, "peak_source": f"{peak_kind} bf16, {peak_src}",
            "kernels": kernels, "roofline": roof, "diagnostics": diag, "cpu_baseline": cpu,
            "e2e": e2e, "gpu_launches": 4 * args.steps, "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    return 0


def run_variant(args, world, rank, local, fa, w, causal, tensors, stream, dev):
    """Block-sparse and / or dropout step: fa_forward_blocksparse +
    fa_backward_blocksparse (--block-mask), fa_forward_dropout +
    fa_backward_dropout (--dropout, with the block mask if one is given)."""
    q, k, v, dO = tensors
    if args.block_mask:
        mask_cpu = band_mask(args.block_mask, w.N)
        mask = mask_cpu.to(dev)
    else:
        mask_cpu = mask = None
    p_drop = args.dropout or 0.0
    seed = 0x5EED
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_backward_workspace_size(w.B, w.H, w.N, w.d), dtype=torch.uint8,
                     device=dev)

    def step(ev=None, offset=0):
        if p_drop > 0.0:
            fa.fa_forward_dropout(q, k, v, p_drop, seed, offset, causal=causal, scale=w.scale,
                                  block_mask=mask, o=o, lse=lse, stream=stream)
        else:
            fa.fa_forward_blocksparse(q, k, v, mask, causal=causal, scale=w.scale, o=o, lse=lse,
                                      stream=stream)
        if ev is not None:
            ev[1].record(stream)
        if p_drop > 0.0:
            fa.fa_backward_dropout(q, k, v, o, dO, lse, p_drop, seed, offset, causal=causal,
                                   scale=w.scale, block_mask=mask, dq=dq, dk=dk, dv=dv,
                                   workspace=ws, stream=stream)
        else:
            fa.fa_backward_blocksparse(q, k, v, o, dO, lse, mask, causal=causal, scale=w.scale,
                                       dq=dq, dk=dk, dv=dv, workspace=ws, stream=stream)
        if ev is not None:
            ev[2].record(stream)

    for i in range(args.warmup):
        step(offset=i)
    torch.cuda.synchronize(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    barrier(world)
    clocks.start()
    for s_ in range(args.steps):
        evs[s_][0].record(stream)
        step(evs[s_], offset=args.warmup + s_)  # a fresh dropout mask every step
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    st, detail = fa.fa_get_device_error(stream)
    if st != 0:
        raise RuntimeError(f"device error: {st} {detail:#x}")
    fwd_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps
    bwd_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / args.steps
    ms = max_over_ranks(fwd_ms + bwd_ms, world)
    if mask_cpu is not None:
        E = kept_elements(mask_cpu, w.N, causal) * w.B * w.H
    else:
        E = w.B * w.H * w.N * w.N * (0.5 if causal else 1.0)
    f_fwd, f_bwd = 4.0 * w.d * E, 10.0 * w.d * E
    peaks, peak_src = read_peaks()
    peak = peaks["bf16_tflops"]
    fwd_tf = f_fwd / (fwd_ms * 1e-3) / 1e12
    if rank == 0:
        dense = w.B * w.H * w.N * w.N * (0.5 if causal else 1.0)
        cfg = workload_config(w, causal)
        if mask_cpu is not None:
            cfg.update({"block_mask": args.block_mask, "kept_fraction": E / dense})
        if p_drop > 0.0:
            cfg.update({"dropout_p": p_drop, "dropout_rng": "Philox4x32-10, new offset per step"})
        what = ", ".join(x for x in ("block-sparse, FLOPs of kept tiles" if mask_cpu is not None
                                     else "", f"dropout p={p_drop}" if p_drop > 0 else "") if x)
        line = {
            "metric": METRIC + f" ({what})",
            "value": aggregate_rate(f_fwd + f_bwd, world, ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": cfg, "fwd_tflops": fwd_tf,
            "bwd_tflops": f_bwd / (bwd_ms * 1e-3) / 1e12,
            "roofline": {"bound": "tensor", "kernel": "fwd", "achieved": fwd_tf, "peak": peak,
                         "unit": "TFLOP/s", "frac": fwd_tf / peak,
                         "traffic": (captured_traffic("fwd_dropout", w.name)
                                     if (p_drop == 0.1 and mask_cpu is None
                                         and causal == w.causal[0]) else None),
                         "peak_kind": f"burst bf16 ({peak_src})"},
            "gpu_launches": 4 * args.steps, "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    return 0


def run_fp8(args, world, rank, local, fa, w, causal, stream, dev):
    """e4m3 forward step: fa_forward_fp8 on the workload's q, k, v quantised
    per tensor (fa_inputs.make_fp8_inputs).  Tensor-bound: FLOPs of the two
    products (4 N^2 d per head, halved when causal) against the fp8 peak =
    measured bf16 peak x 2 (the nominal fp8 : bf16 ratio)."""
    from fa_inputs import make_fp8_inputs

    if w.d != 128:
        raise SystemExit("--fp8 needs a d = 128 workload")
    q8, k8, _, vt8, ds = make_fp8_inputs(w.B, w.H, w.N, w.d, w.seed, w.qk_mult)
    q, k, vt = (t.view(torch.uint8).to(dev) for t in (q8, k8, vt8))
    del q8, k8, vt8
    o = torch.empty((w.B, w.H, w.N, w.d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)

    def step():
        fa.fa_forward_fp8(q, k, vt, *ds, causal=causal, scale=w.scale, o=o, lse=lse,
                          stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    barrier(world)
    clocks.start()
    for s_ in range(args.steps):
        evs[s_][0].record(stream)
        step()
        evs[s_][1].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    st, detail = fa.fa_get_device_error(stream)
    if st != 0:
        raise RuntimeError(f"device error: {st} {detail:#x}")
    ms = max_over_ranks(sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps, world)
    f_fwd, _ = flops(w, causal)
    peaks, peak_src = read_peaks()
    peak = 2.0 * peaks["bf16_tflops"]
    tf = f_fwd / (ms * 1e-3) / 1e12
    if rank == 0:
        cfg = workload_config(w, causal)
        cfg.update({"inputs": "e4m3 q, k, V^T with per-tensor descales (amax / 448)",
                    "l2": "inputs (q, k, v e4m3 = 201 MB per step) larger than L2"})
        line = {
            "metric": "attention forward TFLOP/s at 1 GB300, e4m3 inputs",
            "value": world * tf, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 (fp32 accumulate)",
            "data": "synthetic", "config": cfg,
            "roofline": {"bound": "tensor", "kernel": "fwd_fp8", "achieved": tf, "peak": peak,
                         "unit": "TFLOP/s", "frac": tf / peak,
                         "traffic": (captured_traffic("fwd_fp8", w.name)
                                     if causal == w.causal[0] else None),
                         "peak_kind": f"fp8 = 2 x burst bf16 ({peak_src})"},
            "gpu_launches": args.steps, "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    return 0


def run_decode(args, world, rank, local, fa, w, tensors, stream, dev):
    """Decode step: the last --decode query rows against the whole key/value
    cache of the workload (causal: query i at position N - Nq + i).  HBM-bound:
    reported as GB/s of algorithmic bytes (K, V, q read once; o, lse written)."""
    q_full, k, v = tensors
    Nq = int(args.decode)
    q = q_full[:, :, w.N - Nq:].contiguous()
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, Nq), dtype=torch.float32, device=dev)
    ws = torch.empty(fa.fa_decode_workspace_size(w.B, w.H, Nq, w.N, w.d), dtype=torch.uint8,
                     device=dev)
    # inputs larger than L2 between steps: rotate over copies of the cache
    copies = max(1, int((300e6 // (2 * k.numel() * 2)) + 1))
    caches = [(k, v)] + [(k.clone(), v.clone()) for _ in range(copies - 1)]

    def step(i):
        kk, vv = caches[i % len(caches)]
        fa.fa_decode(q, kk, vv, causal=True, scale=w.scale, o=o, lse=lse, workspace=ws,
                     stream=stream)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    barrier(world)
    clocks.start()
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clk = clocks.stop()
    st, detail = fa.fa_get_device_error(stream)
    if st != 0:
        raise RuntimeError(f"device error: {st} {detail:#x}")
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)
    nbytes = (2 * k.numel() + 2 * q.numel()) * 2 + lse.numel() * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    peaks, peak_src = read_peaks()
    if rank == 0:
        cfg = {"workload": f"decode_q{Nq}_{w.name}", "B": w.B, "H": w.H, "Nq": Nq, "Nk": w.N,
               "d": w.d, "causal": True,
               "l2": f"{len(caches)} rotating copies of the K/V cache ({2 * k.numel() * 2 / 1e6:.0f} MB each)"}
        line = {
            "metric": "attention decode step HBM GB/s (K/V cache read once)", "value": world * gbs,
            "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic", "config": cfg,
            "roofline": {"bound": "hbm", "kernel": "decode_split_tc+decode_combine", "achieved": gbs,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                         "traffic": captured_traffic("decode", cfg["workload"]),
                         "peak_kind": peak_src},
            "gpu_launches": 2 * args.steps, "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=sorted(WORKLOADS) + sorted(SCALING_WORKLOADS))
    ap.add_argument("--causal", type=int, default=None, help="override the workload's mask mode")
    ap.add_argument("--block-mask", default=None,
                    help="time the block-sparse path with mask band:W[:G] (tiles of 128)")
    ap.add_argument("--dropout", type=float, default=None,
                    help="time the dropout path with this probability (0 < p < 1)")
    ap.add_argument("--fp8", action="store_true",
                    help="time the e4m3 forward (fa_forward_fp8) on the workload")
    ap.add_argument("--decode", type=int, default=None,
                    help="time the decode step with this many query rows (<= 16)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        rc = run_reference(args, world, rank)
    else:
        rc = run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return rc


if __name__ == "__main__":
    sys.exit(main())
