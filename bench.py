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


NVML_REASONS = {  # clocks-event reason bits of nvmlDeviceGetCurrentClocksEventReasons
    0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
    0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


class NvmlClocks:
    """Read-only NVML queries (ctypes on the driver's libnvidia-ml): SM clock,
    its maximum, power draw and the active clocks-event reasons of one GPU."""

    def __init__(self, device_index: int):
        import ctypes

        self.c = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.lib = lib
        self.h = ctypes.c_void_p()
        props = torch.cuda.get_device_properties(device_index)
        uuid = getattr(props, "uuid", None)
        ok = False
        if uuid is not None:
            ok = lib.nvmlDeviceGetHandleByUUID(f"GPU-{uuid}".encode(), ctypes.byref(self.h)) == 0
        if not ok:
            cnt = ctypes.c_uint()
            if lib.nvmlDeviceGetCount_v2(ctypes.byref(cnt)) != 0 or cnt.value != 1:
                raise RuntimeError("cannot match the CUDA device to an NVML device")
            if lib.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self.h)) != 0:
                raise RuntimeError("nvmlDeviceGetHandleByIndex failed")
        self.reason_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) != 0:
            raise RuntimeError("nvmlDeviceGetMaxClockInfo failed")
        self.max_mhz = float(mx.value)

    def sample(self):
        c = self.c
        clk, mw, rs = c.c_uint(), c.c_uint(), c.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, 1, c.byref(clk)) != 0:
            return None
        self.lib.nvmlDeviceGetPowerUsage(self.h, c.byref(mw))
        self.reason_fn(self.h, c.byref(rs))
        return float(clk.value), mw.value / 1000.0, int(rs.value)


class ClockSampler:
    """SM clock and throttle-reason samples during a timed region.

    NVML is polled every 2 ms from a thread (so that even a 40 ms region gives
    some twenty samples); where NVML cannot be loaded, nvidia-smi samples every
    200 ms instead.  mark_load() / mark_done() bracket the timed region on the
    host: samples taken in between are the ones under load."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_S = 0.002

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None
        self.nvml = None
        self.thread = None
        self.samples = []
        self.t_load = self.t_done = None

    def start(self):
        import threading

        try:
            self.nvml = NvmlClocks(self.dev)
        except Exception:
            self.nvml = None
        if self.nvml is not None:
            self.stop_flag = threading.Event()

            def run():
                while not self.stop_flag.is_set():
                    s = self.nvml.sample()
                    if s is not None:
                        self.samples.append((time.perf_counter(),) + s)
                    time.sleep(self.INTERVAL_S)

            self.thread = threading.Thread(target=run, daemon=True)
            self.thread.start()
            return
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

    def mark_load(self):
        self.t_load = time.perf_counter()

    def mark_done(self):
        self.t_done = time.perf_counter()

    def stop(self):
        if self.thread is not None:
            self.stop_flag.set()
            self.thread.join(timeout=5)
            return self._summary_nvml()
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
                "samples": len(rows), "samples_under_load": None,
                "source": "nvidia-smi, 200 ms"}

    def _summary_nvml(self):
        if not self.samples:
            return None
        t0 = self.t_load if self.t_load is not None else -math.inf
        t1 = self.t_done if self.t_done is not None else math.inf
        load = [s for s in self.samples if t0 <= s[0] <= t1] or self.samples
        reasons = sorted({name for s in load for bit, name in NVML_REASONS.items()
                          if s[3] & bit})
        return {"sm_mhz": statistics.median(s[1] for s in load),
                "sm_max_mhz": self.nvml.max_mhz,
                "sm_mhz_min": min(s[1] for s in load),
                "power_w_max": max(s[2] for s in load),
                "reasons": reasons, "samples": len(self.samples),
                "samples_under_load": len([s for s in self.samples if t0 <= s[0] <= t1]),
                "source": "NVML every 2 ms (read-only queries)"}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        if args.impl == "ours":
            # each rank on its own GPU before the first collective (a barrier
            # issued earlier would have to guess the rank's device)
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
        else:
            dist.init_process_group("gloo")
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


L2_BYTES = 129e6  # GB300's L2
FLUSH_BYTES = 256 << 20


def step_bytes(w):
    """q, k, v, o, dO of one step (bf16)."""
    return 5 * w.B * w.H * w.N * w.d * 2


def l2_label(nbytes, what="q,k,v,o,dO together"):
    """How a timed region keeps L2 from serving the next step's inputs: they
    exceed L2, or a buffer larger than L2 is rewritten before every step."""
    if nbytes > L2_BYTES:
        return f"inputs larger than L2 ({what} {nbytes / 1e6:.0f} MB per step > 129 MB)"
    return (f"L2 flushed before every step ({FLUSH_BYTES >> 20} MB buffer rewritten outside the "
            f"timed events; {what} {nbytes / 1e6:.0f} MB fit in L2)")


def l2_flush_buffer(nbytes, dev):
    """The buffer l2_label's flush rewrites, or None when the inputs exceed L2."""
    return None if nbytes > L2_BYTES else torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)


def workload_config(w, causal):
    return {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "causal": causal,
            "scale": w.scale, "qk_mult": w.qk_mult, "seed": w.seed, "l2": l2_label(step_bytes(w))}


KERNELS = ["fwd", "bwd_pre", "bwd_dq", "bwd_dkdv"]

# MUFU (special-function unit) rate of ex2 on this part: 32 results per clock
# per SM.  Derived from counters, not from a table: in ncu captures of the
# step kernels the XU pipe's utilisation (sm__inst_executed_pipe_xu, % of peak)
# equals each kernel's ex2 count per second / (32 x SMs x SM clock) to within
# 1.3 points (forward 26.6 % against 25.3 %, dQ 16.0 % against 15.6 %, dK/dV
# 15.4 % against 15.0 %), i.e. ncu's peak is one warp-wide XU instruction per
# clock per SM; the peak is that x SMs x the sampled SM clock.
MUFU_EX2_PER_CLK_PER_SM = 32


def kernel_work(w, causal):
    """Per launch of each step kernel: `flops` = the method's matmul work
    counted once (forward S and P V; backward S recompute, dP, dV and dK in
    the dK/dV kernel and dQ = dS K alone in the dQ kernel, so the two add up
    to the step's 10 N^2 d), `exec_flops` = the matmul work the kernel
    executes (the dQ kernel recomputes S and dP and forms B = P K for the
    exact D), `exp2` = exponentials of visible score elements, `bytes` = the
    algorithmic HBM bytes (every tensor once)."""
    f = 0.5 if causal else 1.0
    base = w.B * w.H * w.N * w.N * w.d * f
    e = w.B * w.H * w.N * w.N * f
    t = w.B * w.H * w.N * w.d * 2  # one bf16 [B,H,N,d] tensor
    r = w.B * w.H * w.N * 4  # one fp32 [B,H,N] vector
    return {
        "fwd": {"flops": 4 * base, "exec_flops": 4 * base, "exp2": e, "bytes": 4 * t + r},
        "bwd_pre": {"flops": 0.0, "exec_flops": 0.0, "exp2": 0.0, "bytes": 2 * t + r},
        # reads q, k, v, dO, lse, D~; writes dq and the exact D
        "bwd_dq": {"flops": 2 * base, "exec_flops": 8 * base, "exp2": e, "bytes": 5 * t + 3 * r},
        # reads q, k, v, dO, lse, D; writes dk, dv
        "bwd_dkdv": {"flops": 8 * base, "exec_flops": 8 * base, "exp2": e,
                     "bytes": 6 * t + 2 * r},
    }


def make_step(fa, w, causal, dev, stream, backward=True, inputs=None):
    """Device tensors of one workload and a step(ev) that launches its kernels
    (forward, D pre-pass, dQ, dK/dV) and records ev[i + 1] after kernel i."""
    q_h, k_h, v_h, dO_h = inputs if inputs is not None else \
        make_inputs(w.B, w.H, w.N, w.d, w.seed, w.qk_mult, with_dO=backward)
    q, k, v = (t.to(dev) for t in (q_h, k_h, v_h))
    dO = dO_h.to(dev) if backward else None
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    D = torch.empty_like(lse)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3)) if backward else (None,) * 3
    names = KERNELS if backward else KERNELS[:1]

    def step(ev=None):
        fa.fa_forward(q, k, v, causal=causal, scale=w.scale, o=o, lse=lse, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        if not backward:
            return
        fa.fa_backward_preprocess(o, dO, D, stream=stream)
        if ev is not None:
            ev[2].record(stream)
        fa.fa_backward_dq(q, k, v, dO, lse, D, causal=causal, scale=w.scale, dq=dq,
                          stream=stream)
        if ev is not None:
            ev[3].record(stream)
        fa.fa_backward_dkdv(q, k, v, dO, lse, D, causal=causal, scale=w.scale, dk=dk, dv=dv,
                            stream=stream)
        if ev is not None:
            ev[4].record(stream)

    return step, names


def time_kernels(fa, step, names, steps, warmup, dev, stream, flush=None):
    """Per-kernel CUDA-event times (ms, summed over `steps`) of step(), after
    `warmup` untimed steps; with `flush` (a buffer larger than L2) the buffer
    is rewritten before every step, outside the timed events."""
    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
           for _ in range(steps)]
    for s_ in range(steps):
        if flush is not None:
            flush.fill_(s_ & 0xff)
        evs[s_][0].record(stream)
        step(evs[s_])
    torch.cuda.synchronize(dev)
    st, detail = fa.fa_get_device_error(stream)
    if st != 0:
        raise RuntimeError(f"device error: {st} {detail:#x}")
    return {n: sum(e[i].elapsed_time(e[i + 1]) for e in evs) for i, n in enumerate(names)}


def kernel_table(w, causal, per_kernel_ms, steps, peak, hbm_gbs, mufu_peak):
    """Per-kernel rates: algorithmic and executed TFLOP/s against the bf16
    peak, exp2/s against the MUFU peak, algorithmic HBM GB/s, time per launch."""
    work = kernel_work(w, causal)
    total = max(sum(per_kernel_ms.values()), 1e-9)
    out = {}
    for n, tot in per_kernel_ms.items():
        ms = tot / steps
        sec = ms * 1e-3
        k = {"ms_per_launch": ms, "us_per_launch": ms * 1e3, "share": tot / total}
        wk = work[n]
        if wk["flops"]:
            k["alg_tflops"] = wk["flops"] / sec / 1e12
            k["frac_of_peak"] = k["alg_tflops"] / peak
            k["exec_tflops"] = wk["exec_flops"] / sec / 1e12
        if wk["exp2"]:
            k["exp2_per_s"] = wk["exp2"] / sec
            k["exp2_frac_of_mufu"] = k["exp2_per_s"] / mufu_peak
        k["hbm_gbs"] = wk["bytes"] / sec / 1e9
        k["hbm_frac"] = k["hbm_gbs"] / hbm_gbs
        out[n] = k
    return out


def secondary_record(fa, name, dev, stream, steps, peaks, mufu_peak, causal=None, flush=False):
    """Forward and backward TFLOP/s of another workload, timed in this run on
    resident inputs (its own warm-up).  Inputs larger than L2, or with
    `flush`, L2 rewritten (256 MB) before every step."""
    w = {**WORKLOADS, **SCALING_WORKLOADS}[name]
    causal = w.causal[0] if causal is None else causal
    step, names = make_step(fa, w, causal, dev, stream)
    fbuf = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if flush else None
    per = time_kernels(fa, step, names, steps, 3, dev, stream, flush=fbuf)
    del fbuf
    f_fwd, f_bwd = flops(w, causal)
    fwd_ms = per["fwd"] / steps
    bwd_ms = sum(per[n] for n in names[1:]) / steps
    peak = peaks["bf16_tflops"]
    del step
    torch.cuda.empty_cache()
    return {"workload": name, "causal": causal, "steps": steps,
            "fwd_tflops": f_fwd / (fwd_ms * 1e-3) / 1e12,
            "bwd_tflops": f_bwd / (bwd_ms * 1e-3) / 1e12,
            "fwd_frac_of_peak": f_fwd / (fwd_ms * 1e-3) / 1e12 / peak,
            "bwd_frac_of_peak": f_bwd / (bwd_ms * 1e-3) / 1e12 / peak,
            "step_tflops": (f_fwd + f_bwd) / ((fwd_ms + bwd_ms) * 1e-3) / 1e12,
            "ms_per_step": fwd_ms + bwd_ms, "peak_tflops": peak,
            "kernels": kernel_table(w, causal, per, steps, peak, peaks["hbm_gbs"], mufu_peak),
            "l2": ("flushed before every step (256 MB buffer rewritten)" if flush
                   else "inputs larger than L2")}


def short_record(fa, name, dev, stream, steps, peaks, mufu_peak):
    """The short-sequence workloads, where tiles are few and launches short:
    per-kernel time per launch and algorithmic HBM GB/s as a share of the
    measured copy bandwidth, L2 flushed (256 MB rewritten) before every step."""
    w = WORKLOADS[name]
    causal = w.causal[0]
    step, names = make_step(fa, w, causal, dev, stream, backward=w.backward)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    per = time_kernels(fa, step, names, steps, 3, dev, stream, flush=flush)
    # host time to enqueue one step (the C ABI calls and their argument checks)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(8):
        step()
    enq_us = (time.perf_counter() - t0) * 1e6 / 8
    torch.cuda.synchronize(dev)
    del step, flush
    torch.cuda.empty_cache()
    f_fwd, f_bwd = flops(w, causal)
    ms = sum(per.values()) / steps
    return {"workload": name, "causal": causal, "steps": steps,
            "l2": "flushed before every step (256 MB buffer rewritten)",
            "us_per_step": ms * 1e3, "host_enqueue_us_per_step": enq_us,
            "step_tflops": (f_fwd + (f_bwd if w.backward else 0.0)) / (ms * 1e-3) / 1e12,
            "kernels": kernel_table(w, causal, per, steps, peaks["bf16_tflops"],
                                    peaks["hbm_gbs"], mufu_peak)}


def timed_variant(fa, step, steps, warmup, dev, stream):
    """Mean forward and backward ms of a variant_step over `steps` steps after
    `warmup` untimed ones, a new Philox offset every step."""
    for i in range(warmup):
        step(offset=i)
    torch.cuda.synchronize(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    for s_ in range(steps):
        evs[s_][0].record(stream)
        step(evs[s_], offset=warmup + s_)
    torch.cuda.synchronize(dev)
    st, detail = fa.fa_get_device_error(stream)
    if st != 0:
        raise RuntimeError(f"device error: {st} {detail:#x}")
    return (sum(e[0].elapsed_time(e[1]) for e in evs) / steps,
            sum(e[1].elapsed_time(e[2]) for e in evs) / steps)


def timed_launches(fa, step, steps, warmup, dev, stream):
    """Mean ms per step(i) over `steps` steps after `warmup` untimed ones."""
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        step(warmup + i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    st, detail = fa.fa_get_device_error(stream)
    if st != 0:
        raise RuntimeError(f"device error: {st} {detail:#x}")
    return e0.elapsed_time(e1) / steps


NEXT_ROW_STEPS = 10
NEXT_ROW_BAND = "band:8:1"
NEXT_ROW_DECODE = ("causal_b1h32n32768d128_qk2", 16)


def next_rows_record(fa, inputs, dev, stream, peaks, steps=NEXT_ROW_STEPS):
    """The widened rows, timed in this run on resident inputs larger than L2
    (3 warm-up steps each): dropout (p = 0.1, a new Philox offset per step,
    causal) and block-sparse (NEXT_ROW_BAND, non-causal) forward + backward
    and the e4m3 forward (causal) on the 8K workload; decode with 16 query
    rows against the 32-head 32K-token cache.  TFLOP/s count the method's
    work on the elements kept (block-sparse: kept tiles); `inputs` are the 8K
    workload's host tensors (None: drawn here)."""
    w = WORKLOADS[DEFAULT_WORKLOAD]
    peak = peaks["bf16_tflops"]
    if inputs is None:
        inputs = make_inputs(w.B, w.H, w.N, w.d, w.seed, w.qk_mult)
    tensors = tuple(t.to(dev) for t in inputs)
    dense = float(w.B * w.H * w.N * w.N)

    def rates(E, fwd_ms, bwd_ms):
        f_fwd, f_bwd = 4.0 * w.d * E, 10.0 * w.d * E
        return {"fwd_tflops": f_fwd / (fwd_ms * 1e-3) / 1e12,
                "bwd_tflops": f_bwd / (bwd_ms * 1e-3) / 1e12,
                "step_tflops": (f_fwd + f_bwd) / ((fwd_ms + bwd_ms) * 1e-3) / 1e12,
                "fwd_frac_of_peak": f_fwd / (fwd_ms * 1e-3) / 1e12 / peak,
                "ms_per_step": fwd_ms + bwd_ms}

    out = {"steps": steps, "peak_tflops": peak}
    step = variant_step(fa, w, True, tensors, None, 0.1, dev, stream)
    out["dropout"] = {"workload": w.name, "causal": True, "p": 0.1,
                      "rng": "Philox4x32-10, new offset per step",
                      **rates(0.5 * dense, *timed_variant(fa, step, steps, 3, dev, stream))}
    mask_cpu = band_mask(NEXT_ROW_BAND, w.N)
    E = kept_elements(mask_cpu, w.N, False) * w.B * w.H
    step = variant_step(fa, w, False, tensors, mask_cpu.to(dev), 0.0, dev, stream)
    out["blocksparse"] = {"workload": w.name, "causal": False, "block_mask": NEXT_ROW_BAND,
                          "kept_fraction": E / dense,
                          **rates(E, *timed_variant(fa, step, steps, 3, dev, stream))}
    del step, tensors
    torch.cuda.empty_cache()

    step = fp8_step(fa, w, True, dev, stream)
    ms = timed_launches(fa, lambda i: step(), steps, 3, dev, stream)
    tf = flops(w, True)[0] / (ms * 1e-3) / 1e12
    out["fp8_forward"] = {"workload": w.name, "causal": True, "tflops": tf,
                          "frac_of_fp8_peak": tf / (2.0 * peak), "ms_per_launch": ms,
                          "peak": "fp8 = 2 x burst bf16 (the nominal fp8 : bf16 ratio)"}
    del step
    torch.cuda.empty_cache()

    name, Nq = NEXT_ROW_DECODE
    wd = WORKLOADS[name]
    qkv = tuple(t.to(dev) for t in make_inputs(wd.B, wd.H, wd.N, wd.d, wd.seed, wd.qk_mult,
                                               with_dO=False)[:3])
    step, nbytes, n_caches, _ = decode_step(fa, wd, qkv, Nq, dev, stream)
    ms = timed_launches(fa, step, steps, 3, dev, stream)
    gbs = nbytes / (ms * 1e-3) / 1e9
    out["decode"] = {"workload": f"decode_q{Nq}_{name}", "Nq": Nq, "Nk": wd.N, "hbm_gbs": gbs,
                     "hbm_frac": gbs / peaks["hbm_gbs"], "us_per_step": ms * 1e3,
                     "cache_copies": n_caches}
    del step, qkv
    torch.cuda.empty_cache()
    return out


def run_ours(args, world, rank, local):
    import exact_io_aware_16_gb300 as fa
    from exact_io_aware_16_gb300 import build as fabuild

    if rank == 0:  # one build; the other ranks load it after the barrier
        fabuild.build()
    barrier(world)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = {**WORKLOADS, **SCALING_WORKLOADS}[args.workload]
    causal = w.causal[0] if args.causal is None else bool(args.causal)
    scale = w.scale
    inputs = make_inputs(w.B, w.H, w.N, w.d, w.seed, w.qk_mult)
    q_h, k_h, v_h, dO_h = inputs
    stream = torch.cuda.current_stream(dev)
    if args.fp8:
        return run_fp8(args, world, rank, local, fa, w, causal, stream, dev)
    if args.block_mask or args.dropout or args.decode:
        tensors = tuple(t.to(dev) for t in inputs)
        if args.decode:
            return run_decode(args, world, rank, local, fa, w, tensors[:3], stream, dev)
        return run_variant(args, world, rank, local, fa, w, causal, tensors, stream, dev)
    step, names = make_step(fa, w, causal, dev, stream, inputs=inputs)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    st, detail = fa.fa_get_device_error(stream)
    if st != 0:
        raise RuntimeError(f"device error during warm-up: {st} {detail:#x}")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    flush = l2_flush_buffer(step_bytes(w), dev)
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.start()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks.mark_load()
    t_start.record(stream)
    h0 = time.perf_counter()
    n_enq = min(args.steps, 8)  # before the launch queue can fill and block the host
    enqueue_us = 0.0
    for s in range(args.steps):
        if flush is not None:
            flush.fill_(s & 0xff)
        evs[s][0].record(stream)
        step(evs[s])
        if s + 1 == n_enq:
            enqueue_us = (time.perf_counter() - h0) * 1e6 / n_enq  # host side, per step
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    clocks.mark_done()
    barrier(world)
    clk = clocks.stop()
    st, detail = fa.fa_get_device_error(stream)
    if st != 0:
        raise RuntimeError(f"device error in timed region: {st} {detail:#x}")
    per_kernel = {n: 0.0 for n in names}
    for s in range(args.steps):
        for i, n in enumerate(names):
            per_kernel[n] += evs[s][i].elapsed_time(evs[s][i + 1])
    # with a flush between steps the step is its kernels' events (the flush outside them)
    total_ms = t_start.elapsed_time(t_end) if flush is None else sum(per_kernel.values())
    del flush
    total_ms_max = max_over_ranks(total_ms, world)
    ms_per_step = total_ms_max / args.steps
    f_fwd, f_bwd = flops(w, causal)
    value = aggregate_rate(f_fwd + f_bwd, world, ms_per_step * 1e-3) / 1e12

    peaks, peak_src = read_peaks()
    long_region = total_ms > 1000.0
    peak = peaks["bf16_tflops_sustained"] if long_region else peaks["bf16_tflops"]
    peak_kind = "sustained" if long_region else "burst"
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sm_mhz = (clk or {}).get("sm_mhz") or peaks.get("sm_max_mhz", 2070.0)
    mufu_peak = MUFU_EX2_PER_CLK_PER_SM * num_sms * sm_mhz * 1e6
    fwd_ms = per_kernel["fwd"] / args.steps
    bwd_ms = (per_kernel["bwd_pre"] + per_kernel["bwd_dkdv"] + per_kernel["bwd_dq"]) / args.steps
    fwd_tf = f_fwd / (fwd_ms * 1e-3) / 1e12
    bwd_tf = f_bwd / (bwd_ms * 1e-3) / 1e12
    kernels = kernel_table(w, causal, per_kernel, args.steps, peak, peaks["hbm_gbs"], mufu_peak)
    fwd_bytes, bwd_bytes = alg_bytes(w)
    diag = {
        "fwd_hbm_gbs": fwd_bytes / (fwd_ms * 1e-3) / 1e9,
        "fwd_hbm_frac": fwd_bytes / (fwd_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
        "bwd_hbm_gbs": bwd_bytes / (bwd_ms * 1e-3) / 1e9,
        "bwd_hbm_frac": bwd_bytes / (bwd_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
        "fwd_exp2_per_s": kernels["fwd"]["exp2_per_s"],
        "mufu_peak_exp2_per_s": mufu_peak,
        "mufu_peak_derivation": (f"{MUFU_EX2_PER_CLK_PER_SM} ex2 per clock per SM (the XU "
                                 f"pipe's peak in ncu's counters on this part) x {num_sms} SMs "
                                 f"x {sm_mhz:.0f} MHz (median SM clock in the timed region)"),
        "host_enqueue_us_per_step": enqueue_us,
        "device_us_per_step": ms_per_step * 1e3,
    }

    # dominant kernel and its roofline: the method's work of that kernel alone,
    # counted once (kernel_work)
    dom = max(names, key=lambda n: per_kernel[n])
    dom_ms = per_kernel[dom] / args.steps
    trace = captured_traffic(dom, w.name) if causal == w.causal[0] else None
    if dom == "bwd_pre":
        ach = kernels[dom]["hbm_gbs"]
        roof = {"bound": "hbm", "kernel": dom, "achieved": ach, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": ach / peaks["hbm_gbs"], "traffic": trace}
    else:
        ach = kernels[dom]["alg_tflops"]
        roof = {"bound": "tensor", "kernel": dom, "achieved": ach, "peak": peak,
                "unit": "TFLOP/s", "frac": ach / peak, "traffic": trace,
                "peak_kind": f"{peak_kind} bf16 ({peak_src})",
                "work": "the method's matmuls of this kernel counted once (dK/dV 8 N^2 d, "
                        "dQ 2 N^2 d, forward 4 N^2 d per head, x1/2 causal)"}
    roof["ms_per_launch"] = dom_ms

    # headline-adjacent workloads, timed in this run (rank 0, one GPU)
    secondary = short = config2 = next_rows = None
    if rank == 0 and world == 1 and not args.no_secondary:
        del step
        torch.cuda.empty_cache()
        sec_steps = max(3, min(args.steps, 20))
        secondary = secondary_record(fa, "causal_b1h32n32768d128_qk2", dev, stream, sec_steps,
                                     peaks, mufu_peak)
        config2 = [secondary_record(fa, "b4h16n2048d64", dev, stream, sec_steps, peaks,
                                    mufu_peak, causal=c, flush=True) for c in (True, False)]
        short = [short_record(fa, n, dev, stream, 50, peaks, mufu_peak)
                 for n in ("fwd_b1h2n256d64", "short_b64h12n512d64")]
        next_rows = next_rows_record(fa, inputs if w.name == DEFAULT_WORKLOAD else None, dev,
                                     stream, peaks)

    # end to end through the C ABI's host-buffer runtime (fa_host_step): every
    # step copies its inputs in from pinned host memory and its outputs
    # (o, lse, dq, dk, dv) back; copies of neighbouring steps overlap the
    # kernels of the current one; host wall clock from the first call to the
    # end of fa_host_wait, over at least E2E_MIN_STEPS steps and E2E_MIN_SECONDS
    e2e = None
    if not args.no_e2e:
        step = None
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

        n_warm = max(4, args.warmup)
        e2e_step(0)  # the first step pays one-time set-up: not part of the estimate
        plan.wait()
        t0 = time.perf_counter()
        for i in range(n_warm):
            e2e_step(i + 1)
        plan.wait()
        est = (time.perf_counter() - t0) / n_warm
        # a short burst includes filling and draining the copy pipeline: aim
        # 50 % above the minimum
        n_e2e = int(min(E2E_MAX_STEPS,
                        max(E2E_MIN_STEPS, math.ceil(1.5 * E2E_MIN_SECONDS / est))))
        torch.cuda.synchronize(dev)
        barrier(world)
        eclk = ClockSampler(local)
        eclk.start()
        eclk.mark_load()
        t0 = time.perf_counter()
        for i in range(n_e2e):
            e2e_step(i)
        plan.wait()
        e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3, world) / n_e2e
        eclk.mark_done()
        e_clk = eclk.stop()
        plan.close()
        h2d = sum(t.numel() * t.element_size() for t in sets[0][0])
        d2h = sum(t.numel() * t.element_size() for t in sets[0][1])
        e2e = {"value": aggregate_rate(f_fwd + f_bwd, world, e_ms * 1e-3) / 1e12,
               "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
               "steps": n_e2e, "seconds": n_e2e * e_ms * 1e-3,
               "how": "fa_host_step (C ABI, pinned host buffers, two-slot copy/compute "
                      "pipeline), host wall clock"}
        if e_clk:  # the SM clock the kernels ran at here (the power cap lowers it in long runs)
            e2e["clocks"] = {k: e_clk[k] for k in ("sm_mhz", "sm_mhz_min", "power_w_max",
                                                    "reasons", "samples_under_load")
                             if k in e_clk}

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
            "secondary": secondary, "config2": config2, "short_sequence": short,
            "next_rows": next_rows,
        }
        print(json.dumps(line), flush=True)
    return 0


E2E_MIN_STEPS = 100
E2E_MIN_SECONDS = 1.0
E2E_MAX_STEPS = 4000


def variant_step(fa, w, causal, tensors, mask, p_drop, dev, stream, seed=0x5EED):
    """step(ev=None, offset=0) of the block-sparse and / or dropout path:
    fa_forward_blocksparse + fa_backward_blocksparse (mask given, p_drop 0),
    fa_forward_dropout + fa_backward_dropout (p_drop > 0, with the mask if
    given) at Philox offset `offset`; ev[1] is recorded after the forward and
    ev[2] after the backward."""
    q, k, v, dO = tensors
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

    return step


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
    step = variant_step(fa, w, causal, (q, k, v, dO), mask, p_drop, dev, stream)

    for i in range(args.warmup):
        step(offset=i)
    torch.cuda.synchronize(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    flush = l2_flush_buffer(step_bytes(w), dev)
    clocks = ClockSampler(local)
    barrier(world)
    clocks.start()
    for s_ in range(args.steps):
        if flush is not None:
            flush.fill_(s_ & 0xff)
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


def fp8_step(fa, w, causal, dev, stream):
    """step() of the e4m3 forward on the workload's q, k, v quantised per
    tensor (fa_inputs.make_fp8_inputs; V transposed per head); d = 128."""
    from fa_inputs import make_fp8_inputs

    q8, k8, _, vt8, ds = make_fp8_inputs(w.B, w.H, w.N, w.d, w.seed, w.qk_mult)
    q, k, vt = (t.view(torch.uint8).to(dev) for t in (q8, k8, vt8))
    del q8, k8, vt8
    o = torch.empty((w.B, w.H, w.N, w.d), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)

    def step():
        fa.fa_forward_fp8(q, k, vt, *ds, causal=causal, scale=w.scale, o=o, lse=lse,
                          stream=stream)

    return step


def run_fp8(args, world, rank, local, fa, w, causal, stream, dev):
    """e4m3 forward step: fa_forward_fp8 on the workload's q, k, v quantised
    per tensor (fa_inputs.make_fp8_inputs).  Tensor-bound: FLOPs of the two
    products (4 N^2 d per head, halved when causal) against the fp8 peak =
    measured bf16 peak x 2 (the nominal fp8 : bf16 ratio)."""
    if w.d != 128:
        raise SystemExit("--fp8 needs a d = 128 workload")
    step = fp8_step(fa, w, causal, dev, stream)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    fp8_bytes = 3 * w.B * w.H * w.N * w.d + 2 * w.B * w.H * w.N * w.d  # e4m3 q, k, V^T; bf16 o
    flush = l2_flush_buffer(fp8_bytes, dev)
    clocks = ClockSampler(local)
    barrier(world)
    clocks.start()
    for s_ in range(args.steps):
        if flush is not None:
            flush.fill_(s_ & 0xff)
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
                    "l2": l2_label(fp8_bytes, "e4m3 q, k, V^T and bf16 o")})
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


def decode_step(fa, w, tensors, Nq, dev, stream):
    """step(i) of the decode path: the last Nq query rows of the workload
    against its whole key/value cache (causal: query i at position N - Nq + i),
    rotating over enough copies of the cache that the inputs of consecutive
    steps exceed L2.  Returns (step, algorithmic bytes per step (K, V, q read
    once; o, lse written), copies, MB per cache)."""
    q_full, k, v = tensors
    q = q_full[:, :, w.N - Nq:].contiguous()
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, Nq), dtype=torch.float32, device=dev)
    ws = torch.empty(fa.fa_decode_workspace_size(w.B, w.H, Nq, w.N, w.d), dtype=torch.uint8,
                     device=dev)
    copies = max(1, int((300e6 // (2 * k.numel() * 2)) + 1))
    caches = [(k, v)] + [(k.clone(), v.clone()) for _ in range(copies - 1)]

    def step(i):
        kk, vv = caches[i % len(caches)]
        fa.fa_decode(q, kk, vv, causal=True, scale=w.scale, o=o, lse=lse, workspace=ws,
                     stream=stream)

    nbytes = (2 * k.numel() + 2 * q.numel()) * 2 + lse.numel() * 4
    return step, nbytes, len(caches), 2 * k.numel() * 2 / 1e6


def run_decode(args, world, rank, local, fa, w, tensors, stream, dev):
    """Decode step: the last --decode query rows against the whole key/value
    cache of the workload (causal: query i at position N - Nq + i).  HBM-bound:
    reported as GB/s of algorithmic bytes (K, V, q read once; o, lse written)."""
    Nq = int(args.decode)
    step, nbytes, n_caches, cache_mb = decode_step(fa, w, tensors, Nq, dev, stream)
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
    gbs = nbytes / (ms * 1e-3) / 1e9
    peaks, peak_src = read_peaks()
    if rank == 0:
        cfg = {"workload": f"decode_q{Nq}_{w.name}", "B": w.B, "H": w.H, "Nq": Nq, "Nk": w.N,
               "d": w.d, "causal": True,
               "l2": f"{n_caches} rotating copies of the K/V cache ({cache_mb:.0f} MB each)"}
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
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the records timed after the main one (32K, B4 H16 N2048 d64, "
                         "short sequences, the widened rows)")
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
