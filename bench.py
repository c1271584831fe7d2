#!/usr/bin/env python3
"""Benchmark of the selective-scan forward on B300 (one JSON line on rank 0).

Step = one ssm_scan_fwd over the Mamba-2.8B-like layer workload (bf16 io, fp32
state, batch 8, dim 5120, dstate 16, seqlen 2048, silu gate): softplus, ZOH
discretisation, recurrence, C contraction, D skip and gate fused in one kernel.
Inputs (672 MB per step) are larger than the 126 MB L2, so no flush is needed.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun every rank runs the same workload on its own GPU (independent
problems: weak scaling, no data-path collective); the timing is the max over
ranks and `value` counts the elements of all ranks.

The decode state update (batch 256, dim 5120, dstate 16, 1024 steps) is measured
after the main loop and reported under "decode".
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from selective_state_space_115_b300 import workloads as W  # noqa: E402

METRIC = "selective-scan elements/s (B·D·L) and achieved HBM GB/s vs B300 roofline"
CFG = W.SCAN_CONFIGS["2p8b"]
FLUSH_L2 = False
DEC = W.DECODE_CONFIGS["decode"]
DECODE_STEPS = DEC.steps
SM_COUNT = 148              # B300; the GPU arm reads the device's own count
SM_MAX_MHZ = 2032.0
EX2_PER_CLK_SM = 32          # measured on B300: ex2.approx.ftz.f32 per clock per SM
FP32_LANES_PER_CLK_SM = 128  # fp32 FMA lanes per clock per SM
FALLBACK_HBM_GBS = 6400.0
SUB_CONFIGS = ("130m", "long", "tiny")  # scan workloads reported beside the headline one
L2_BYTES = 126 * 2**20


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS, "sm_max_mhz": SM_MAX_MHZ}, "fallback"


def scan_bytes(cfg) -> int:
    """Algorithmic bytes of one scan: u, delta, z read and y written at io width,
    B and C read, fp32 A, D and bias read."""
    s = 2 if cfg.io == W.BF16 else 4
    e = cfg.batch * cfg.dim * cfg.seqlen
    n_io = 3 + (1 if cfg.gate else 0)
    return (n_io * e + 2 * cfg.batch * cfg.dstate * cfg.seqlen) * s + \
        4 * (cfg.dim * cfg.dstate + 2 * cfg.dim)


def decode_bytes(cfg) -> int:
    s = 2 if cfg.io == W.BF16 else 4
    ch = cfg.batch * cfg.dim
    return 2 * 4 * ch * cfg.dstate + (3 + (1 if cfg.gate else 0)) * s * ch + \
        2 * s * cfg.batch * cfg.dstate + 4 * (cfg.dim * cfg.dstate + 2 * cfg.dim)


def scan_roofline(cfg, ms: float, sms: int, sm_mhz: float, hbm_gbs: float) -> dict:
    """The method's roofline for one scan: the slowest of the algorithmic bytes at the
    HBM peak, the B*D*L*N exps at the ex2 peak and the 2 FMA per state update at the
    fp32 peak; the fraction is taken against the binding term."""
    nbytes, units = scan_bytes(cfg), cfg.updates
    ex2_rate = EX2_PER_CLK_SM * sms * sm_mhz * 1e6
    t_hbm = nbytes / (hbm_gbs * 1e9)
    t_ex2 = units / ex2_rate
    t_fp32 = 2 * units / (FP32_LANES_PER_CLK_SM * sms * sm_mhz * 1e6)
    t = ms * 1e-3
    if t_hbm >= max(t_ex2, t_fp32):
        ach = nbytes / t / 1e9
        r = {"bound": "hbm", "achieved": ach, "peak": hbm_gbs, "unit": "GB/s",
             "frac": ach / hbm_gbs}
    else:
        ach, peak = units / t / 1e12, ex2_rate / 1e12
        r = {"bound": "alu", "achieved": ach, "peak": peak, "unit": "Texp/s",
             "frac": ach / peak,
             "peak_note": f"{sms} SMs x {EX2_PER_CLK_SM} ex2/clk/SM (measured "
                          f"ex2.approx.f32 throughput) x {sm_mhz:.0f} MHz max SM clock"}
    r["roof_us"] = {"hbm": t_hbm * 1e6, "ex2": t_ex2 * 1e6, "fp32_2fma": t_fp32 * 1e6}
    r["units_per_launch"] = units
    r["bytes_per_launch"] = nbytes
    return r


# device sources each profiled kernel is compiled from
KERNEL_SOURCES = {
    "scan_channel_2p8b": ("scan_channel.cuh", "ssm_device.cuh"),
    "scan_channel_long": ("scan_channel.cuh", "ssm_device.cuh"),
    "scan_chunk_130m": ("scan_chunk.cuh", "scan_channel.cuh", "ssm_device.cuh"),
    "state_update_decode": ("state_update.cuh", "ssm_device.cuh"),
    "scan_bwd_2p8b": ("scan_bwd.cuh", "ssm_device.cuh"),
    "conv1d_2p8b": ("conv1d.cuh", "ssm_device.cuh"),
}


def source_sha(kernel: str) -> str:
    """Short hash of the device sources of a profiled kernel."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "selective_state_space_115_b300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on the
    current kernel sources (else None)."""
    if kernel not in KERNEL_SOURCES:
        return None
    path = os.path.join(ROOT, "profiles", f"{kernel}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_sha256") != source_sha(kernel):
        return None
    try:
        return float(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id=None, period_ms=50):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", str(period_ms)]
        if gpu_id:
            cmd += ["-i", gpu_id]
        self.lines = []
        self.marks = []
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()
        deadline = time.time() + 5
        while not self.lines and time.time() < deadline:
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        t0, t1 = (self.marks + [0, 0])[:2] if len(self.marks) >= 2 else (0, time.time())
        sm, mx, reasons = [], [], set()
        for ts, line in self.lines:
            if not (t0 <= ts <= t1 + 0.06):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, v in zip(self.NAMES, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# distributed plumbing (timing only; no data-path collective)
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# CPU oracle baseline (bounded sample of the same workload)
# ---------------------------------------------------------------------------
class OracleSample:
    """The oracle on the first `dim` channels of batch row 0 of a workload (inputs
    widened to fp64 once); `run(rows, nthreads)` scans the first `rows` of them and
    returns the seconds it took."""

    def __init__(self, cfg, max_rows: int = 4096):
        import oracle
        self.oracle, self.cfg = oracle, cfg
        self.max_rows = min(cfg.dim, max_rows)
        x = W.make_scan_inputs(cfg, seed=0, batch=1, dim=self.max_rows)
        f = lambda a: None if a is None else W.to_f64(a, cfg.io)  # noqa: E731
        self.u, self.dl, self.z = f(x["u"]), f(x["delta"]), f(x.get("z"))
        self.B, self.C = f(x["B"]), f(x["C"])
        self.A, self.D, self.bias = x["A"], x.get("D"), x.get("delta_bias")

    def run(self, rows: int, nthreads: int) -> float:
        r = slice(0, rows)
        opt = lambda a: None if a is None else a[r]  # noqa: E731
        t = time.perf_counter()
        self.oracle.scan_fwd(self.u[:, r], self.dl[:, r], self.A[r], self.B, self.C,
                             D=opt(self.D), z=None if self.z is None else self.z[:, r],
                             delta_bias=opt(self.bias), nthreads=nthreads)
        return time.perf_counter() - t

    def per_row_seconds(self) -> float:
        k = min(self.max_rows, 4)
        self.run(k, 1)  # warm: library load, page-in
        return self.run(k, 1) / k

    def describe(self, rows: int, threads: int) -> str:
        cfg = self.cfg
        return (f"{rows} of {cfg.batch * cfg.dim} (b,d) rows of the workload (batch row 0), "
                f"full seqlen {cfg.seqlen}, dstate {cfg.dstate}, inputs widened to fp64, fp64 "
                f"sequential loops, {'OpenMP over rows, ' + str(threads) + ' threads' if threads > 1 else 'one thread'}")


def cpu_baseline(cfg, cores: int, target_s: float) -> dict:
    """The oracle as it stands, warmed up, timed on a bounded row sample of `cfg`: all
    host cores (about 2/3 of `target_s`) and one core (the rest).  elements/s =
    rows x seqlen / seconds.  Timed in a fresh process (as the reference arm is), so
    the GPU arm's torch threads and CUDA context do not share the cores."""
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-baseline-only", cfg.name,
           "--cpu-target-s", str(target_s), "--cpu-cores", str(cores)]
    if cfg.batch != W.SCAN_CONFIGS[cfg.name].batch:
        cmd += ["--batch", str(cfg.batch)]
    r = subprocess.run(cmd, capture_output=True, text=True, check=True)
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline_local(cfg, cores: int, target_s: float) -> dict:
    """cpu_baseline's measurement, in this process."""
    smp = OracleSample(cfg)
    per_row = smp.per_row_seconds()
    L = cfg.seqlen

    def timed(rows, threads, budget):
        # repeat the sample until the budget is spent (at least once)
        reps, total = 0, 0.0
        while reps == 0 or total < budget:
            total += smp.run(rows, threads)
            reps += 1
        return reps, total

    rows1 = int(max(1, min(smp.max_rows, target_s / 3 / per_row)))
    reps1, t1 = timed(rows1, 1, target_s / 3)
    rows = int(max(min(cores, smp.max_rows), min(smp.max_rows, target_s * 2 / 3 * cores / per_row)))
    smp.run(rows, cores)  # warm: the thread pool and the output pages
    reps, tn = timed(rows, cores, target_s * 2 / 3)
    return {"value": reps * rows * L / tn, "unit": "elements/s", "cores": cores, "kind": "oracle",
            "sample": f"{reps} x " + smp.describe(rows, cores),
            "single_core": {"value": reps1 * rows1 * L / t1, "unit": "elements/s", "cores": 1,
                            "sample": f"{reps1} x " + smp.describe(rows1, 1)}}


def oracle_sample_rate(target_core_seconds: float, cores: int, steps: int = 1):
    """The reference arm's steps: the oracle on a row sample of the bench workload sized
    to `target_core_seconds` of one core's work, on all cores; returns (elements/s, rows,
    seconds, sample description)."""
    smp = OracleSample(CFG)
    per_row = smp.per_row_seconds()
    rows = int(max(min(cores, smp.max_rows), min(smp.max_rows, target_core_seconds / per_row)))
    smp.run(min(rows, 2 * cores), cores)  # warm the thread pool
    total = sum(smp.run(rows, cores) for _ in range(steps))
    return rows * CFG.seqlen * steps / total, rows, total, smp.describe(rows, cores)


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    cores = os.cpu_count() or 1
    steps, warm = args.steps, args.warmup
    budget = 120.0  # seconds for the whole run
    per_step_core_s = max(0.05, budget * cores / max(1, steps + warm))
    # warm-up steps: tiny calibration runs
    if warm:
        oracle_sample_rate(min(per_step_core_s, 0.5), cores, steps=1)
    rate, rows, secs, desc = oracle_sample_rate(per_step_core_s, cores, steps=steps)
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": "elements/s",
        "n_gpus": args.gpus, "steps": steps, "warmup": warm,
        "ms_per_step": 1e3 * secs / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": bench_config("oracle (fp64 CPU loops) on host cores"),
        "cpu_baseline": {"value": rate, "unit": "elements/s", "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": rate, "unit": "elements/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def bench_config(impl_note: str):
    io = "bf16" if CFG.io == W.BF16 else "fp32"
    names = {"2p8b": "Mamba-2.8B-like", "130m": "Mamba-130M-like", "long": "long-sequence",
             "tiny": "tiny"}
    gate = "silu(z) gate" if CFG.gate else "no gate"
    desc = (f"{names.get(CFG.name, CFG.name)} selective scan: {io} io, fp32 state, batch "
            f"{CFG.batch}, dim {CFG.dim}, dstate {CFG.dstate}, seqlen {CFG.seqlen}, {gate}, "
            f"dt bias = inverse softplus of log-uniform dt, A[d,n] = -(n+1), D ~ N(0,1)")
    mb = scan_bytes(CFG) / 1e6
    if FLUSH_L2:
        l2 = f"L2 flushed before every step (256 MB write, untimed); {mb:.0f} MB per step"
    else:
        l2 = (f"inputs larger than L2 ({mb:.0f} MB per step vs 126 MB L2); no flush"
              if mb > 126 else f"inputs ({mb:.0f} MB) fit in the 126 MB L2: unflushed, L2-warm")
    return {"workload": desc, "batch": CFG.batch, "dim": CFG.dim, "dstate": CFG.dstate,
            "seqlen": CFG.seqlen, "io": io, "impl": impl_note, "l2": l2,
            "parallelism": "one independent problem per GPU (weak scaling)"}


# ---------------------------------------------------------------------------
# main (GPU) arm
# ---------------------------------------------------------------------------
def to_dev_io(a, dev):
    import torch
    if a is None:
        return None
    if CFG.io == W.BF16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(a).to(dev)


def run_gpu(args):
    import torch
    world, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    from selective_state_space_115_b300 import binding as S
    S.library()

    x = W.make_scan_inputs(CFG, seed=rank)
    u, dl, z = to_dev_io(x["u"], dev), to_dev_io(x["delta"], dev), to_dev_io(x["z"], dev)
    B, C = to_dev_io(x["B"], dev), to_dev_io(x["C"], dev)
    A = torch.from_numpy(x["A"]).to(dev)
    Dv = torch.from_numpy(x["D"]).to(dev)
    bias = torch.from_numpy(x["delta_bias"]).to(dev)
    y = torch.empty_like(u)
    stream = torch.cuda.current_stream(dev)

    def step():
        S.scan_fwd(u, dl, A, B, C, D=Dv, z=z, delta_bias=bias, algo=args.algo, out=y)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert S.read_device_status() == 0, "device-side wait timed out during warm-up"

    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:  # noqa: BLE001
        gpu_id = None
    sampler = ClockSampler(gpu_id) if rank == 0 else None
    barrier(world)
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    if sampler:
        sampler.mark()
    t0 = time.perf_counter()
    if args.flush_l2:
        # every step starts from a cold L2: a 256 MB write (twice the L2) before it,
        # outside the step's own pair of events
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for a, b in evs:
            flush.fill_(1)
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize()
        dev_ms = sum(a.elapsed_time(b) for a, b in evs)
    else:
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize()
        dev_ms = ev0.elapsed_time(ev1)
    wall = time.perf_counter() - t0
    if sampler:
        sampler.mark()
    barrier(world)
    clocks = sampler.stop() if sampler else None
    assert S.read_device_status() == 0, "device-side wait timed out in the timed region"
    ms_step = max_over_ranks(dev_ms / args.steps, world, dev)

    plan = S.last_plan()
    elems = CFG.elements
    value = world * elems / (ms_step * 1e-3)
    peaks, peak_kind = measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    sm_mhz = float(peaks.get("sm_max_mhz", SM_MAX_MHZ))
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    bytes_step = scan_bytes(CFG)
    ex2_peak = EX2_PER_CLK_SM * sms * sm_mhz * 1e6 / 1e12   # Texp/s
    roof = scan_roofline(CFG, dev_ms / args.steps, sms, sm_mhz, hbm_peak)
    roof["traffic"] = profiled_traffic({"2p8b": "scan_channel_2p8b",
                                        "long": "scan_channel_long",
                                        "130m": "scan_chunk_130m"}.get(CFG.name, ""))
    roof["kernel"] = plan

    # ---- end to end through the C ABI's host-buffer call (ssm_scan_fwd_host): every
    # step copies its inputs in from pinned host memory and its output back; the
    # library pipelines the batch in pieces (copy-in, scan, copy-out overlap)
    e2e_steps = max(3, min(20, args.steps))
    pin = lambda t: None if t is None else t.cpu().pin_memory()  # noqa: E731
    hu, hd, hz, hB, hC = pin(u), pin(dl), pin(z), pin(B), pin(C)
    hA, hDv, hbias = pin(A), pin(Dv), pin(bias)
    hy = torch.empty(y.shape, dtype=y.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size()
              for t in (hu, hd, hz, hB, hC, hA, hDv, hbias) if t is not None)
    d2h = hy.numel() * hy.element_size()

    def e2e_step():
        S.scan_fwd_host(hu, hd, hA, hB, hC, D=hDv, z=hz, delta_bias=hbias, out=hy,
                        algo=args.algo, device=dev.index)

    e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    torch.cuda.synchronize()
    e2e_s = max_over_ranks((time.perf_counter() - t0) / e2e_steps, world, dev)
    e2e_value = world * elems / e2e_s
    link = link_peak(dev) if rank == 0 else None

    # ---- decode state update (rank 0's measurement)
    decode = run_decode(dev, S) if (rank == 0 and not args.no_decode) else None
    conv = run_conv(dev, S) if (rank == 0 and not args.no_decode) else None
    bwd = run_bwd(dev, S) if (rank == 0 and not args.no_decode) else None
    train = run_train_step(dev, S) if (rank == 0 and not args.no_decode) else None
    euler = None
    if rank == 0 and not args.no_decode:
        # the same scan with the Euler input term (Bbar = dt B)
        def step_euler():
            S.scan_fwd(u, dl, A, B, C, D=Dv, z=z, delta_bias=bias, algo=args.algo, out=y,
                       discretization="euler")
        for _ in range(3):
            step_euler()
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(50):
            step_euler()
        ev1.record(stream)
        torch.cuda.synchronize()
        ms_e = ev0.elapsed_time(ev1) / 50
        euler = {"ms_per_step": ms_e, "value": elems / (ms_e * 1e-3), "unit": "elements/s",
                 "roofline_frac": CFG.updates / (ms_e * 1e-3) / 1e12 / ex2_peak}
    barrier(world)

    # ---- the other scan workloads (rank 0)
    subs = {}
    if rank == 0 and not args.no_sub_configs:
        for name in SUB_CONFIGS:
            if name != CFG.name:
                subs["scan_" + name] = run_scan_config(
                    dev, S, W.SCAN_CONFIGS[name], sms, sm_mhz, hbm_peak,
                    cpu=(world == 1 and not args.no_cpu_baseline))
        torch.cuda.synchronize()

    # ---- CPU baseline (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(CFG, os.cpu_count() or 1, 24.0)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "elements/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": bench_config("libssm scan_channel kernel (TMA, "
                                                        "lanes over channels)"),
            "hbm": {"achieved_gbs": bytes_step / (ms_step * 1e-3) / 1e9, "peak_gbs": hbm_peak,
                    "frac": bytes_step / (ms_step * 1e-3) / 1e9 / hbm_peak,
                    "bytes_per_step": bytes_step, "peak_kind": peak_kind},
            "roofline": roof,
            "e2e": {"value": e2e_value, "unit": "elements/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_s * 1e3,
                    "link": link_fraction(link, h2d, d2h, e2e_s)},
            "gpu_launches": args.steps,
            "clocks": clocks,
            "wall_s_timed": wall,
        }
        if decode:
            line["decode"] = decode
        if conv:
            line["conv1d"] = conv
        if euler:
            line["scan_euler"] = euler
        if bwd:
            line["scan_bwd"] = bwd
        if train:
            line["train_step"] = train
        line.update(subs)
        if cpu:
            line["cpu_baseline"] = cpu
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_scan_config(dev, S, cfg, sms, sm_mhz, hbm_peak, cpu=True) -> dict:
    """One more scan workload through the C ABI (inputs resident on the device): its
    time per scan, elements/s, algorithmic GB/s, roofline against its binding term,
    the plan the library chose, and (cpu) the oracle's rate on a sample of it.
    Workloads that fit in L2 are timed one scan at a time after a 256 MB write (cold
    L2), and also back to back (L2-warm)."""
    import torch
    x = W.make_scan_inputs(cfg, seed=0)
    io = lambda a: None if a is None else to_dev_io_cfg(a, cfg, dev)  # noqa: E731
    f32 = lambda a: None if a is None else torch.from_numpy(a).to(dev)  # noqa: E731
    u, dl, z, B, C = io(x["u"]), io(x["delta"]), io(x.get("z")), io(x["B"]), io(x["C"])
    A, Dv, bias = f32(x["A"]), f32(x.get("D")), f32(x.get("delta_bias"))
    y = torch.empty_like(u)
    stream = torch.cuda.current_stream(dev)

    def step():
        S.scan_fwd(u, dl, A, B, C, D=Dv, z=z, delta_bias=bias, out=y)

    for _ in range(5):
        step()
    torch.cuda.synchronize()
    assert S.read_device_status() == 0
    plan = S.last_plan()
    nbytes = scan_bytes(cfg)
    steps = 20 if cfg.elements > 1e8 else 200
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ms_warm = e0.elapsed_time(e1) / steps
    ms, l2 = ms_warm, f"inputs ({nbytes / 1e6:.0f} MB) larger than L2; back to back"
    if nbytes < L2_BYTES:
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for a, b in evs:
            flush.fill_(1)
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(b) for a, b in evs) / steps
        l2 = (f"inputs ({nbytes / 1e6:.1f} MB) fit in L2: each scan timed alone after a "
              f"256 MB write (cold L2); ms_per_step_l2_warm back to back")
    assert S.read_device_status() == 0
    roof = scan_roofline(cfg, ms, sms, sm_mhz, hbm_peak)
    roof["traffic"] = profiled_traffic({"long": "scan_channel_long",
                                        "130m": "scan_chunk_130m"}.get(cfg.name, ""))
    roof["kernel"] = plan
    rec = {"workload": cfg.description, "batch": cfg.batch, "dim": cfg.dim,
           "dstate": cfg.dstate, "seqlen": cfg.seqlen,
           "io": "bf16" if cfg.io == W.BF16 else "fp32",
           "ms_per_step": ms, "ms_per_step_l2_warm": ms_warm,
           "value": cfg.elements / (ms * 1e-3), "unit": "elements/s",
           "hbm": {"achieved_gbs": nbytes / (ms * 1e-3) / 1e9, "bytes_per_step": nbytes,
                   "frac": nbytes / (ms * 1e-3) / 1e9 / hbm_peak},
           "roofline": roof, "l2": l2, "steps": steps,
           "gpu_launches": steps * (2 if "segmented" in plan else 1)}
    del u, dl, z, B, C, y
    if cpu:
        rec["cpu_baseline"] = cpu_baseline(cfg, os.cpu_count() or 1, 4.0)
    return rec


def to_dev_io_cfg(a, cfg, dev):
    import torch
    if cfg.io == W.BF16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def link_peak(dev, nbytes: int = 512 << 20) -> dict:
    """Pinned host <-> device copy bandwidth: one cudaMemcpyAsync of 512 MB each way,
    best of 5, timed with CUDA events."""
    import torch
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    out = {}
    for name, dst, src in (("h2d", d, h), ("d2h", h, d)):
        best = None
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            dst.copy_(src, non_blocking=True)
            e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        out[name + "_gbs"] = nbytes / (best * 1e-3) / 1e9
    out["bytes"] = nbytes
    return out


def link_fraction(link, h2d: int, d2h: int, e2e_s: float):
    """The host link's floor for one end-to-end step (copy-in and copy-out of its bytes
    at the measured peaks, the two directions overlapped) and the fraction of the step
    that floor is."""
    if not link:
        return None
    floor = max(h2d / (link["h2d_gbs"] * 1e9), d2h / (link["d2h_gbs"] * 1e9))
    return dict(link, floor_ms=floor * 1e3, frac=floor / e2e_s,
                note="floor = the larger of the step's host-to-device and device-to-host "
                     "bytes at the measured pinned-copy peaks (directions overlapped)")


def run_conv(dev, S, iters=50):
    """The causal depthwise conv1d + silu that precedes the scan, on the scan
    workload's x shape (width 4), through the C ABI."""
    import torch
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    shape = (CFG.batch, CFG.dim, CFG.seqlen)
    dt = torch.bfloat16 if CFG.io == W.BF16 else torch.float32
    x = torch.randn(shape, generator=g, device=dev).to(dt)
    w = torch.randn((CFG.dim, 4), generator=g, device=dev) * 0.5
    bias = torch.randn((CFG.dim,), generator=g, device=dev)
    out = torch.empty_like(x)
    for _ in range(3):
        S.conv1d_fwd(x, w, bias, out=out)
    stream = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(iters):
        S.conv1d_fwd(x, w, bias, out=out)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / iters
    nbytes = 2 * x.numel() * x.element_size() + 4 * 5 * CFG.dim
    peaks, kind = measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"workload": f"causal depthwise conv1d + silu, width 4, x {list(shape)} "
                        f"{'bf16' if CFG.io == W.BF16 else 'fp32'}",
            "ms_per_call": ms, "bytes_per_call": nbytes, "gpu_launches": iters,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                         "frac": gbs / hbm_peak,
                         "traffic": profiled_traffic("conv1d_2p8b") if CFG.name == "2p8b"
                         else None, "peak_kind": kind}}


def bwd_bytes(cfg) -> int:
    """Algorithmic HBM bytes of one scan backward: u, delta, dy (and z) read, du,
    ddelta (and dz) written per element; B, C read and dB, dC written per
    position; fp32 A, D, bias read and dA, dD, bias gradient written."""
    s = 2 if cfg.io == W.BF16 else 4
    per_elem = (5 + (2 if cfg.gate else 0)) * s  # u, delta, dy, du, ddelta (+ z, dz)
    per_pos = 4 * s * cfg.dstate
    params = 2 * 4 * (cfg.dim * cfg.dstate + 2 * cfg.dim)
    return cfg.elements * per_elem + cfg.batch * cfg.seqlen * per_pos + params


def bwd_split(cfg) -> bool:
    """Whether the library splits this gradient's sequence into segments (fewer
    than two 32-channel CTAs per SM, and room for two segments of 256 positions)."""
    return (cfg.batch * ((cfg.dim + 31) // 32) < 2 * SM_COUNT) and cfg.seqlen >= 512


def bwd_ckpt_pass_launches(cfg) -> int:
    """Kernels of the gradient's checkpoint pass on the forward's kernels: one for the
    channel kernel (batch * dim >= 8192), two for the segmented plan (a long sequence
    over few channels); none where the gradient kernel forms its checkpoints itself."""
    if cfg.batch * cfg.dim >= 8192:
        return 1
    return 2 if cfg.seqlen >= 8192 else 0


def run_train_step(dev, S, iters=10):
    """A training step of the bench workload through the C ABI: the forward that writes
    the state checkpoints (ssm_scan_fwd_train) and the gradient that reads them
    (ssm_scan_bwd_ckpt), each timed with CUDA events, and their sum."""
    import torch
    x = W.make_scan_inputs(CFG, seed=0)
    gr = W.make_scan_grads(CFG, seed=0)
    u, dl, z = to_dev_io(x["u"], dev), to_dev_io(x["delta"], dev), to_dev_io(x["z"], dev)
    B, C = to_dev_io(x["B"], dev), to_dev_io(x["C"], dev)
    dy = to_dev_io(gr["dy"], dev)
    A = torch.from_numpy(x["A"]).to(dev)
    Dv = torch.from_numpy(x["D"]).to(dev)
    bias = torch.from_numpy(x["delta_bias"]).to(dev)
    ck = torch.empty(S.ckpt_shape(CFG.batch, CFG.dim, CFG.dstate, CFG.seqlen),
                     dtype=torch.float32, device=dev)
    y = torch.empty_like(u)
    stream = torch.cuda.current_stream(dev)

    def fwd():
        S.scan_fwd(u, dl, A, B, C, D=Dv, z=z, delta_bias=bias, out=y, ckpt=ck)

    def bwd():
        return S.scan_bwd(u, dl, A, B, C, dy, D=Dv, z=z, delta_bias=bias, ckpt=ck)

    out = {}
    for name, fn in (("forward_ms", fwd), ("gradient_ms", bwd)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(iters):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        out[name] = e0.elapsed_time(e1) / iters
    ms = out["forward_ms"] + out["gradient_ms"]
    ck_mb = ck.numel() * 4 / 1e6
    return {"workload": f"training step of the {CFG.name} scan: forward writing the state "
                        f"entering every 8 positions ({ck_mb:.0f} MB), gradient from them",
            **out, "ms_per_step": ms, "value": CFG.elements / (ms * 1e-3),
            "unit": "elements/s",
            "gpu_launches": iters * (1 + ((1 if CFG.io == W.BF16 else 0)
                                          + (2 if CFG.io == W.BF16 else 1)
                                          * (2 if bwd_split(CFG) else 1) + 2))}


def run_bwd(dev, S, iters=20):
    """The scan's gradient on the bench workload (dy ~ N(0, 1)), through the C ABI."""
    import torch
    x = W.make_scan_inputs(CFG, seed=0)
    gr = W.make_scan_grads(CFG, seed=0)
    u, dl, z = to_dev_io(x["u"], dev), to_dev_io(x["delta"], dev), to_dev_io(x["z"], dev)
    B, C = to_dev_io(x["B"], dev), to_dev_io(x["C"], dev)
    dy = to_dev_io(gr["dy"], dev)
    A = torch.from_numpy(x["A"]).to(dev)
    Dv = torch.from_numpy(x["D"]).to(dev)
    bias = torch.from_numpy(x["delta_bias"]).to(dev)

    def call():
        return S.scan_bwd(u, dl, A, B, C, dy, D=Dv, z=z, delta_bias=bias)

    for _ in range(3):
        call()
    stream = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(iters):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / iters
    peaks, kind = measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    peaks_mhz = float(peaks.get("sm_max_mhz", SM_MAX_MHZ))
    ex2_peak = (EX2_PER_CLK_SM * torch.cuda.get_device_properties(dev).multi_processor_count
                * peaks_mhz * 1e6 / 1e12)
    texp = CFG.updates / (ms * 1e-3) / 1e12
    nbytes = bwd_bytes(CFG)
    return {"workload": f"gradient of the {CFG.name} scan (du, ddelta, dz, dA, dB, dC, dD, "
                        "ddelta_bias, dh0)",
            "ms_per_call": ms, "value": CFG.elements / (ms * 1e-3), "unit": "elements/s",
            "checkpoints": ("the forward's kernels in a checkpoint-only pass"
                            if bwd_ckpt_pass_launches(CFG) else "the gradient kernel's own "
                            "forward pass"),
            # the checkpoint pass; bf16 ZOH: the classify kernel, then the gradient kernel
            # as two launches (the CTAs on the series coefficients, then those on the fast
            # ones); the segments' first pass when the sequence is split (as many again);
            # the two fixed-order reductions
            "gpu_launches": (bwd_ckpt_pass_launches(CFG) + (1 if CFG.io == W.BF16 else 0)
                             + (2 if CFG.io == W.BF16 else 1) * (2 if bwd_split(CFG) else 1)
                             + 2) * iters,
            "roofline": {"bound": "alu", "achieved": texp, "peak": ex2_peak, "unit": "Texp/s",
                         "frac": texp / ex2_peak,
                         "traffic": profiled_traffic("scan_bwd_2p8b") if CFG.name == "2p8b"
                         else None,
                         "note": "one ex2 per state update, as the forward; the "
                                 "checkpoint pass and the gradient kernel's recompute of each "
                                 "block's states add two more passes of ex2"},
            "hbm": {"bytes_per_call": nbytes, "achieved_gbs": nbytes / (ms * 1e-3) / 1e9,
                    "frac": nbytes / (ms * 1e-3) / 1e9 / hbm_peak, "peak_kind": kind}}


def run_decode(dev, S):
    """1024 sequential single-token updates of the decode workload, h in place."""
    import torch
    cfg = DEC
    g = torch.Generator(device=dev)
    g.manual_seed(1234)
    static = W.make_decode_static(cfg, seed=0)
    h = torch.from_numpy(static["h"]).to(dev)
    A = torch.from_numpy(static["A"]).to(dev)
    Dv = torch.from_numpy(static["D"]).to(dev)
    bias = torch.from_numpy(static["delta_bias"]).to(dev)
    steps = DECODE_STEPS
    bd = (steps, cfg.batch, cfg.dim)
    bn = (steps, cfg.batch, cfg.dstate)
    u = torch.randn(bd, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    dl = torch.randn(bd, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    z = torch.randn(bd, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    B = torch.randn(bn, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    C = torch.randn(bn, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    y = torch.empty(bd, dtype=torch.bfloat16, device=dev)

    def loop():
        for t in range(steps):
            S.state_update(h, u[t], dl[t], A, B[t], C[t], D=Dv, z=z[t], delta_bias=bias, out=y[t])

    loop()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    loop()
    e1.record(stream)
    torch.cuda.synchronize()
    ms_plain = e0.elapsed_time(e1) / steps
    # the same loop captured once in a CUDA graph
    ms_graph = None
    try:
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            loop()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            loop()
        graph.replay()
        torch.cuda.synchronize()
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        ms_graph = e0.elapsed_time(e1) / steps
    except Exception as e:  # noqa: BLE001
        ms_graph = f"graph capture failed: {e}"
    peaks, kind = measured_peaks()
    hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    nb = decode_bytes(cfg)
    best = ms_plain if not isinstance(ms_graph, float) else min(ms_plain, ms_graph)
    return {"workload": f"decode: batch 256, dim 5120, dstate 16, bf16 io, fp32 state, "
                        f"{steps} sequential steps, h in place",
            "ms_per_step_plain": ms_plain, "ms_per_step_graph": ms_graph,
            "bytes_per_step": nb, "gpu_launches": 2 * steps,
            "roofline": {"bound": "hbm", "achieved": nb / (best * 1e-3) / 1e9,
                         "peak": hbm_peak, "unit": "GB/s",
                         "frac": nb / (best * 1e-3) / 1e9 / hbm_peak,
                         "traffic": profiled_traffic("state_update_decode"),
                         "peak_kind": kind,
                         "note": "h (84 MB) fits in L2, so DRAM bytes can be below the "
                                 "algorithmic bytes"}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="libssm", choices=["libssm", "reference"])
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sub-configs", action="store_true",
                    help="skip the 130M-like, long and tiny scan sub-records")
    ap.add_argument("--cpu-baseline-only", default=None, choices=sorted(W.SCAN_CONFIGS),
                    help="time the oracle on a sample of this workload and print its JSON "
                         "(the bench runs this in a fresh process)")
    ap.add_argument("--cpu-target-s", type=float, default=20.0)
    ap.add_argument("--cpu-cores", type=int, default=0)
    ap.add_argument("--algo", default="auto",
                    choices=["auto", "channel", "chunk", "channel_l1", "channel_l2", "channel_l4"],
                    help="scan kernel family (default: the library's own choice)")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the batch of the scan workload (smaller cases for ncu)")
    ap.add_argument("--workload", default="2p8b", choices=sorted(W.SCAN_CONFIGS),
                    help="scan workload (profiling of the other configurations; the bench "
                         "line is quoted on 2p8b)")
    ap.add_argument("--decode-only", action="store_true",
                    help="run only the decode loop and print its JSON (profiling)")
    ap.add_argument("--flush-l2", action="store_true",
                    help="write 256 MB between timed steps (each step timed alone from a cold "
                         "L2; for workloads whose inputs fit in L2)")
    ap.add_argument("--conv-only", action="store_true",
                    help="run only the conv1d timing and print its JSON (profiling)")
    ap.add_argument("--bwd-only", action="store_true",
                    help="run only the scan backward timing and print its JSON (profiling)")
    ap.add_argument("--decode-steps", type=int, default=None,
                    help="decode loop length (default 1024; fewer for ncu)")
    args = ap.parse_args()
    global CFG, DECODE_STEPS, FLUSH_L2
    CFG = W.SCAN_CONFIGS[args.workload]
    FLUSH_L2 = args.flush_l2
    if args.batch:
        CFG = dataclasses.replace(CFG, batch=args.batch)
    if args.decode_steps:
        DECODE_STEPS = args.decode_steps
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.cpu_baseline_only:
        cfg = W.SCAN_CONFIGS[args.cpu_baseline_only]
        if args.batch:
            cfg = dataclasses.replace(cfg, batch=args.batch)
        print(json.dumps(cpu_baseline_local(cfg, args.cpu_cores or (os.cpu_count() or 1),
                                            args.cpu_target_s)), flush=True)
        return 0
    if args.impl == "reference":
        return run_reference(args)
    if args.decode_only:
        import torch
        from selective_state_space_115_b300 import binding as S
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        print(json.dumps(run_decode(dev, S)), flush=True)
        return 0
    if args.conv_only:
        import torch
        from selective_state_space_115_b300 import binding as S
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        print(json.dumps(run_conv(dev, S, iters=max(1, min(args.steps, 50)))), flush=True)
        return 0
    if args.bwd_only:
        import torch
        from selective_state_space_115_b300 import binding as S
        dev = torch.device("cuda", 0)
        torch.cuda.set_device(dev)
        print(json.dumps(run_bwd(dev, S, iters=max(1, min(args.steps, 20)))), flush=True)
        return 0
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
