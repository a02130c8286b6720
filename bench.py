"""Throughput bench of the exact attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--all]

One step = one fa_fwd call over the whole workload (every (b, h) and every
query row: the complete hot path).  Default workload: the causal bf16 d=128
T=4096 point of the single-head sweep at B=64 (the shape the throughput target
is stated on); Q, K, V are seeded N(0,1) synthetic tensors.  Prints ONE JSON
line (rank 0):

  value      TFLOP/s, flops = 4*B*Hq*T^2*d halved when causal, inputs resident
             in HBM, CUDA events on the launching stream, max over ranks
  e2e        the same metric with pinned-host inputs copied in and the
             outputs copied out inside every timed step, through the C ABI's
             host-buffer entry points fa_fwd_host / fa_bwd_host (batch chunks
             pipelined so that the copies overlap the kernels)
  roofline   the kernel against the measured bf16 dense peak (burst figure:
             each launch is timed as a kernel of its own)
  cpu_baseline  the fp64 CPU oracle, as it stands, on a bounded sample of the
             same workload on this host's cores (rank 0, N=1 only)

--pass bwd times the backward instead: one step = one fa_bwd call (row
preparation, the dK/dV kernel and the dQ kernel) for an upstream gradient dO,
O and LSE from one forward call before the timed region; flops = 2.5 x the
forward's (the five T x T x d products S, dP, dV, dK, dQ; the kernels
recompute S and dP a second time, which is not counted).

--impl reference times that oracle alone, as the reference arm, with the same
metric, unit and config.  Under torchrun (N > 1) every rank runs its own
replica of the workload on its own GPU (no collective on the data path):
value = all ranks' flops / the slowest rank's time ("scaling": "weak").
"""

from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s (causal-adjusted) and % of GB300 BF16 dense peak"
METRIC_BWD = ("attention bwd TFLOP/s (2.5x the causal-adjusted forward flops: S, dP, dV, dK, "
              "dQ products) and % of GB300 BF16 dense peak")
BWD_FLOP_FACTOR = 2.5
UNIT = "TFLOP/s"
L2_BYTES = 129e6
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# sources of the profiled forward kernel (device code and launch); an ncu
# summary taken on other sources does not describe it
KERNEL_SOURCES = ["fa_tc.cu", "ptx.cuh", "tc_layout.cuh", "wait.cuh", "row_store.cuh"]


# ---------------------------------------------------------------- helpers
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def init_dist(world: int, use_cuda: bool):
    if world <= 1:
        return None
    import torch.distributed as dist

    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend="nccl" if use_cuda else "gloo")
    return dist


def reduce_max(dist, x: float, device=None) -> float:
    """Max of a float over ranks (identity without a process group)."""
    if dist is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(values_per_rank_flops: float, world: int, max_seconds: float) -> float:
    """Whole-job TFLOP/s: every rank's flops over the slowest rank's time."""
    return values_per_rank_flops * world / max_seconds / 1e12


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


PIPE_RATES_FILE = os.path.join(ROOT, "profiles", "pipe_rates_gb300.md")


def measured_pipe_rates() -> dict:
    """Per-SM, per-clock instruction rates of the special-function and FMA
    pipes, from the committed record of `bench.py --measure-pipe-rates`
    (lines `key = value`); empty if that record is absent."""
    out = {}
    if os.path.exists(PIPE_RATES_FILE):
        with open(PIPE_RATES_FILE) as f:
            for line in f:
                line = line.strip().lstrip("- ")
                if " = " in line:
                    k, v = line.split(" = ", 1)
                    try:
                        out[k.strip()] = float(v.split()[0])
                    except ValueError:
                        pass
    return out


def alu_peaks(peaks: dict, sms: int) -> dict:
    """Peaks of the two non-tensor pipes the forward can be bound by, from the
    measured per-clock rates (`bench.py --measure-pipe-rates`, recorded in
    profiles/pipe_rates_gb300.md) x SMs x the maximum SM clock
    (``sm_max_mhz`` of the measured peaks, else 2070 MHz):
      fp32_tflops: FMAs per clock per SM (the larger of the scalar and
                   paired rates) x 2 flops (the true-fp32 CUDA-core kernel is
                   bound by FFMA); 128 lanes per SM if no record exists;
      exp_per_s:   ex2 instructions per clock per SM -- one exponential per
                   kept (row, key) pair bounds the small-d shapes; 32 per clock
                   (one warp instruction per 4 clocks per SMSP) if no record."""
    hz = float(peaks.get("sm_max_mhz", 2070.0)) * 1e6
    rates = measured_pipe_rates()
    # the FMA pipe's capacity: the larger of the scalar and paired FMA rates
    ffma = max(rates.get("ffma_per_clock_per_sm", 0.0),
               rates.get("ffma2_fma_per_clock_per_sm", 0.0)) or 128.0
    ex2 = rates.get("ex2_per_clock_per_sm", 32.0)
    return {"fp32_tflops": sms * ffma * 2 * hz / 1e12, "exp_per_s": sms * ex2 * hz,
            "source": "measured" if rates else "assumed"}


def measure_pipe_rates(args) -> int:
    """Runs the pipe-rate probe (fa_unit_pipe_rate) on one GPU and prints one
    JSON line: instructions per clock per SM (median over the CTAs, one per
    SM, from clock64 spans) for ex2, scalar FFMA and paired FFMA, and the
    aggregate rate per second from CUDA events."""
    import torch

    import exact_attention_90_gb300 as fa

    fa.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    sink = torch.zeros(512, dtype=torch.float32, device=dev)
    cycles = torch.zeros(sms, dtype=torch.int64, device=dev)
    iters = 1 << 14
    out = {"metric": "pipe rates", "sms": sms, "iters": iters, "threads_per_cta": 512,
           "chains_per_thread": 8}
    names = {0: "ex2", 1: "ffma", 2: "ffma2"}
    for kind, name in names.items():
        instr_per_cta = 512 * (8 if kind < 2 else 4) * iters
        for _ in range(2):  # warm-up
            if fa.fa_unit_pipe_rate(kind, iters, sms, sink, cycles) != 0:
                raise RuntimeError("fa_unit_pipe_rate failed")
        torch.cuda.synchronize(dev)
        per_clk, per_s = [], []
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            if fa.fa_unit_pipe_rate(kind, iters, sms, sink, cycles) != 0:
                raise RuntimeError("fa_unit_pipe_rate failed")
            e1.record()
            torch.cuda.synchronize(dev)
            c = cycles.cpu().tolist()
            per_clk.append(statistics.median(instr_per_cta / x for x in c))
            per_s.append(instr_per_cta * sms / (e0.elapsed_time(e1) / 1e3))
        out[f"{name}_per_clock_per_sm"] = round(statistics.median(per_clk), 2)
        out[f"{name}_per_s"] = float(f"{statistics.median(per_s):.4g}")
    # paired FMA: each instruction is two FMAs
    out["ffma2_fma_per_clock_per_sm"] = round(2 * out["ffma2_per_clock_per_sm"], 2)
    print(json.dumps(out), flush=True)
    return 0


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "exact_attention_90_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload_name: str):
    """DRAM bytes per launch from the committed ncu summary of this workload,
    if it was taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", f"fa_fwd_tc_{workload_name}.md")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if "=" in line and line.strip().startswith("- "):
                k, v = line.strip()[2:].split("=", 1)
                vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_sha256") != kernel_source_hash():
        return None
    try:
        return float(vals["traffic_per_launch_bytes"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi samples (every 200 ms) of SM clock and throttle reasons."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.rows = []
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [x.strip() for x in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self, t0: float, t1: float):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"]}
        inside = [r for t, r in self.rows if t0 - 0.25 <= t <= t1 + 0.25]
        note = None
        if not inside:  # timed region shorter than the sampling period: nearest samples
            inside = [min(self.rows, key=lambda tr: abs(tr[0] - (t0 + t1) / 2))[1]]
            note = "timed region shorter than the 200 ms sampling period: nearest sample"
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in inside:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for name, flag in zip(names, r[5:9]):
                if flag.strip().lower() == "active":
                    reasons.add(name)
        out = {"sm_mhz": statistics.median(sm) if sm else None,
               "sm_max_mhz": max(smax) if smax else None,
               "reasons": sorted(reasons), "samples": len(inside)}
        if note:
            out["note"] = note
        return out


# ---------------------------------------------------------------- oracle timing
def blas_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def time_oracle(w, budget_s: float):
    """Times the fp64 oracle on whole (b, h) heads of the workload, one after
    another, until about budget_s seconds have passed (at least one head).
    Returns (TFLOP/s in the metric's causal-adjusted convention, sample text,
    seconds)."""
    import oracle
    from exact_attention_90_gb300.inputs import make_qkv

    q, k, v = make_qkv(1, 1, 1, w.T, w.d, dtype=w.dtype, seed=w.seed, mult=w.mult)
    heads, t_total = 0, 0.0
    while True:
        t0 = time.perf_counter()
        oracle.attention_ref(q, k, v, w.scale, w.causal)
        t_total += time.perf_counter() - t0
        heads += 1
        if t_total >= budget_s or heads >= w.B * w.Hq:
            break
    per_head = 4.0 * w.T * w.T * w.d / (2 if w.causal else 1)
    value = heads * per_head / t_total / 1e12
    sample = (f"the oracle on one (b, h) head of the workload (T={w.T} d={w.d} {w.dtype} "
              f"{'causal' if w.causal else 'non-causal'}; the workload has {w.B * w.Hq} heads), "
              f"run {heads} time(s): {heads}/{w.B * w.Hq} of the workload's work in "
              f"{t_total:.1f} s")
    return value, sample, t_total


def time_oracle_rows(w, budget_s: float, seed: int):
    """One reference-arm step: the oracle on a random set of query rows of the
    workload, sized to take about budget_s seconds.  Returns (TFLOP/s, rows)."""
    import numpy as np

    import oracle
    from exact_attention_90_gb300.inputs import make_qkv

    q, k, v = make_qkv(1, 1, 1, w.T, w.d, dtype=w.dtype, seed=w.seed, mult=w.mult)
    rng = np.random.default_rng(seed)
    rows_per_s = getattr(time_oracle_rows, "_rate", None)
    if rows_per_s is None:
        t0 = time.perf_counter()
        oracle.attention_rows_ref(q, k, v, w.scale, w.causal, 0, 0, np.arange(64))
        rows_per_s = 64 / max(time.perf_counter() - t0, 1e-6)
        time_oracle_rows._rate = rows_per_s
    n = int(max(16, min(w.T, rows_per_s * budget_s)))
    rows = np.sort(rng.choice(w.T, size=n, replace=False))
    t0 = time.perf_counter()
    oracle.attention_rows_ref(q, k, v, w.scale, w.causal, 0, 0, rows)
    dt = time.perf_counter() - t0
    flops = 4.0 * n * w.T * w.d / (2 if w.causal else 1)  # the rows' share of the head
    return flops / dt / 1e12, n, dt


# ---------------------------------------------------------------- arms
def run_reference(args, w):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    os.environ.setdefault("OMP_NUM_THREADS", str(blas_threads()))
    step_budget = max(0.2, min(3.0, 150.0 / max(1, args.steps + args.warmup)))
    for i in range(args.warmup):
        time_oracle_rows(w, step_budget, seed=i)
    vals, rows_done, secs = [], 0, 0.0
    for i in range(args.steps):
        v, n, dt = time_oracle_rows(w, step_budget, seed=1000 + i)
        vals.append(v)
        rows_done += n
        secs += dt
    value = 4.0 * rows_done * w.T * w.d / (2 if w.causal else 1) / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(),
                         "kind": "oracle",
                         "sample": f"{args.steps} steps x ~{step_budget:.2f} s: random query "
                                   f"rows of one head ({rows_done} rows in all)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def config_of(w, world):
    in_bytes = (w.B * w.Hq + 2 * w.B * w.Hkv) * w.T * w.d * (2 if w.dtype == "bf16" else 4)
    return {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "T": w.T, "d": w.d,
            "dtype": w.dtype, "causal": w.causal, "scale": w.scale,
            "layout": "[B,H,T,d] contiguous",
            "l2": (f"no flush: inputs {in_bytes / 2**20:.0f} MiB > 129 MB L2"
                   if in_bytes > L2_BYTES else "L2 flushed between steps"),
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


def run_ours(args, w):
    import torch

    import exact_attention_90_gb300 as fa
    from exact_attention_90_gb300.inputs import make_grad_out, make_qkv

    rank, local_rank, world = dist_env()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = init_dist(world, True)
    fa.load_library()  # raises if the CUDA library is missing: no fallback

    bwd = args.pass_ == "bwd"
    flops = w.flops * (BWD_FLOP_FACTOR if bwd else 1.0)
    code = {"bf16": fa.FA_DTYPE_BF16, "f16": fa.FA_DTYPE_F16, "f32": fa.FA_DTYPE_F32}[w.dtype]
    qh, kh, vh = make_qkv(w.B, w.Hq, w.Hkv, w.T, w.d, dtype=w.dtype, seed=w.seed, mult=w.mult)
    q, k, v = qh.to(dev), kh.to(dev), vh.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.T), dtype=torch.float32, device=dev)
    in_bytes = sum(x.numel() * x.element_size() for x in (q, k, v))
    stream = torch.cuda.current_stream(dev)
    if bwd:
        doh = make_grad_out(w.B, w.Hq, w.T, w.d, dtype=w.dtype, seed=w.seed)
        do = doh.to(dev)
        fa.fwd(q, k, v, causal=w.causal, scale=w.scale, out=o, lse=lse)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws_bytes = fa.fa_bwd_workspace_size(w.B, w.Hq, w.T)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        in_bytes += 2 * o.numel() * o.element_size()
    flush = None if in_bytes > L2_BYTES else torch.empty(int(256e6), dtype=torch.uint8, device=dev)

    def step():
        if flush is not None:
            flush.zero_()
        if bwd:
            st = fa.fa_bwd(q, k, v, o, lse, do, dq, dk, dv, w.B, w.Hq, w.Hkv, w.T, w.d, w.scale,
                           int(w.causal), -1, -1, code, ws, ws_bytes, stream)
        else:
            st = fa.fa_fwd(q, k, v, o, lse, w.B, w.Hq, w.Hkv, w.T, w.d, w.scale, int(w.causal),
                           code, stream)
        if st != 0:
            raise fa.FaError(st, "fa_bwd" if bwd else "fa_fwd")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if fa.fa_debug_sync_check(stream) != 0:
        raise RuntimeError("kernel barrier wait timed out during warm-up")

    if args.profile:
        for _ in range(args.steps):
            step()
        torch.cuda.synchronize(dev)
        st = fa.fa_debug_sync_check(stream)
        print(json.dumps({"profile": w.name, "steps": args.steps, "status": st}), flush=True)
        return 0 if st == 0 else 1

    sampler = ClockSampler(int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local_rank)).split(",")[0])
                           if os.environ.get("CUDA_VISIBLE_DEVICES", "").isdigit() else local_rank)
    sampler.start()
    time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    if dist is not None:
        dist.barrier()
    time.sleep(0.3)
    sampler.stop()
    ms = e0.elapsed_time(e1)
    ms_max = reduce_max(dist, ms, dev)
    value = aggregate(flops * args.steps, world, ms_max / 1e3)
    if fa.fa_debug_sync_check(stream) != 0:
        raise RuntimeError("kernel barrier wait timed out during the timed region")

    # ---- end to end: pinned host inputs in, outputs out, every step (forward:
    # Q, K, V in, O and LSE out; backward: Q, K, V, O, LSE, dO in, dQ, dK, dV out)
    e2e_steps = max(3, min(args.steps, 50))
    qp, kp, vp = (x.pin_memory() for x in (qh, kh, vh))
    if bwd:
        ins = [(q, qp), (k, kp), (v, vp), (o, o.cpu().pin_memory()),
               (lse, lse.cpu().pin_memory()), (do, doh.pin_memory())]
        outs = [(x, torch.empty(x.shape, dtype=x.dtype).pin_memory()) for x in (dq, dk, dv)]
    else:
        ins = [(q, qp), (k, kp), (v, vp)]
        outs = [(x, torch.empty(x.shape, dtype=x.dtype).pin_memory()) for x in (o, lse)]

    # forward: the C ABI's host-buffer entry point, which pipelines batch
    # chunks so that copies overlap the kernels (about 256 work units per chunk)
    chunks = max(1, min(w.B, w.B * w.Hq * ((w.T + 255) // 256) // 256))
    if args.e2e_chunks > 0:
        chunks = min(w.B, args.e2e_chunks)
    size_fn = fa.fa_bwd_host_workspace_size if bwd else fa.fa_fwd_host_workspace_size
    hws_bytes = size_fn(w.B, w.Hq, w.Hkv, w.T, w.d, code, chunks)
    hws = torch.empty(hws_bytes, dtype=torch.uint8, device=dev)

    def e2e_step():
        if bwd:
            h = [src for _, src in ins]  # q, k, v, o, lse, dO (pinned)
            st = fa.fa_bwd_host(h[0], h[1], h[2], h[3], h[4], h[5], outs[0][1], outs[1][1],
                                outs[2][1], w.B, w.Hq, w.Hkv, w.T, w.d, w.scale, int(w.causal),
                                -1, -1, code, chunks, hws, hws_bytes, stream)
            if st != 0:
                raise fa.FaError(st, "fa_bwd_host")
        else:
            st = fa.fa_fwd_host(qp, kp, vp, outs[0][1], outs[1][1], w.B, w.Hq, w.Hkv, w.T, w.d,
                                w.scale, int(w.causal), code, chunks, hws, hws_bytes, stream)
            if st != 0:
                raise fa.FaError(st, "fa_fwd_host")

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = reduce_max(dist, e0.elapsed_time(e1), dev)
    e2e_value = aggregate(flops * e2e_steps, world, e2e_ms / 1e3)
    h2d = sum(src.numel() * src.element_size() for _, src in ins)
    d2h = sum(dst.numel() * dst.element_size() for _, dst in outs)

    peaks, src = load_peaks()
    ms_per = ms / args.steps
    achieved = flops / (ms_per / 1e3) / 1e12
    # fp16 and bf16 share the dense tensor rate (nominal ratio 1:1); the fp32
    # kernel runs on the CUDA cores, bound by FFMA (alu_peaks)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    alu = alu_peaks(peaks, sms)
    tensor_path = w.dtype in ("bf16", "f16")
    peak = float(peaks["bf16_tflops"]) if tensor_path else alu["fp32_tflops"]
    pairs = w.flops / (4.0 * w.d)  # kept (row, key) pairs: one exponential each
    traffic = None if bwd else ncu_traffic(w.name)
    clocks = sampler.summary(t_wall0, t_wall1)

    line = {
        "metric": METRIC_BWD if bwd else METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic (seeded N(0,1) Q, K, V" + (", dO)" if bwd else ")"),
        "config": config_of(w, world),
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "path": (f"{'fa_bwd_host' if bwd else 'fa_fwd_host'}: pinned host buffers, "
                         f"{chunks} batch chunks pipelined over 2 streams")},
        "gpu_launches": args.steps * (3 if bwd else 1),
        "roofline": {"bound": "tensor" if tensor_path else "alu", "achieved": achieved,
                     "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": (f"bf16_tflops (burst) of {src}" if tensor_path else
                                     f"derived: {sms} SMs x FFMA per clock per SM "
                                     f"({alu['source']}) x 2 flops x "
                                     f"{float(peaks.get('sm_max_mhz', 2070.0)):.0f} MHz"),
                     "exp_peak_source": (f"{sms} SMs x ex2 per clock per SM ({alu['source']}, "
                                         "profiles/pipe_rates_gb300.md) x max SM clock"),
                     "exp_frac": (None if bwd else
                                  pairs / (ms_per / 1e3) / alu["exp_per_s"]),
                     "algorithmic_flops_per_launch": flops,
                     "algorithmic_bytes_per_launch": w.bytes,
                     "hbm_gbs": w.bytes / (ms_per / 1e3) / 1e9,
                     "hbm_frac": w.bytes / (ms_per / 1e3) / 1e9 / float(peaks["hbm_gbs"]),
                     "kernel": (("fa_bwd_prep_kernel + fa_bwd_dkdv_tc_kernel + fa_bwd_dq_tc_kernel "
                                 "(one fa_bwd call)") if bwd else
                                ("fa_fwd_simt_kernel" if w.dtype == "f32" else "fa_fwd_tc_kernel"))},
        "clocks": clocks,
    }
    if bwd:
        line["config"]["pass"] = "backward"
    if world == 1 and rank == 0 and not args.no_cpu_baseline and not bwd:
        os.environ.setdefault("OMP_NUM_THREADS", str(blas_threads()))
        cv, sample, _ = time_oracle(w, args.cpu_budget)
        line["cpu_baseline"] = {"value": cv, "unit": UNIT, "cores": blas_threads(),
                                "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_all(args):
    """One line per workload (for the tables); not the headline contract."""
    import torch

    import exact_attention_90_gb300 as fa
    from exact_attention_90_gb300.inputs import make_grad_out, make_qkv
    from exact_attention_90_gb300.workloads import all_workloads

    fa.load_library()
    peaks, src = load_peaks()
    dev = torch.device("cuda", 0)
    alu = alu_peaks(peaks, torch.cuda.get_device_properties(dev).multi_processor_count)
    flush = torch.empty(int(256e6), dtype=torch.uint8, device=dev)
    bwd = args.pass_ == "bwd"
    for w in all_workloads():
        if args.filter and args.filter not in w.name:
            continue
        q, k, v = (x.to(dev) for x in make_qkv(w.B, w.Hq, w.Hkv, w.T, w.d, dtype=w.dtype,
                                               seed=w.seed, mult=w.mult))
        o, lse = fa.fwd(q, k, v, causal=w.causal, scale=w.scale)
        if bwd:
            do = make_grad_out(w.B, w.Hq, w.T, w.d, dtype=w.dtype, seed=w.seed).to(dev)
            grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))

            def call():
                fa.bwd(q, k, v, o, lse, do, causal=w.causal, scale=w.scale, dq=grads[0],
                       dk=grads[1], dv=grads[2])
        else:
            def call():
                fa.fwd(q, k, v, causal=w.causal, scale=w.scale, out=o, lse=lse)
        call()
        torch.cuda.synchronize()
        times = []
        for _ in range(max(3, args.steps)):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            call()
            e1.record()
            torch.cuda.synchronize()
            times.append(e0.elapsed_time(e1))
        if fa.fa_debug_sync_check() != 0:
            raise RuntimeError(f"{w.name}: kernel barrier wait timed out")
        ms = statistics.median(times)
        flops = w.flops * (BWD_FLOP_FACTOR if bwd else 1.0)
        tf = flops / (ms / 1e3) / 1e12
        gbs = w.bytes / (ms / 1e3) / 1e9
        print(json.dumps({"workload": w.name, "pass": "bwd" if bwd else "fwd", "ms": ms,
                          "tflops": tf, "frac_bf16_peak": tf / float(peaks["bf16_tflops"]),
                          "frac_fp32_alu": (tf / alu["fp32_tflops"]) if w.dtype == "f32" else None,
                          "frac_exp": (None if bwd else
                                       w.flops / (4.0 * w.d) / (ms / 1e3) / alu["exp_per_s"]),
                          "hbm_gbs": gbs, "frac_hbm": gbs / float(peaks["hbm_gbs"]),
                          "peaks": src, "l2": "flushed (256 MB write) before each call"}),
              flush=True)
        del q, k, v, o, lse
    return 0


def main(argv=None):
    from exact_attention_90_gb300.workloads import HEADLINE, by_name

    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "bwd"], default="fwd",
                    help="time the forward (default) or the backward (fa_bwd)")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--all", action="store_true", help="one line per workload shape")
    ap.add_argument("--filter", default="", help="with --all: substring of workload names")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile", action="store_true",
                    help="device steps only (no e2e, oracle or clock sampling): for ncu")
    ap.add_argument("--B", type=int, default=0, help="override the workload's batch size")
    ap.add_argument("--e2e-chunks", type=int, default=0,
                    help="batch chunks of the host-buffer (e2e) leg; 0: the default rule")
    ap.add_argument("--measure-pipe-rates", action="store_true",
                    help="measure the ex2 and FMA instruction rates per clock per SM (the "
                         "denominators of the exp and fp32 rooflines) and exit")
    args = ap.parse_args(argv)
    if args.measure_pipe_rates:
        return measure_pipe_rates(args)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    _, _, world = dist_env()
    if world != args.gpus and world > 1:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    w = by_name(args.workload)
    if args.B:
        w = dataclasses.replace(w, B=args.B, name=f"{w.name}@B{args.B}")
    if args.impl == "reference":
        return run_reference(args, w)
    if args.all:
        return run_all(args)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
