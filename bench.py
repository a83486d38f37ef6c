#!/usr/bin/env python
"""Selective-scan forward throughput on one (or N) B300 GPUs.

One step = one call of the fused selective-scan forward (discretise, scan,
readout, gate) over one batch of seeded synthetic input of the workload: by
default the Mamba-130M-layer shape (batch 8, L 2048, dim 1536, N 16, bf16
inputs and output, fp32 state, softplus + bias, SiLU gate).  Prints ONE JSON
line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--all]

Under torchrun (N > 1) every rank runs its own full-size replica of the
workload on its GPU (weak scaling; the path shards over batch rows with no
exchange), the timed region is bracketed by a barrier and a device
synchronise, and the slowest rank's time is used.

Token = one (batch row, step) pair: tokens per step = batch * L, the tokens/s
convention of the pages' benchmark_inference harness (youngju.dev page).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import ssm_workloads as W  # noqa: E402

METRIC = "selective-scan fwd tokens/s and HBM GB/s as % of B300 peak (D=1536,N=16)"
HBM_FALLBACK_GBS = 6400.0
KERNEL_SRC = os.path.join(ROOT, "selective_state_space_150_b300", "csrc", "ssmscan.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


# ----------------------------------------------------------------- accounting
def algorithmic_bytes(wl: W.Workload) -> int:
    """Bytes one call must move at least: every input element read once, every
    output element written once; the (batch, L, dim, N) state never moves."""
    es = 2 if wl.dtype == "bf16" else 4
    bld = wl.batch * wl.L * wl.dim
    n = bld * es * (2 + (1 if wl.gate else 0))          # u, delta, z
    n += bld * es                                      # y
    n += 2 * wl.batch * wl.L * wl.N * es               # B, C
    n += 4 * wl.batch * wl.dim * wl.N                  # h_last
    n += 4 * wl.dim * wl.N                             # A
    n += 4 * wl.dim * ((1 if wl.skip else 0) + (1 if wl.delta_bias else 0))
    return n


def algorithmic_ops(wl: W.Workload):
    """(MUFU ops, FP32 lane ops) one call needs: per (b, t, d, n) one exp and
    four FP32 ops (dt*A, (dt*u)*B, the state FMA, the readout FMA); per
    (b, t, d) an exp + log for softplus, an exp + reciprocal for the SiLU gate,
    and the bias add, dt*u, D*u and gate multiply."""
    bld = wl.batch * wl.L * wl.dim
    mufu = bld * wl.N + bld * ((2 if wl.softplus else 0) + (2 if wl.gate else 0))
    fp32 = 4 * bld * wl.N + bld * (1 + (1 if wl.delta_bias else 0) + (1 if wl.skip else 0)
                                   + (1 if wl.gate else 0))
    return mufu, fp32


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json, bf16 copy)"
    except Exception:
        return HBM_FALLBACK_GBS, "fallback (6.4 TB/s recipe figure)"


def kernel_hash() -> str:
    with open(KERNEL_SRC, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, only if it was
    taken on the current kernel source."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
        e = d.get(workload)
        if e and e.get("kernel_sha") == kernel_hash():
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """Polls NVML every 10 ms: SM clock, max SM clock, clock-event reasons."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x2: "applications_clocks_setting", 0x1: "gpu_idle"}

    SMI_FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.sw_power_cap,"
                  "clocks_event_reasons.hw_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
                  "clocks_event_reasons.hw_thermal_slowdown")

    def __init__(self, index: int):
        self.index = index
        self.samples, self.reasons, self.ok, self.err = [], set(), False, None
        self.max_mhz = None
        self.source = "NVML, 10 ms polling"
        self._stop = threading.Event()
        self.proc = None
        try:
            import pynvml
            pynvml.nvmlInit()
            self.nv = pynvml
            self.h = pynvml.nvmlDeviceGetHandleByIndex(index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.ok = True
        except Exception as e:  # fall back to polling nvidia-smi
            self.err = f"NVML unavailable ({type(e).__name__}: {e}); used nvidia-smi"
            self.source = "nvidia-smi -lms 50"

    def _run(self):
        while not self._stop.is_set():
            try:
                self.samples.append(self.nv.nvmlDeviceGetClockInfo(self.h, self.nv.NVML_CLOCK_SM))
                bits = self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)
                for b, name in self.REASONS.items():
                    if bits & b:
                        self.reasons.add(name)
            except Exception:
                pass
            time.sleep(0.01)

    def __enter__(self):
        if self.ok:
            self.t = threading.Thread(target=self._run, daemon=True)
            self.t.start()
        else:
            import subprocess
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.SMI_FIELDS,
                     "--format=csv,noheader,nounits", "-lms", "50"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except Exception as e:
                self.err = f"no clock source: {e}"
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self.ok:
            self.t.join()
        elif self.proc is not None:
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            names = ("sw_power_cap", "hw_slowdown", "sw_thermal_slowdown", "hw_thermal_slowdown")
            for line in out.splitlines():
                f = [x.strip() for x in line.split(",")]
                if len(f) < 6:
                    continue
                try:
                    self.samples.append(float(f[0]))
                    self.max_mhz = float(f[1])
                except ValueError:
                    continue
                for name, v in zip(names, f[2:6]):
                    if v.lower() == "active":
                        self.reasons.add(name)

    def summary(self):
        d = {"sm_mhz": (statistics.median(self.samples) if self.samples else None),
             "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons - {"gpu_idle"}),
             "samples": len(self.samples), "source": self.source}
        if self.err:
            d["note"] = self.err
        return d


# ----------------------------------------------------------------- distributed
def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------- cpu side
def oracle_rate(wl: W.Workload, inp, budget_s: float, threads: int, seed: int = 2):
    """Time the fp64 oracle on a bounded sample of the workload: all batch rows
    and all steps of a seeded subset of channels, sized to about budget_s of
    thread-time.  Returns (tokens/s scaled to the full channel count, sample
    description, wall seconds)."""
    import oracle
    rng = np.random.default_rng(seed)
    # calibrate on a tiny piece
    probe_d = np.arange(min(4, wl.dim))
    sub = W.gather(inp, np.arange(1), probe_d)
    t0 = time.perf_counter()
    oracle.selective_scan_fwd(sub["u"], sub["delta"], sub["A"], sub["B"], sub["C"], sub["D"],
                              sub["z"], sub["delta_bias"], sub["softplus"])
    per_btd = (time.perf_counter() - t0) / (wl.L * len(probe_d))
    n_dim = int(budget_s / max(per_btd * wl.batch * wl.L, 1e-12))
    n_dim = max(threads, min(wl.dim, n_dim))
    ds = np.sort(rng.choice(wl.dim, size=n_dim, replace=False))
    sub = W.gather(inp, np.arange(wl.batch), ds)
    t0 = time.perf_counter()
    oracle.selective_scan_fwd_threads(sub["u"], sub["delta"], sub["A"], sub["B"], sub["C"],
                                      sub["D"], sub["z"], sub["delta_bias"], sub["softplus"],
                                      threads=threads)
    wall = time.perf_counter() - t0
    tokens_equiv = wl.batch * wl.L * n_dim / wl.dim
    desc = (f"all {wl.batch} batch rows x {wl.L} steps x {n_dim} of {wl.dim} channels "
            f"(N={wl.N}), fp64 C loop on {threads} host threads; tokens scaled by "
            f"{n_dim}/{wl.dim}")
    return tokens_equiv / wall, desc, wall


def l2_note_for(wl: W.Workload) -> str:
    """How the timed steps keep their working set out of the L2 cache: the GPU
    arm alternates two resident copies of the inputs and outputs."""
    return (f"inputs and outputs rotate over 2 resident copies "
            f"({2 * algorithmic_bytes(wl) / 1e6:.0f} MB > 126 MB L2); no flush")


def config_of(wl: W.Workload, l2_note: str):
    return {"workload": wl.name, "batch": wl.batch, "L": wl.L, "dim": wl.dim, "N": wl.N,
            "io_dtype": wl.dtype, "state_dtype": "f32", "softplus": wl.softplus,
            "delta_bias": wl.delta_bias, "gate": wl.gate, "skip": wl.skip,
            "tokens_per_step": wl.tokens, "l2": l2_note}


# ----------------------------------------------------------------- reference arm
def run_reference(args, wl):
    world, rank = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    threads = os.cpu_count() or 1
    inp = W.make_inputs(wl, seed=0)
    rates = []
    desc = ""
    for i in range(args.warmup + args.steps):
        r, desc, _ = oracle_rate(wl, inp, budget_s=args.ref_step_seconds * threads,
                                 threads=threads, seed=100 + i)
        if i >= args.warmup:
            rates.append(r)
    value = float(np.mean(rates))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * wl.tokens / value, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        # the same workload keys as the GPU arm's line
        "config": config_of(wl, l2_note_for(wl)),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": desc + "; each step a fresh channel sample"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    return line


# ----------------------------------------------------------------- our arm
def run_ours(args, wl, world, rank, local):
    import torch
    import selective_state_space_150_b300 as ssm

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    sptr = stream.cuda_stream
    inp = W.make_inputs(wl, seed=rank)
    bf = wl.dtype == "bf16"
    tdt = torch.bfloat16 if bf else torch.float32

    def host(a, pin=True):
        if a is None:
            return None
        t = (torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16
             else torch.from_numpy(a))
        return t.pin_memory() if pin else t

    hin = {k: host(inp[k]) for k in ("u", "delta", "B", "C", "z", "A", "D", "delta_bias")}

    def device_set():
        return {k: (None if v is None else v.to(dev)) for k, v in hin.items()}

    # Two resident copies of the inputs (and outputs), alternated step by step,
    # so that each step streams a working set larger than the 126 MB L2.
    sets = [device_set(), device_set()]
    outs = [(torch.empty((wl.batch, wl.L, wl.dim), dtype=tdt, device=dev),
             torch.empty((wl.batch, wl.dim, wl.N), dtype=torch.float32, device=dev))
            for _ in range(2)]
    fn = ssm.ssm_scan_fwd_bf16 if bf else ssm.ssm_scan_fwd
    P = lambda t: 0 if t is None else t.data_ptr()  # noqa: E731

    def launch(i):
        s, (y, h) = sets[i & 1], outs[i & 1]
        st = fn(P(s["u"]), P(s["delta"]), P(s["A"]), P(s["B"]), P(s["C"]), P(s["D"]), P(s["z"]),
                P(s["delta_bias"]), int(wl.softplus), P(y), P(h), wl.batch, wl.L, wl.dim, wl.N,
                sptr)
        if st != 0:
            raise RuntimeError(ssm.ssm_status_string(st))

    plan = ssm.ssm_scan_plan(wl.batch, wl.L, wl.dim, wl.N, 1 if bf else 0)
    # a call runs one kernel, or two (segment summaries, then the main pass)
    launches_per_call = 2 if plan["segments"] > 1 else 1
    l2_note = l2_note_for(wl)

    for i in range(args.warmup):
        launch(i)
    torch.cuda.synchronize(dev)

    # pipe peaks for the compute roofline (measured on this GPU, this run)
    peaks = pipe_peaks(sptr)

    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    sampler = ClockSampler(local)
    with sampler:
        # keep the GPU busy for a short untimed window so the clock samples
        # include the steady state, then the timed region
        t_end = time.perf_counter() + args.clock_window
        i = 0
        while time.perf_counter() < t_end:
            launch(i)
            i += 1
            if i % 64 == 0:
                torch.cuda.synchronize(dev)
        torch.cuda.synchronize(dev)
        barrier(world)
        torch.cuda.synchronize(dev)
        for k in range(K):
            starts[k].record(stream)
            launch(k)
            ends[k].record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
    total_ms = starts[0].elapsed_time(ends[-1])
    per_launch_ms = [starts[k].elapsed_time(ends[k]) for k in range(K)]
    total_ms = max_over_ranks(total_ms, world, dev)
    kern_ms = statistics.mean(per_launch_ms)

    value = world * wl.tokens * K / (total_ms * 1e-3)
    bytes_launch = algorithmic_bytes(wl)
    hbm_gbs, hbm_src = measured_peaks()
    achieved_gbs = bytes_launch / (kern_ms * 1e-3) / 1e9
    mufu, fp32 = algorithmic_ops(wl)
    t_hbm = bytes_launch / (hbm_gbs * 1e9)
    roof = None
    if peaks and "ex2_per_s" in peaks:
        t_mufu = mufu / peaks["ex2_per_s"]
        t_fp32 = fp32 / peaks["fma_lane_ops_per_s"]
        t_alu = max(t_mufu, t_fp32)
        if t_alu > t_hbm:
            pipe = "mufu_ex2" if t_mufu >= t_fp32 else "fp32_fma"
            ops = mufu if pipe == "mufu_ex2" else fp32
            peak = peaks["ex2_per_s"] if pipe == "mufu_ex2" else peaks["fma_lane_ops_per_s"]
            roof = {"bound": "alu", "pipe": pipe, "achieved": ops / (kern_ms * 1e-3) / 1e9,
                    "peak": peak / 1e9, "unit": "Gop/s",
                    "frac": (ops / (kern_ms * 1e-3)) / peak,
                    "peak_source": "measured on this GPU by libpipepeaks (8 chains/thread, "
                                   "64 warps/SM), same run"}
    if roof is None:
        roof = {"bound": "hbm", "achieved": achieved_gbs, "peak": hbm_gbs, "unit": "GB/s",
                "frac": achieved_gbs / hbm_gbs, "peak_source": hbm_src}
    roof["traffic"] = recorded_traffic(wl.name)
    roof["algorithmic_bytes_per_launch"] = bytes_launch
    roof["mufu_ops_per_launch"] = mufu
    roof["fp32_ops_per_launch"] = fp32
    roof["kernel_ms"] = kern_ms
    roof["launches_per_call"] = launches_per_call

    # ---- end to end through the C ABI on HOST buffers: every step uploads the
    #      step's inputs from pinned host memory, runs the scan and downloads y
    #      and h_last, inside the library call (parts of the batch overlap their
    #      copies with each other's compute)
    hy = torch.empty((wl.batch, wl.L, wl.dim), dtype=tdt).pin_memory()
    hh = torch.empty((wl.batch, wl.dim, wl.N), dtype=torch.float32).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in hin.values() if v is not None)
    d2h = hy.numel() * hy.element_size() + hh.numel() * hh.element_size()
    Ke = max(3, min(K, args.e2e_steps))
    ws_bytes = ssm.ssm_scan_host_workspace_bytes(wl.batch, wl.L, wl.dim, wl.N, 1 if bf else 0)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    fn_host = ssm.ssm_scan_fwd_bf16_host if bf else ssm.ssm_scan_fwd_host

    def e2e_step():
        st = fn_host(P(hin["u"]), P(hin["delta"]), P(hin["A"]), P(hin["B"]), P(hin["C"]),
                     P(hin["D"]), P(hin["z"]), P(hin["delta_bias"]), int(wl.softplus), P(hy),
                     P(hh), wl.batch, wl.L, wl.dim, wl.N, P(ws), ws_bytes, sptr)
        if st != 0:
            raise RuntimeError(ssm.ssm_status_string(st))

    e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(Ke):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    e2e_value = world * wl.tokens * Ke / (e2e_ms * 1e-3)
    st = ssm.ssm_scan_last_device_status(sptr)
    if st != 0:
        raise RuntimeError("device status: " + ssm.ssm_status_string(st))
    del ws
    link = link_peaks(dev, stream)
    t_h2d = h2d / (link["h2d_gbs"] * 1e9)
    t_d2h = d2h / (link["d2h_gbs"] * 1e9)
    step_ms = e2e_ms / Ke
    link.update({
        # the host-buffer call overlaps uploads, downloads and compute, so the
        # link bound of a step is the slower direction (a full-duplex link);
        # the serial bound adds both directions
        "bound_ms": max(t_h2d, t_d2h) * 1e3, "serial_bound_ms": (t_h2d + t_d2h) * 1e3,
        "e2e_ms_per_step": step_ms, "frac": max(t_h2d, t_d2h) * 1e3 / step_ms})

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": total_ms / K,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic (seeded; see ssm_workloads.py)",
        "config": config_of(wl, l2_note),
        "hbm": {"achieved_gbs": achieved_gbs, "peak_gbs": hbm_gbs, "frac": achieved_gbs / hbm_gbs,
                "peak_source": hbm_src, "roofline_ms": t_hbm * 1e3},
        "roofline": roof,
        "pipe_peaks": peaks,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": Ke, "link": link,
                "path": f"{fn_host.__name__} (C ABI on pinned host buffers: uploads, scan "
                        "and downloads overlapped across parts of the batch)"},
        "gpu_launches": K * launches_per_call,
        "clocks": sampler.summary(),
        "plan": plan,
        "impl": "ours",
    }
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        r, desc, _ = oracle_rate(wl, inp, budget_s=args.cpu_seconds, threads=threads)
        line["cpu_baseline"] = {"value": r, "unit": "tokens/s", "cores": threads,
                                "kind": "oracle", "sample": desc}
    return line


def link_peaks(dev, stream, nbytes: int = 256 << 20, reps: int = 5):
    """The host link's copy rate in each direction, measured alone: one large
    cudaMemcpyAsync between pinned host memory and the device, timed with
    CUDA events after one untimed copy."""
    import torch
    hbuf = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    out = {"bytes_per_copy": nbytes, "copies": reps,
           "how": "pinned host <-> device, one cudaMemcpyAsync per copy, CUDA events"}
    for name, dst, src in (("h2d_gbs", dbuf, hbuf), ("d2h_gbs", hbuf, dbuf)):
        dst.copy_(src, non_blocking=True)
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            dst.copy_(src, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize(dev)
        out[name] = nbytes * reps / (a.elapsed_time(b) * 1e-3) / 1e9
    return out


def pipe_peaks(stream_ptr):
    """MUFU ex2 and FP32 lane-op rates of this GPU, measured now by the
    libpipepeaks microbenchmarks on the given stream."""
    try:
        import ctypes
        lib = ctypes.CDLL(os.path.join(ROOT, "selective_state_space_150_b300", "libpipepeaks.so"))
        out = (ctypes.c_double * 4)()
        if lib.ssm_pipe_peaks(out, ctypes.c_void_p(stream_ptr)) == 0:
            return {"ex2_per_s": out[0], "fma_lane_ops_per_s": out[1],
                    "fma2_lane_ops_per_s": out[2], "sms": int(out[3])}
        return {"error": "ssm_pipe_peaks failed"}
    except Exception as e:  # measurement support missing: report without it
        return {"error": str(e)}


def bwd_accounting(wl: W.Workload, es: int = 4):
    """(bytes, MUFU ops, FP32 lane ops) of one backward call whose tensors are
    es bytes per element.  Bytes: u, delta, z, dy, B, C read once, du, ddelta,
    dz, dB, dC written once, plus A, D, bias and their fp32 gradients.  MUFU
    ops: the recomputation evaluates exp(dt A) three times per (b, t, d, n) --
    the checkpoint pass, the chunk's recomputed states and the adjoint step --
    and per (b, t, d) a softplus (ex2, lg2) in each pass and the gate's
    exponential in the reverse pass.  FP32 lane ops per (b, t, d, n): 3 for
    each of the two forward walks (dt A, (dt u) B, the state FMA), 11 for the
    adjoint step (readout, lambda, dt A, e h_prev, lambda e h_prev, dA, the dt
    term, lambda B, the dB and dC shares, the carry) and 2 for the channel sums
    of the dB and dC shares; per (b, t, d) 8 (bias, dt u twice, skip, du,
    ddelta, dD and dbias sums) and 6 more with the gate."""
    bld, bln = wl.batch * wl.L * wl.dim, wl.batch * wl.L * wl.N
    gate = 1 if wl.gate else 0
    nbytes = es * bld * (2 * (2 + gate) + 1) + es * bln * 4 + 8 * wl.dim * (wl.N + 2)
    mufu = 3 * bld * wl.N + bld * ((4 if wl.softplus else 0) + gate)
    fp32 = 19 * bld * wl.N + bld * (8 + 6 * gate)
    return nbytes, mufu, fp32


def op_cpu_baseline(kind: str, wl: W.Workload, inp, rows: int = 1, n_dim: int = 16,
                    L_s: int = 0, extra=None):
    """The oracle, as it stands, timed single-threaded on a small sample of
    the workload for one of the --op calls: batch rows 0 .. rows-1, n_dim
    seeded channels, the first L_s steps (all when 0).  Returns the
    cpu_baseline object, its value scaled to the full problem in tokens/s."""
    import oracle
    L_s = L_s or wl.L
    ds = np.sort(np.random.default_rng(3).choice(wl.dim, size=min(n_dim, wl.dim), replace=False))
    sub = W.gather(inp, np.arange(rows), ds)
    cut = {k: (v[:, :L_s] if k in ("u", "delta", "B", "C", "z") and v is not None else v)
           for k, v in sub.items()}
    args = (cut["u"], cut["delta"], cut["A"], cut["B"], cut["C"], cut["D"], cut["z"],
            cut["delta_bias"], cut["softplus"])
    t0 = time.perf_counter()
    if kind == "conv_scan":
        w, cb = extra
        oracle.conv_selective_scan_fwd(cut["u"], w[ds], cb[ds], *args[1:])
    elif kind == "zoh_scan":
        oracle.selective_scan_fwd(*args, zoh=True)
    elif kind == "bwd":
        from oracle.backward import selective_scan_bwd as oracle_bwd
        dy = np.random.default_rng(4).standard_normal(cut["u"].shape)
        oracle_bwd(*args, dy)
    wall = time.perf_counter() - t0
    tokens = rows * L_s * len(ds) / wl.dim
    return {"value": tokens / wall, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{rows} batch row(s) x {L_s} steps x {len(ds)} of {wl.dim} channels "
                      f"(N={wl.N}), fp64, one host thread; tokens scaled by {len(ds)}/{wl.dim}"}


def compute_roofline(mufu_ops: int, fp32_ops: int, ms: float, peaks) -> dict:
    """The compute roofline of a call: its MUFU and FP32 lane ops against the
    pipe rates measured in the same run; the slower pipe binds, and the line
    reports its fraction (the other pipe's beside it)."""
    roof = {"bound": "alu", "unit": "Gop/s", "mufu_ops_per_launch": mufu_ops,
            "fp32_ops_per_launch": fp32_ops}
    if "ex2_per_s" not in peaks:
        return roof
    t_mufu = mufu_ops / peaks["ex2_per_s"]
    t_fp32 = fp32_ops / peaks["fma_lane_ops_per_s"]
    pipe = "mufu_ex2" if t_mufu >= t_fp32 else "fp32_fma"
    ops, peak = ((mufu_ops, peaks["ex2_per_s"]) if pipe == "mufu_ex2"
                 else (fp32_ops, peaks["fma_lane_ops_per_s"]))
    roof.update({"pipe": pipe, "achieved": ops / (ms * 1e-3) / 1e9, "peak": peak / 1e9,
                 "frac": ops / (ms * 1e-3) / peak,
                 "mufu_frac": mufu_ops / (ms * 1e-3) / peaks["ex2_per_s"],
                 "fp32_frac": fp32_ops / (ms * 1e-3) / peaks["fma_lane_ops_per_s"],
                 "floor_ms": max(t_mufu, t_fp32) * 1e3,
                 "peak_source": "measured on this GPU by libpipepeaks, same run"})
    return roof


def zoh_ops(wl: W.Workload):
    """(MUFU ops, FP32 lane ops) of the exact zero-order-hold scan: the Euler
    scan's, plus per (b, t, d, n) the factor (e - 1) / A applied to B u: a
    subtraction and two multiplications (no further exponential: e is the
    decay's)."""
    mufu, fp32 = algorithmic_ops(wl)
    return mufu, fp32 + 3 * wl.batch * wl.L * wl.dim * wl.N


def mufu_roofline(mufu_ops: int, ms: float, peaks) -> dict:
    """The compute roofline of a call bound by the MUFU exponentials."""
    roof = {"bound": "alu", "pipe": "mufu_ex2", "unit": "Gop/s", "mufu_ops_per_launch": mufu_ops,
            "achieved": mufu_ops / (ms * 1e-3) / 1e9, "traffic": None}
    if "ex2_per_s" in peaks:
        roof["peak"] = peaks["ex2_per_s"] / 1e9
        roof["frac"] = roof["achieved"] / roof["peak"]
        roof["peak_source"] = "measured on this GPU by libpipepeaks, same run"
    return roof


def _events_mean_ms(fn, reps, stream):
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for i, (a, b) in enumerate(ev):
        a.record(stream)
        fn(i)
        b.record(stream)
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in ev)


def run_op(args, wl):
    """Secondary operations on one workload's shape, one JSON line each:
    conv_scan  the scan with the fused causal conv1d + SiLU prologue, timed
               beside the plain scan on the same inputs;
    zoh_scan   the scan with the exact zero-order-hold B, timed beside the
               Euler scan on the same inputs;
    bwd        the backward pass on the workload's values in fp32, timed
               beside the fp32 forward;
    step       the one-token recurrent step over (batch, dim, N) states,
               timed through a CUDA graph of 100 steps (device time only)."""
    import torch
    import selective_state_space_150_b300 as ssm

    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    inp = W.make_inputs(wl, seed=0)
    bf = wl.dtype == "bf16"

    def dev(a):
        if a is None:
            return None
        t = (torch.from_numpy(a.view(np.int16)).view(torch.bfloat16) if a.dtype == np.uint16
             else torch.from_numpy(a))
        return t.cuda()

    rng = np.random.default_rng(1)
    es = 2 if bf else 4
    hbm_gbs, hbm_src = measured_peaks()
    if args.op == "bwd":
        # the backward pass works on fp32 inputs: the workload's values, widened
        f32 = {k: (None if inp[k] is None else torch.from_numpy(
                   np.ascontiguousarray(W.decode(inp[k]) if inp[k].dtype == np.uint16
                                        else inp[k]).astype(np.float32)).cuda())
               for k in ("u", "delta", "B", "C", "z", "A", "D", "delta_bias")}
        dy = torch.randn((wl.batch, wl.L, wl.dim), device="cuda",
                         generator=torch.Generator(device="cuda").manual_seed(0))

        def bwd_call(i):
            ssm.selective_scan_bwd(f32["u"], f32["delta"], f32["A"], f32["B"], f32["C"], dy,
                                   f32["D"], f32["z"], f32["delta_bias"], wl.softplus)

        # and on the workload's own storage (bf16 tensors through the bf16 entry)
        io = {k: dev(inp[k]) for k in ("u", "delta", "B", "C", "z", "A", "D", "delta_bias")}
        dy_io = dy.to(torch.bfloat16) if bf else dy

        def bwd_io_call(i):
            ssm.selective_scan_bwd(io["u"], io["delta"], io["A"], io["B"], io["C"], dy_io,
                                   io["D"], io["z"], io["delta_bias"], wl.softplus)

        def fwd_call(i):
            ssm.selective_scan_fwd(f32["u"], f32["delta"], f32["A"], f32["B"], f32["C"], f32["D"],
                                   f32["z"], f32["delta_bias"], wl.softplus)

        for i in range(args.warmup):
            bwd_call(i)
            bwd_io_call(i)
            fwd_call(i)
        torch.cuda.synchronize()
        ms_f32 = _events_mean_ms(bwd_call, args.steps, stream)
        ms_io = _events_mean_ms(bwd_io_call, args.steps, stream)
        ms_fwd = _events_mean_ms(fwd_call, args.steps, stream)
        ms_bwd = ms_io
        peaks = pipe_peaks(stream.cuda_stream)
        nbytes, mufu, fp32 = bwd_accounting(wl, es)
        roof = compute_roofline(mufu, fp32, ms_bwd, peaks)
        roof.update({"algorithmic_bytes_per_launch": nbytes, "traffic": None,
                     "hbm_frac": nbytes / (ms_bwd * 1e-3) / 1e9 / hbm_gbs})
        return {
            "op": "bwd", "metric": "selective-scan backward (recomputation) tokens/s",
            "value": wl.tokens / (ms_bwd * 1e-3), "unit": "tokens/s", "higher_is_better": True,
            "ms_per_step": ms_bwd, "steps": args.steps, "warmup": args.warmup,
            "io_dtype": wl.dtype, "fp32_io_ms": ms_f32, "fp32_forward_ms": ms_fwd,
            "roofline": roof, "dtype": "f32",
            "cpu_baseline": None if args.no_cpu_baseline else op_cpu_baseline(
                "bwd", wl, inp, n_dim=8, L_s=256),
            "data": "synthetic (seeded; see ssm_workloads.py); fp32_io_ms: the same values "
                    "widened to fp32",
            "config": config_of(wl, "one resident copy"), "impl": "ours"}
    if args.op == "zoh_scan":
        sets = [{k: dev(inp[k]) for k in ("u", "delta", "B", "C", "z", "A", "D", "delta_bias")}
                for _ in range(2)]
        outs = [(torch.empty_like(s["u"]),
                 torch.empty((wl.batch, wl.dim, wl.N), dtype=torch.float32, device="cuda"))
                for s in sets]

        def call(i, zoh):
            s, (y, h) = sets[i & 1], outs[i & 1]
            ssm.selective_scan_fwd(s["u"], s["delta"], s["A"], s["B"], s["C"], s["D"], s["z"],
                                   s["delta_bias"], wl.softplus, y=y, h_last=h, zoh=zoh)

        for i in range(args.warmup):
            call(i, True)
            call(i, False)
        torch.cuda.synchronize()
        ms_zoh = _events_mean_ms(lambda i: call(i, True), args.steps, stream)
        ms_scan = _events_mean_ms(lambda i: call(i, False), args.steps, stream)
        st = ssm.ssm_scan_last_device_status(stream.cuda_stream)
        if st != 0:
            raise RuntimeError(ssm.ssm_status_string(st))
        return {
            "op": "zoh_scan", "metric": "selective-scan fwd with exact zero-order-hold B tokens/s",
            "value": wl.tokens / (ms_zoh * 1e-3), "unit": "tokens/s", "higher_is_better": True,
            "ms_per_step": ms_zoh, "steps": args.steps, "warmup": args.warmup,
            "euler_scan_ms": ms_scan, "zoh_cost_ms": ms_zoh - ms_scan,
            "zoh_over_euler": ms_zoh / ms_scan,
            "roofline": compute_roofline(*zoh_ops(wl), ms_zoh, pipe_peaks(stream.cuda_stream)),
            "cpu_baseline": None if args.no_cpu_baseline else op_cpu_baseline(
                "zoh_scan", wl, inp, n_dim=256),
            "dtype": "f32", "data": "synthetic (seeded; see ssm_workloads.py)",
            "config": config_of(wl, "inputs rotate over 2 resident copies"), "impl": "ours"}
    if args.op == "conv_scan":
        sets = [{k: dev(inp[k]) for k in ("u", "delta", "B", "C", "z", "A", "D", "delta_bias")}
                for _ in range(2)]
        w = torch.from_numpy((0.5 * rng.standard_normal((wl.dim, 4))).astype(np.float32)).cuda()
        cb = torch.from_numpy((0.1 * rng.standard_normal(wl.dim)).astype(np.float32)).cuda()
        outs = [(torch.empty_like(s["u"]),
                 torch.empty((wl.batch, wl.dim, wl.N), dtype=torch.float32, device="cuda"))
                for s in sets]

        def conv_call(i):
            s, (y, h) = sets[i & 1], outs[i & 1]
            ssm.conv_selective_scan_fwd(s["u"], w, cb, s["delta"], s["A"], s["B"], s["C"], s["D"],
                                        s["z"], s["delta_bias"], wl.softplus, y=y, h_last=h)

        def scan_call(i):
            s, (y, h) = sets[i & 1], outs[i & 1]
            ssm.selective_scan_fwd(s["u"], s["delta"], s["A"], s["B"], s["C"], s["D"], s["z"],
                                   s["delta_bias"], wl.softplus, y=y, h_last=h)

        for i in range(args.warmup):
            conv_call(i)
            scan_call(i)
        torch.cuda.synchronize()
        ms_conv = _events_mean_ms(conv_call, args.steps, stream)
        ms_scan = _events_mean_ms(scan_call, args.steps, stream)
        st = ssm.ssm_scan_last_device_status(stream.cuda_stream)
        if st != 0:
            raise RuntimeError(ssm.ssm_status_string(st))
        bytes_launch = algorithmic_bytes(wl) + wl.dim * 5 * 4
        # a separate conv kernel would read x and write u once more
        unfused_extra = 2 * es * wl.batch * wl.L * wl.dim
        return {
            "op": "conv_scan", "metric": "selective-scan fwd with causal conv1d(k=4)+SiLU "
            "prologue tokens/s", "value": wl.tokens / (ms_conv * 1e-3), "unit": "tokens/s",
            "higher_is_better": True, "ms_per_step": ms_conv, "steps": args.steps,
            "warmup": args.warmup, "plain_scan_ms": ms_scan,
            "prologue_cost_ms": ms_conv - ms_scan,
            "unfused_conv_floor_ms": unfused_extra / (hbm_gbs * 1e9) * 1e3,
            "hbm": {"achieved_gbs": bytes_launch / (ms_conv * 1e-3) / 1e9, "peak_gbs": hbm_gbs,
                    "frac": bytes_launch / (ms_conv * 1e-3) / 1e9 / hbm_gbs,
                    "peak_source": hbm_src},
            # the prologue's SiLU adds an exponential and a reciprocal per (b, t, d)
            "roofline": mufu_roofline(algorithmic_ops(wl)[0] + 2 * wl.batch * wl.L * wl.dim,
                                      ms_conv, pipe_peaks(stream.cuda_stream)),
            "cpu_baseline": None if args.no_cpu_baseline else op_cpu_baseline(
                "conv_scan", wl, inp, n_dim=256, extra=(w.cpu().numpy(), cb.cpu().numpy())),
            "dtype": "f32", "data": "synthetic (seeded; see ssm_workloads.py)",
            "config": config_of(wl, "inputs rotate over 2 resident copies"), "impl": "ours"}
    # one-token step over the workload's (batch, dim, N) states
    tok = {k: (None if inp[k] is None else dev(inp[k][:, 0].copy()) if inp[k].ndim == 3
               else dev(inp[k])) for k in ("u", "delta", "B", "C", "z", "A", "D", "delta_bias")}
    h = torch.zeros((wl.batch, wl.dim, wl.N), dtype=torch.float32, device="cuda")
    y = torch.empty_like(tok["u"])

    def step_call():
        ssm.selective_scan_step(tok["u"], tok["delta"], tok["A"], tok["B"], tok["C"], h,
                                tok["D"], tok["z"], tok["delta_bias"], wl.softplus, y=y)

    for _ in range(args.warmup):
        step_call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(100):
            step_call()
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = max(1, args.steps // 20)
    a.record()
    for _ in range(reps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    us = a.elapsed_time(b) * 1e3 / (reps * 100)
    # the same graph shape around a kernel that does nothing (torch's spin
    # kernel for 0 cycles): the launch and scheduling floor of a graph node
    ge = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ge):
        for _ in range(100):
            torch.cuda._sleep(0)
    ge.replay()
    torch.cuda.synchronize()
    a.record()
    for _ in range(reps):
        ge.replay()
    b.record()
    torch.cuda.synchronize()
    empty_us = a.elapsed_time(b) * 1e3 / (reps * 100)
    state_bytes = wl.batch * wl.dim * wl.N * 8 + wl.dim * wl.N * 4
    cpu = None
    if not args.no_cpu_baseline:
        # the oracle's step over every channel of the workload, one host thread
        import oracle
        x = W.decoded({k: (None if inp[k] is None else inp[k][:, :1]) if k in
                       ("u", "delta", "B", "C", "z") else inp[k] for k in inp})
        t0 = time.perf_counter()
        oracle.selective_scan_step(np.zeros((wl.batch, wl.dim, wl.N)), x["u"][:, 0],
                                   x["delta"][:, 0], x["A"], x["B"][:, 0], x["C"][:, 0], x["D"],
                                   None if x["z"] is None else x["z"][:, 0], x["delta_bias"],
                                   x["softplus"])
        cpu = {"value": (time.perf_counter() - t0) * 1e6, "unit": "us", "cores": 1,
               "kind": "oracle", "sample": f"one step of all {wl.batch} x {wl.dim} channels "
                                           f"(N={wl.N}), fp64, one host thread"}
    return {
        "op": "step", "metric": "one-token recurrent step latency", "value": us, "unit": "us",
        "higher_is_better": False, "tokens_per_s": wl.batch / (us * 1e-6),
        "steps_timed": reps * 100,
        "hbm": {"achieved_gbs": state_bytes / (us * 1e-6) / 1e9, "peak_gbs": hbm_gbs,
                "frac": state_bytes / (us * 1e-6) / 1e9 / hbm_gbs, "peak_source": hbm_src},
        "timing": "CUDA graph of 100 steps, device time per step",
        "empty_kernel_graph_us": empty_us,
        "above_empty_kernel_us": us - empty_us,
        "cpu_baseline": cpu,
        "dtype": "f32", "data": "synthetic (seeded; see ssm_workloads.py)",
        "config": {"workload": wl.name, "batch": wl.batch, "dim": wl.dim, "N": wl.N,
                   "io_dtype": wl.dtype}, "impl": "ours"}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="mamba130m_bf16", choices=sorted(W.WORKLOADS))
    ap.add_argument("--all", action="store_true", help="one line per workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="thread-seconds of oracle work in the cpu_baseline sample")
    ap.add_argument("--ref-step-seconds", type=float, default=1.5,
                    help="wall seconds of oracle work per reference step")
    ap.add_argument("--clock-window", type=float, default=0.5)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--op", choices=["scan", "conv_scan", "zoh_scan", "step", "bwd"],
                    default="scan",
                    help="scan (the headline); conv_scan / zoh_scan / step / bwd: secondary lines")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    names = sorted(W.WORKLOADS) if args.all else [args.workload]
    if args.impl == "reference":
        if int(os.environ.get("RANK", "0")) != 0:
            return 0
        for n in names:
            line = run_reference(args, W.WORKLOADS[n])
            print(json.dumps(line), flush=True)
        return 0

    if args.op != "scan":
        for n in names:
            print(json.dumps(run_op(args, W.WORKLOADS[n])), flush=True)
        return 0

    world, rank, local = dist_init()
    for n in names:
        line = run_ours(args, W.WORKLOADS[n], world, rank, local)
        if rank == 0:
            print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
