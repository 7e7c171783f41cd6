#!/usr/bin/env python
"""Benchmark of the FlashAttention-2 forward pass on GB300.

One step = one forward pass (one kernel launch) over the whole workload:
B=2, H=16, N=4096, D=128, bf16, causal (the N >= 4096, D = 128 workload on
which the tensor-peak target is set).  FLOPs = 4 B H N^2 D / 2 (causal).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME | --shape B,H,N,D[,causal]] [--splits S] [--bwd]

``--bwd`` times the backward pass (fa_bwd: the row statistic and the dK/dV
and dQ kernels) on the same workload instead; its FLOPs are the five
contractions, 2.5x the forward count.

Prints ONE JSON line (rank 0).  Inputs are resident in HBM before the timed
region; they rotate over enough copies that the bytes touched between two
uses of the same copy exceed the 129 MB L2, so every step starts cold.
``e2e`` repeats the measurement through the public call with pinned HOST
buffers, host->device copies of Q, K, V and device->host copies of O, L
inside the timed region.  ``--impl reference`` times the float64 CPU oracle
(the only reference implementation there is) on a bounded sample of rows.

The default run (this workload, one GPU) adds three objects to the line:
``per_config`` times the other benchmark workloads (C1, C2, C4, C5) the same
way, each for at least ``--config-seconds`` of device time so that the clock
sampler (NVML, read every 2 ms; nvidia-smi where NVML does not load) sees
its timed region; ``sustained`` repeats this workload for at least
``--sustained-seconds`` and sets its rate against the sustained bf16 peak,
with the median SM clock and the cycles per step; ``e2e.host_link_gbs`` is
the raw pinned host <-> device copy rate that bounds the end-to-end leg.

Under ``torchrun`` (N > 1) every rank runs its own copy of the workload on
its own GPU (weak scaling, independent problems, no collective on the data
path); the time is the max over ranks.
"""

from __future__ import annotations

import argparse
import dataclasses
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

METRIC = "attention fwd TFLOP/s (bf16, causal & non-causal) and % of GB300 BF16 peak"
UNIT = "TFLOP/s"
L2_BYTES = 129 * 1000 * 1000
FALLBACK_BF16_TFLOPS = 1900.0
# fp32 FFMA (the C1 kernel): 152 SMs x 128 fp32 lanes x 2 flop per FFMA at the
# 2.07 GHz maximum SM clock -- nominal unit counts and clock, not a measurement
FFMA_PEAK_TFLOPS = round(152 * 128 * 2 * 2.07e9 / 1e12, 1)
FFMA_PEAK_SOURCE = "nominal FFMA: 152 SMs x 128 lanes x 2 flop x 2.07 GHz"
E2E_RUNS = 4          # fa_fwd_host runs in the end-to-end measurement of a dense batch
HEADLINE = "B2_H16_N4096_D128_bf16_causal"


# ------------------------------------------------------------ distributed --
def dist_env():
    """(rank, world, local_rank) from torchrun's environment (1 GPU default)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return world > 1


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(x: float, world: int, device="cpu") -> float:
    """Max of a float over ranks (the slowest rank sets the job time)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed(base_seed: int, rank: int) -> int:
    """Each rank draws its own independent problem of the same shape."""
    return base_seed + 1000 * rank


# ------------------------------------------------------------------ peaks --
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, 6800.0, "fallback"


def load_traffic(kernel_tag: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if the sources of
    that kernel family have not changed since it was taken (else None)."""
    from exact_attention_24_gb300.build import kernel_digest
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    e = rec.get(f"{kernel_tag}/{workload}")
    if not e or e.get("source_digest") != kernel_digest(kernel_tag):
        return None
    return e.get("dram_bytes_per_launch")


_NCU_BYTE_UNITS = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "Tbyte": 1e12}


def record_traffic(csv_path: str, kernel_tag: str, workload: str, captured_with: str) -> dict:
    """Sum dram__bytes_read.sum / dram__bytes_write.sum over every launch in
    an `ncu --csv` capture (one forward launch, or the launches of one
    backward step) and store them in profiles/traffic.json under the current
    digest of that kernel family's sources, which `load_traffic` checks."""
    import csv
    from exact_attention_24_gb300.build import kernel_digest
    with open(csv_path) as f:
        lines = [ln for ln in f if ln.startswith('"')]
    rd = wr = 0.0
    launches = set()
    for row in csv.DictReader(lines):
        name, unit = row["Metric Name"], row["Metric Unit"]
        if name not in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
            continue
        if unit not in _NCU_BYTE_UNITS:
            raise ValueError(f"unexpected unit {unit!r} for {name}")
        v = float(row["Metric Value"].replace(",", "")) * _NCU_BYTE_UNITS[unit]
        launches.add(row["ID"])
        if name == "dram__bytes_read.sum":
            rd += v
        else:
            wr += v
    if not launches:
        raise ValueError(f"no DRAM byte metrics in {csv_path}")
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        rec = {}
    entry = {"source_digest": kernel_digest(kernel_tag), "dram_bytes_per_launch": int(round(rd + wr)),
             "dram_bytes_read": int(round(rd)), "dram_bytes_write": int(round(wr)),
             "launches_summed": len(launches), "captured_with": captured_with,
             "note": "1-pass metrics; ncu flushes the caches before each launch; O lines still "
                     "dirty in L2 at kernel end are not counted as DRAM writes"}
    rec[f"{kernel_tag}/{workload}"] = entry
    with open(path, "w") as f:
        json.dump(dict(sorted(rec.items())), f, indent=1)
        f.write("\n")
    return entry


# ----------------------------------------------------------------- clocks --
class ClockSampler:
    """nvidia-smi clocks/throttle sampling in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.idx = gpu_id
        self.lines = []
        self.proc = None
        self.marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.lines and time.time() - t0 < 5:
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        """Median SM clock and the throttle reasons seen in the timed region
        (between the two marks); all samples if none fell inside it."""
        if not self.lines:
            return None
        if len(self.marks) >= 2:
            t0, t1 = self.marks[0], self.marks[-1] + 0.15
            rows = [l for (t, l) in self.lines if t0 <= t <= t1]
        else:
            rows = []
        in_region = bool(rows)
        rows = rows or [l for _, l in self.lines]
        sm, smax, reasons = [], [], set()
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm),
                "in_timed_region": in_region}


class NvmlSampler:
    """SM clock and clock-event reasons read from NVML (libnvidia-ml, through
    ctypes) every few milliseconds in a background thread, so that even a
    timed region of a few milliseconds holds samples.  Reads only; sets
    nothing.  ``ok`` is False where NVML cannot be loaded (then the
    nvidia-smi sampler above is used)."""

    # clock-event reason bits of nvmlDeviceGetCurrentClocksEventReasons
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_id: str, period_s: float = 0.002):
        import ctypes
        self.period = period_s
        self.samples = []          # (time, sm_mhz, reason mask)
        self.marks = []
        self.ok = False
        self._stop = threading.Event()
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            if gpu_id.isdigit():
                r = lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(int(gpu_id)), ctypes.byref(h))
            else:
                r = lib.nvmlDeviceGetHandleByUUID(gpu_id.encode(), ctypes.byref(h))
            if r != 0:
                return
            self.reason_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint()
            lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx))   # 1 = NVML_CLOCK_SM
            self.max_mhz = float(mx.value)
            self.lib, self.h, self.ctypes = lib, h, ctypes
            self.ok = True
        except (OSError, AttributeError):
            self.ok = False

    def _read(self):
        ct = self.ctypes
        mhz, mask = ct.c_uint(), ct.c_ulonglong()
        while not self._stop.is_set():
            if (self.lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(mhz)) == 0 and
                    self.reason_fn(self.h, ct.byref(mask)) == 0):
                self.samples.append((time.time(), float(mhz.value), int(mask.value)))
            time.sleep(self.period)

    def start(self):
        if self.ok:
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            t0 = time.time()
            while not self.samples and time.time() - t0 < 2:
                time.sleep(0.001)

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        self._stop.set()
        if self.ok:
            self.thread.join(timeout=2)

    def summary(self, region=None):
        """Median SM clock and the reasons seen between two marks (``region``
        = their indices, default the first and last); all samples if none
        fell inside."""
        if not self.samples:
            return None
        rows = []
        if len(self.marks) >= 2:
            a, b = region or (0, len(self.marks) - 1)
            t0, t1 = self.marks[a], self.marks[b]
            rows = [x for x in self.samples if t0 <= x[0] <= t1]
        in_region = bool(rows)
        rows = rows or self.samples
        reasons = set()
        for _, _, m in rows:
            for bit, name in self.REASONS.items():
                if m & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[1] for r in rows), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(rows), "in_timed_region": in_region,
                "source": "nvml"}


def make_sampler(gpu_id: str):
    """The NVML sampler where NVML loads, else nvidia-smi."""
    s = NvmlSampler(gpu_id)
    return s if s.ok else ClockSampler(gpu_id)


def smi_gpu_id(local: int) -> str:
    """nvidia-smi --id for CUDA device `local` (honours CUDA_VISIBLE_DEVICES)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        if local < len(ids):
            return ids[local]
    return str(local)


# ------------------------------------------------------------- our arm --
class FwdRunner:
    """A workload's inputs resident on the device, rotated over enough copies
    that the bytes touched between two uses of one copy exceed twice the L2
    (every launch starts with a cold L2), and the library call that runs one
    step (one forward pass over the whole workload) on ``stream``."""

    def __init__(self, fa, w, dev, stream, seed, splits=None):
        import torch
        from exact_attention_24_gb300.workloads import make_inputs
        self.fa, self.w, self.dev, self.stream, self.splits = fa, w, dev, stream, splits
        q, k, v = make_inputs(dataclasses.replace(w, seed=seed))
        self.host = (q, k, v)
        self.f32 = w.dtype == "f32"                 # C1: fp32 in and out, the FFMA kernel
        self.code = fa.FA_F32 if self.f32 else fa.FA_BF16
        self.o_dtype = torch.float32 if self.f32 else torch.bfloat16
        self.o_size = 4 if self.f32 else 2
        self.in_bytes = 3 * q.numel() * q.element_size()
        self.out_bytes = q.numel() * self.o_size + q.numel() // w.D * 4
        self.copies = max(2, math.ceil(2 * L2_BYTES / (self.in_bytes + self.out_bytes)) + 1)
        self.l_shape = (w.H, w.total) if w.varlen else q.shape[:-1]
        self.bufs = []
        with torch.cuda.stream(stream):
            self.cu = torch.as_tensor(w.cu_seqlens, dtype=torch.int32).to(dev) if w.varlen else None
            for _ in range(self.copies):
                self.bufs.append((q.to(dev), k.to(dev), v.to(dev),
                                  torch.empty(q.shape, dtype=self.o_dtype, device=dev),
                                  torch.empty(self.l_shape, dtype=torch.float32, device=dev)))
        self.ws, self.ws_bytes = None, 0
        if splits is not None:
            self.ws_bytes = fa.fa_fwd_splitkv_workspace_size(w.B, w.H, w.N, w.D, splits)
            self.ws = torch.empty(max(self.ws_bytes, 16), dtype=torch.uint8, device=dev)
        torch.cuda.synchronize(dev)

    @property
    def launches_per_step(self) -> int:
        return 2 if self.splits not in (None, 1) and self.ws_bytes else 1

    @property
    def l2_note(self) -> str:
        return (f"inputs rotated over {self.copies} resident copies "
                f"({self.copies * (self.in_bytes + self.out_bytes) / 1e6:.0f} MB > 129 MB L2)")

    def call(self, qd, kd, vd, O, L):
        fa, w, stream, code = self.fa, self.w, self.stream, self.code
        if self.splits is not None:
            st = fa.fa_fwd_splitkv(qd, kd, vd, O, L, w.B, w.H, w.N, w.D, w.scale, int(w.causal),
                                   code, self.splits, self.ws, self.ws_bytes, stream)
        elif w.window:
            st = fa.fa_fwd_window(qd, kd, vd, O, L, w.B, w.H, w.N, w.D, w.scale, w.window[0],
                                  w.window[1], code, stream)
        elif w.varlen:
            st = fa.fa_fwd_varlen(qd, kd, vd, O, L, self.cu, len(w.lengths), w.total, w.max_seqlen,
                                  w.H, w.D, w.scale, int(w.causal), code, stream)
        else:
            st = fa.fa_fwd(qd, kd, vd, O, L, w.B, w.H, w.N, w.D, w.scale, int(w.causal),
                           code, stream)
        if st != fa.FA_OK:
            raise fa.FaError(st, "fa_fwd")

    def launch(self, i):
        self.call(*self.bufs[i % self.copies])

    def check(self, what):
        st = self.fa.fa_check_device_error(self.stream)
        if st != self.fa.FA_OK:
            raise self.fa.FaError(st, what)

    def timed(self, steps, sampler=None, world=1):
        """Device time (ms) of `steps` launches between two CUDA events on
        the launching stream, with a barrier and a synchronize on both sides;
        the sampler's marks bracket the region."""
        import torch
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize(self.dev)
        if sampler:
            sampler.mark()
        ev0.record(self.stream)
        for i in range(steps):
            self.launch(i)
        ev1.record(self.stream)
        torch.cuda.synchronize(self.dev)
        if sampler:
            sampler.mark()
        barrier(world)
        return ev0.elapsed_time(ev1)


def roofline_for(w, t_launch: float, o_size: int) -> dict:
    """The roofline of one launch of `w` that took `t_launch` seconds: the
    FFMA ALU rate for float32 (nominal), HBM for a step whose algorithmic
    bytes take longer at the measured copy rate than its FLOPs at the bf16
    peak, the tensor peak otherwise."""
    peak, hbm_peak, peak_kind = load_peaks()
    flops = w.flops()
    achieved = flops / t_launch / 1e12
    min_bytes = w.min_bytes(o_size)
    if w.dtype == "f32":
        return {"bound": "alu", "achieved": round(achieved, 4), "peak": FFMA_PEAK_TFLOPS,
                "unit": "TFLOP/s", "frac": round(achieved / FFMA_PEAK_TFLOPS, 5),
                "peak_source": FFMA_PEAK_SOURCE}
    if min_bytes / (hbm_peak * 1e9) > flops / (peak * 1e12):
        return {"bound": "hbm", "achieved": round(min_bytes / t_launch / 1e9, 1),
                "peak": hbm_peak, "unit": "GB/s",
                "frac": round(min_bytes / t_launch / 1e9 / hbm_peak, 4),
                "peak_source": f"hbm_gbs of {peak_kind}"}
    return {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4), "peak_source": f"bf16_tflops (burst) of {peak_kind}"}


def bench_ours(args, w, rank, world, local):
    import torch
    import exact_attention_24_gb300 as fa
    from exact_attention_24_gb300.build import build

    build()
    fa.load_library()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    run = FwdRunner(fa, w, dev, stream, rank_seed(w.seed, rank), args.splits)
    q, k, v = run.host
    f32, code, o_dtype, o_size = run.f32, run.code, run.o_dtype, run.o_size

    for i in range(args.warmup):
        run.launch(i)
    run.check("warm-up")

    sampler = make_sampler(smi_gpu_id(local))
    sampler.start()
    ms_local = run.timed(args.steps, sampler, world)
    sampler.stop()
    run.check("timed region")
    ms = reduce_max(ms_local, world, device=dev)
    per_step_ms = ms / args.steps
    flops = w.flops()
    value = world * flops * args.steps / (ms * 1e-3) / 1e12

    # ----------------------------------------------------------- e2e
    e2e_steps = max(3, min(args.steps, 30))
    qh = q.pin_memory()
    kh = k.pin_memory()
    vh = v.pin_memory()
    oh = torch.empty(q.shape, dtype=o_dtype).pin_memory()
    lh = torch.empty(run.l_shape, dtype=torch.float32).pin_memory()
    qd, kd, vd, O, L = run.bufs[0]

    # A dense batch goes through fa_fwd_host: the public call for host
    # tensors, which overlaps the copies with the kernels run by run.  Other
    # workloads copy in, call, copy out on the one stream.
    host_api = not (w.varlen or w.window or args.splits is not None)

    def e2e_step():
        if host_api:
            st = fa.fa_fwd_host(qh, kh, vh, oh, lh, qd, kd, vd, O, L, w.B, w.H, w.N, w.D, w.scale,
                                int(w.causal), code, args.e2e_runs, stream)
            if st != fa.FA_OK:
                raise fa.FaError(st, "fa_fwd_host")
            return
        with torch.cuda.stream(stream):
            qd.copy_(qh, non_blocking=True)
            kd.copy_(kh, non_blocking=True)
            vd.copy_(vh, non_blocking=True)
            run.call(qd, kd, vd, O, L)
            oh.copy_(O, non_blocking=True)
            lh.copy_(L, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = reduce_max(e0.elapsed_time(e1), world, device=dev)
    barrier(world)
    e2e_value = world * flops * e2e_steps / (e2e_ms * 1e-3) / 1e12

    min_bytes = w.min_bytes(o_size)
    t_launch = ms_local / args.steps * 1e-3
    roofline = roofline_for(w, t_launch, o_size)
    roofline["traffic"] = load_traffic("fa_simt" if f32 else "fa_tc", w.name)
    rec = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(per_step_ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32" if f32 else "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "D": w.D,
                   "causal": w.causal, "window": list(w.window) or None,
                   "out_dtype": "f32" if f32 else "bf16", "seed": w.seed,
                   "lengths": list(w.lengths) if w.varlen else None,
                   "splits": args.splits,
                   "flops_per_step": flops,
                   "l2": run.l2_note,
                   "parallelism": f"replicas{world}" if world > 1 else "single-gpu"},
        "roofline": roofline,
        "io": {"min_bytes": min_bytes,
               "achieved_hbm_gbs": round(min_bytes / t_launch / 1e9, 1),
               "tile_model_bytes": io_model_bytes(w, 256, 128),
               "tile_model_bytes_64x64": io_model_bytes(w, 64, 64)},
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT,
                "h2d_bytes_per_step": run.in_bytes,
                "d2h_bytes_per_step": oh.numel() * o_size + lh.numel() * 4,
                "steps": e2e_steps,
                "call": f"fa_fwd_host, {args.e2e_runs} runs" if host_api else "copies, then the call"},
        "gpu_launches": args.steps * run.launches_per_step,
        "clocks": sampler.summary(),
    }
    # the default run (the headline workload on one GPU) also measures the
    # other workloads, a seconds-long run of the headline, and the host link
    if world == 1 and args.extras and w.name == HEADLINE and args.splits is None:
        rec["e2e"]["host_link_gbs"] = host_link_rate(dev, stream)
        del run
        torch.cuda.empty_cache()
        rec["per_config"] = per_config(fa, dev, stream, local, args)
        rec["sustained"] = sustained(fa, w, dev, stream, local, args)
    return rec


def host_link_rate(dev, stream, nbytes: int = 256 << 20, reps: int = 5) -> dict:
    """Raw pinned host <-> device copy rate on this machine (one 256 MiB copy at a
    time, best of `reps`), the bound of the end-to-end leg's copies."""
    import torch
    h = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    out = {}
    for name, dst, src in (("h2d", d, h), ("d2h", h, d)):
        best = None
        for _ in range(reps + 1):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                e0.record(stream)
                dst.copy_(src, non_blocking=True)
                e1.record(stream)
            torch.cuda.synchronize(dev)
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        out[name] = round(nbytes / (best * 1e-3) / 1e9, 1)
    out["bytes_per_copy"] = nbytes
    return out


def _timed_record(run, w, local, min_seconds: float, warmup: int) -> dict:
    """Time `w` for at least `min_seconds` of device time (the step count is
    sized from a short trial) with the clock sampler running, and return its
    value, roofline and clocks."""
    for i in range(warmup):
        run.launch(i)
    run.check("warm-up")
    trial = run.timed(20)
    steps = max(20, int(math.ceil(min_seconds / (trial / 20 * 1e-3))))
    sampler = make_sampler(smi_gpu_id(local))
    sampler.start()
    ms = run.timed(steps, sampler)
    sampler.stop()
    run.check("timed region")
    t_launch = ms / steps * 1e-3
    roof = roofline_for(w, t_launch, run.o_size)
    roof["traffic"] = load_traffic("fa_simt" if run.f32 else "fa_tc", w.name)
    return {"value": round(w.flops() / t_launch / 1e12, 3), "unit": UNIT,
            "ms_per_step": round(ms / steps, 5), "steps": steps,
            "achieved_hbm_gbs": round(w.min_bytes(run.o_size) / t_launch / 1e9, 1),
            "roofline": roof, "l2": run.l2_note,
            "gpu_launches": steps * run.launches_per_step, "clocks": sampler.summary()}


def per_config(fa, dev, stream, local, args) -> dict:
    """The other benchmark workloads (C1, C2, C4, C5), each timed the way the
    headline is, for at least `--config-seconds` of device time so that the
    clock sampler sees the timed region."""
    import torch
    from exact_attention_24_gb300.workloads import C1, C2, C4, C5
    out = {}
    for w in (C1, C2, C4, C5):
        run = FwdRunner(fa, w, dev, stream, w.seed)
        rec = _timed_record(run, w, local, args.config_seconds, args.warmup)
        rec["config"] = {"B": w.B, "H": w.H, "N": w.N, "D": w.D, "causal": w.causal,
                         "dtype": w.dtype, "seed": w.seed,
                         "lengths": list(w.lengths) if w.varlen else None}
        out[w.name] = rec
        del run
        torch.cuda.empty_cache()
    return out


def sustained(fa, w, dev, stream, local, args) -> dict:
    """The headline workload repeated for at least `--sustained-seconds` of
    timed device time: its rate once clocks have settled under load, against
    the sustained bf16 peak, with the clock seen and time x clock (the cycles
    a step takes), so that clock dependence shows."""
    import torch
    run = FwdRunner(fa, w, dev, stream, w.seed)
    rec = _timed_record(run, w, local, args.sustained_seconds, args.warmup)
    del run
    torch.cuda.empty_cache()
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            sus_peak, kind = float(json.load(f)["bf16_tflops_sustained"]), "measured"
    except (OSError, KeyError, ValueError):
        sus_peak, kind = 1700.0, "fallback"
    mhz = (rec["clocks"] or {}).get("sm_mhz")
    rec["frac_of_sustained_peak"] = round(rec["value"] / sus_peak, 4)
    rec["sustained_peak"] = {"value": sus_peak, "unit": UNIT,
                             "source": f"bf16_tflops_sustained of {kind}"}
    if mhz:
        rec["mcycles_per_step"] = round(rec["ms_per_step"] * mhz / 1e3, 4)
        rec["tflops_per_ghz"] = round(rec["value"] / (mhz / 1e3), 2)
    rec["workload"] = w.name
    return rec


# -------------------------------------------------------------- backward --
METRIC_BWD = "attention bwd TFLOP/s (bf16, five-matmul count) and % of GB300 BF16 peak"


def bwd_flops(w) -> float:
    """The five contractions S, dP, dV, dK, dQ at 2 n^2 d each (halved
    under the causal mask): 2.5x the forward count.  The recomputation of S
    and dP that the two-kernel split repeats is not counted."""
    return 2.5 * w.flops()


def bench_bwd(args, w, rank, world, local):
    import torch
    import exact_attention_24_gb300 as fa
    from exact_attention_24_gb300.build import build
    from exact_attention_24_gb300.workloads import make_inputs

    build()
    fa.load_library()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    wr = dataclasses.replace(w, seed=rank_seed(w.seed, rank))
    q, k, v = make_inputs(wr)
    do = make_inputs(dataclasses.replace(wr, seed=wr.seed + 50_000))[0]
    code = fa.FA_BF16
    shape = q.shape
    tensor_b = q.numel() * 2
    l_b = q.numel() // w.D * 4
    per_copy = 5 * tensor_b + l_b + 3 * tensor_b
    copies = max(2, math.ceil(2 * L2_BYTES / per_copy) + 1)
    ws_bytes = (fa.fa_bwd_varlen_workspace_size(w.total, w.H) if w.varlen
                else fa.fa_bwd_workspace_size(w.B, w.H, w.N))
    with torch.cuda.stream(stream):
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
        cu = torch.as_tensor(w.cu_seqlens, dtype=torch.int32).to(dev) if w.varlen else None
        bufs = []
        for _ in range(copies):
            qd, kd, vd, dod = q.to(dev), k.to(dev), v.to(dev), do.to(dev)
            if w.varlen:
                O, L = fa.attention_varlen(qd, kd, vd, cu, w.max_seqlen, causal=w.causal, scale=w.scale,
                                           stream=stream)
            elif w.window:
                O = torch.empty(shape, dtype=torch.bfloat16, device=dev)
                L = torch.empty(shape[:-1], dtype=torch.float32, device=dev)
                st = fa.fa_fwd_window(qd, kd, vd, O, L, w.B, w.H, w.N, w.D, w.scale, w.window[0],
                                      w.window[1], code, stream)
                if st != fa.FA_OK:
                    raise fa.FaError(st, "fa_fwd_window")
            else:
                O, L = fa.attention(qd, kd, vd, causal=w.causal, scale=w.scale, stream=stream)
            grads = [torch.empty(shape, dtype=torch.bfloat16, device=dev) for _ in range(3)]
            bufs.append((qd, kd, vd, O, dod, L, *grads))
    torch.cuda.synchronize(dev)

    def call(b):
        if w.varlen:
            st = fa.fa_bwd_varlen(*b, cu, len(w.lengths), w.total, w.max_seqlen, w.H, w.D, w.scale,
                                  int(w.causal), code, ws, ws_bytes, stream)
        elif w.window:
            st = fa.fa_bwd_window(*b, w.B, w.H, w.N, w.D, w.scale, w.window[0], w.window[1], code, ws,
                                  ws_bytes, stream)
        else:
            st = fa.fa_bwd(*b, w.B, w.H, w.N, w.D, w.scale, int(w.causal), code, ws, ws_bytes, stream)
        if st != fa.FA_OK:
            raise fa.FaError(st, "fa_bwd")

    for i in range(args.warmup):
        call(bufs[i % copies])
    st = fa.fa_check_device_error(stream)
    if st != fa.FA_OK:
        raise fa.FaError(st, "warm-up")
    sampler = make_sampler(smi_gpu_id(local))
    sampler.start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    sampler.mark()
    ev0.record(stream)
    for i in range(args.steps):
        call(bufs[i % copies])
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    sampler.mark()
    barrier(world)
    sampler.stop()
    st = fa.fa_check_device_error(stream)
    if st != fa.FA_OK:
        raise fa.FaError(st, "timed region")
    ms_local = ev0.elapsed_time(ev1)
    ms = reduce_max(ms_local, world, device=dev)
    flops = bwd_flops(w)
    value = world * flops * args.steps / (ms * 1e-3) / 1e12
    achieved = flops / (ms_local / args.steps * 1e-3) / 1e12

    # e2e: inputs (Q, K, V, O, dO, L) from pinned host memory, gradients back
    e2e_steps = max(3, min(args.steps, 20))
    O0, L0 = bufs[0][3].cpu(), bufs[0][5].cpu()
    hosts = [x.pin_memory() for x in (q, k, v, O0, do, L0)]
    outs = [torch.empty(shape, dtype=torch.bfloat16).pin_memory() for _ in range(3)]
    b0 = bufs[0]

    def e2e_step():
        with torch.cuda.stream(stream):
            for dst, src in zip(b0[:6], hosts):
                dst.copy_(src, non_blocking=True)
            call(b0)
            for dst, src in zip(outs, b0[6:]):
                dst.copy_(src, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = reduce_max(e0.elapsed_time(e1), world, device=dev)
    barrier(world)
    peak, hbm_peak, peak_kind = load_peaks()
    # algorithmic bytes: Q, K, V, O, dO read, dQ, dK, dV written, L and delta
    min_bytes = 8 * tensor_b + 2 * l_b
    t_launch = ms_local / args.steps * 1e-3
    if min_bytes / (hbm_peak * 1e9) > flops / (peak * 1e12):
        roofline = {"bound": "hbm", "achieved": round(min_bytes / t_launch / 1e9, 1), "peak": hbm_peak,
                    "unit": "GB/s", "frac": round(min_bytes / t_launch / 1e9 / hbm_peak, 4),
                    "peak_source": f"hbm_gbs of {peak_kind}"}
    else:
        roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                    "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                    "peak_source": f"bf16_tflops (burst) of {peak_kind}"}
    roofline["traffic"] = load_traffic("fa_bwd", w.name)
    return {
        "metric": METRIC_BWD,
        "value": round(value, 2),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "pass": "backward", "B": w.B, "H": w.H, "N": w.N, "D": w.D,
                   "causal": w.causal, "window": list(w.window) or None,
                   "lengths": list(w.lengths) if w.varlen else None,
                   "out_dtype": "bf16", "seed": w.seed,
                   "flops_per_step": flops,
                   "l2": f"inputs rotated over {copies} resident copies "
                         f"({copies * per_copy / 1e6:.0f} MB > 129 MB L2)",
                   "parallelism": f"replicas{world}" if world > 1 else "single-gpu"},
        "roofline": roofline,
        "e2e": {"value": round(world * flops * e2e_steps / (e2e_ms * 1e-3) / 1e12, 2), "unit": UNIT,
                "h2d_bytes_per_step": 5 * tensor_b + l_b, "d2h_bytes_per_step": 3 * tensor_b,
                "steps": e2e_steps},
        "gpu_launches": 3 * args.steps,
        "clocks": sampler.summary(),
    }


def _bwd_oracle_sample(w, views, dos, it, count, seed):
    """Random dQ rows and dK/dV keys of one head and their five-matmul FLOPs
    (2 d per visible pair for each contraction a row or key touches)."""
    import numpy as np
    from oracle import attention_bwd_sampled
    h = it % len(views)
    q, k, v = views[h]
    n = q.shape[0]
    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(n, size=min(count, n), replace=False))
    keys = np.sort(rng.choice(n, size=min(count, n), replace=False))
    vis_r = w.visible_keys(rows, n)
    # rows that see each key: i in [j - wr, j + wl], i >= j under the causal mask
    wl, wr = w.window if w.window else (-1, -1)
    lo = np.maximum(0, keys - wr) if wr >= 0 else np.zeros_like(keys)
    if w.causal:
        lo = np.maximum(lo, keys)
    hi = np.minimum(n - 1, keys + wl) if wl >= 0 else np.full_like(keys, n - 1)
    vis_k = np.maximum(hi - lo + 1, 0)
    fl = float(np.sum(3 * 2 * vis_r * w.D) + np.sum(4 * 2 * vis_k * w.D))
    t0 = time.perf_counter()
    attention_bwd_sampled(q, k, v, dos[h], w.scale, w.causal, rows, keys, window=tuple(w.window) or None)
    return fl, time.perf_counter() - t0, len(rows) + len(keys)


def _bwd_views(w):
    from exact_attention_24_gb300.workloads import make_inputs
    q, k, v = make_inputs(w)
    do = make_inputs(dataclasses.replace(w, seed=w.seed + 50_000))[0]
    qf, kf, vf, dof = (x.double().numpy() for x in (q, k, v, do))
    views = head_views(w, qf, kf, vf)
    dos = [x[0] for x in head_views(w, dof, dof, dof)]
    return views, dos


def cpu_baseline_bwd(w, seconds: float):
    views, dos = _bwd_views(w)
    done, t_total, outs, it = 0.0, 0.0, 0, 0
    while t_total < seconds:
        fl, dt, c = _bwd_oracle_sample(w, views, dos, it, 32, it)
        done += fl
        t_total += dt
        outs += c
        it += 1
    return {"value": done / t_total / 1e12, "unit": UNIT, "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle", "host": host_info(),
            "sample": f"{outs} gradient rows and keys ({it} heads x 32 random dQ rows and 32 random "
                      f"dK/dV keys, each head's forward recomputed) of {w.name}, float64 NumPy, "
                      f"{t_total:.1f} s"}


def bench_reference_bwd(args, w, rank, world):
    """The backward oracle as it stands, on bounded samples sized so that
    warm-up + steps take about 90 s."""
    if rank != 0:
        return None
    views, dos = _bwd_views(w)
    _, dt, c = _bwd_oracle_sample(w, views, dos, 0, 8, 0)
    per_head = max(dt, 1e-4)
    heads = max(1, int(90.0 / max(1, args.steps + args.warmup) / per_head))
    for i in range(args.warmup):
        _bwd_oracle_sample(w, views, dos, 1000 + i, 8, 1000 + i)
    fl_total, t_total = 0.0, 0.0
    for i in range(args.steps):
        for h in range(heads):
            fl, dt, _ = _bwd_oracle_sample(w, views, dos, i * heads + h, 8, i * heads + h)
            fl_total += fl
            t_total += dt
    value = fl_total / t_total / 1e12
    sample = (f"{heads} head(s) per step, 8 random dQ rows and 8 random dK/dV keys each "
              f"(each head's forward recomputed), {args.steps} steps, of {w.name}; "
              f"float64 NumPy backward oracle")
    return {
        "impl": "reference", "metric": METRIC_BWD, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_total / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "pass": "backward", "B": w.B, "H": w.H, "N": w.N,
                   "D": w.D, "causal": w.causal},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": len(os.sched_getaffinity(0)),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# -------------------------------------------------------------- IO model --
def io_model_bytes(w, br: int, bc: int) -> int:
    """HBM bytes of the tiled loop under the byte-counting rule of
    "FlashAttention -- for programmers, not researchers.", STAGE 0 and
    STAGE 4: per head, each br-row query block loads its Q rows once and
    every bc-key K/V tile it needs, then writes its O rows once; nothing is
    cached between blocks.  Here with the workload's element size, only the
    key tiles that the mask leaves visible to some row of the block, and
    the 4-byte L per row that the page's counter leaves out."""
    import numpy as np
    e = 4 if w.dtype == "f32" else 2
    lens = w.lengths if w.varlen else (w.N,) * w.B
    total = 0
    for n in lens:
        kv_rows = 0
        for r0 in range(0, n, br):
            lo, hi = w.visible_range(np.arange(r0, min(n, r0 + br)), n)
            live = hi >= lo
            if live.any():
                first = int(lo[live].min()) // bc * bc
                kv_rows += min(n, (int(hi[live].max()) // bc + 1) * bc) - first
        total += w.H * (e * (2 * n * w.D + 2 * kv_rows * w.D) + 4 * n)
    return int(total)


# --------------------------------------------------------- CPU oracle arm --
def head_views(w, qf, kf, vf):
    """(q, k, v) [n, D] float64 views of every attention problem: each
    (b, h) of a dense batch, or each (sequence, h) of a packed one."""
    views = []
    if w.varlen:
        cu = w.cu_seqlens
        for s in range(len(w.lengths)):
            a, b = int(cu[s]), int(cu[s + 1])
            for h in range(w.H):
                views.append((qf[a:b, h], kf[a:b, h], vf[a:b, h]))
    else:
        for b in range(w.B):
            for h in range(w.H):
                views.append((qf[b, h], kf[b, h], vf[b, h]))
    return views


def oracle_rows_sample(w, view, rows: int, seed: int):
    """Random query rows of one head view and their algorithmic FLOPs."""
    import numpy as np
    n = view[0].shape[0]
    rng = np.random.default_rng(seed)
    picks = np.sort(rng.choice(n, size=min(rows, n), replace=False))
    keys = w.visible_keys(picks, n)
    return picks, float(np.sum(4.0 * keys * w.D))


def run_oracle_sample(w, view, picks):
    from oracle import attention_rows
    attention_rows(view[0], view[1], view[2], w.scale, w.causal, picks,
                   window=tuple(w.window) or None)


def _f64_views(w):
    from exact_attention_24_gb300.workloads import make_inputs
    q, k, v = make_inputs(w)
    qf, kf, vf = (x.double().numpy() for x in (q, k, v))
    return head_views(w, qf, kf, vf)


def host_info() -> dict:
    """The host the oracle runs on: CPU model and the BLAS thread setting."""
    model = ""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu part", "hardware") and not model:
                    model = line.split(":", 1)[1].strip()
    except OSError:
        pass
    threads = {k: os.environ[k] for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
               if k in os.environ}
    return {"cpu_model": model or os.uname().machine, "blas_threads": threads or "library default (all cores)"}


def cpu_baseline(w, seconds: float, seed: int = 0, one_core: bool = True):
    """Time the oracle as it stands on this host's cores, on a bounded sample
    of the workload's rows (float64; causal rows count only their keys)."""
    views = _f64_views(w)
    rows = 64
    done_flops, t_total, n_rows, it = 0.0, 0.0, 0, 0
    while t_total < seconds:
        view = views[it % len(views)]
        picks, fl = oracle_rows_sample(w, view, rows, seed + it)
        t0 = time.perf_counter()
        run_oracle_sample(w, view, picks)
        t_total += time.perf_counter() - t0
        done_flops += fl
        n_rows += len(picks)
        it += 1
    cores = len(os.sched_getaffinity(0))
    rec = {"value": done_flops / t_total / 1e12, "unit": UNIT, "cores": cores,
           "kind": "oracle", "host": host_info(),
           "sample": f"{n_rows} query rows ({it} heads x up to {rows} random rows) of {w.name}, "
                     f"float64 NumPy, {t_total:.1f} s"}
    if one_core and w.flops() < ONE_CORE_MAX_FLOPS:
        rec["one_core"] = cpu_baseline_one_core(w, seconds)
    return rec


# workloads small enough that the oracle is also timed on one core (C1, C2)
ONE_CORE_MAX_FLOPS = 1e10


def cpu_baseline_one_core(w, seconds: float):
    """The same oracle timing in a child process pinned to one core, with the
    BLAS thread pools limited to one thread (set before NumPy loads)."""
    from exact_attention_24_gb300.workloads import WORKLOADS
    if WORKLOADS.get(w.name) is not w:
        return None
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--workload", w.name,
                        "--cpu-one-core", "--cpu-seconds", str(seconds)],
                       env=env, capture_output=True, text=True, timeout=600)
    if r.returncode != 0 or not r.stdout.strip():
        return {"error": (r.stderr.strip().splitlines() or ["no output"])[-1][:200]}
    return json.loads(r.stdout.strip().splitlines()[-1])


def bench_reference(args, w, rank, world):
    if rank != 0:
        return None
    views = _f64_views(w)
    # each step: 64-row samples of successive heads (the size cpu_baseline
    # uses) until the step's share of ~90 s is spent
    rows = 64
    budget = args.ref_seconds / max(1, args.steps + args.warmup)

    def step(seed):
        t, fl, it = 0.0, 0.0, 0
        while t < budget:
            view = views[(seed + it) % len(views)]
            p, f = oracle_rows_sample(w, view, rows, 10_000 * seed + it)
            t0 = time.perf_counter()
            run_oracle_sample(w, view, p)
            t += time.perf_counter() - t0
            fl += f
            it += 1
        return t, fl, it

    for i in range(args.warmup):
        step(1_000 + i)
    t_total, fl_total, n_samples = 0.0, 0.0, 0
    for i in range(args.steps):
        t, fl, it = step(i)
        t_total += t
        fl_total += fl
        n_samples += it
    value = fl_total / t_total / 1e12
    cores = len(os.sched_getaffinity(0))
    sample = (f"{n_samples} samples of up to {rows} random query rows of one head, over {args.steps} "
              f"steps of ~{budget:.0f} s each, of {w.name}; float64 NumPy oracle")
    return {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t_total / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "D": w.D,
                   "causal": w.causal, "window": list(w.window) or None},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


# ------------------------------------------------------------------ main --
def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="seconds of oracle time for cpu_baseline (0 = leave it out)")
    ap.add_argument("--splits", type=int, default=None,
                    help="time fa_fwd_splitkv with this many key splits (0 = automatic)")
    ap.add_argument("--bwd", action="store_true",
                    help="time the backward pass (fa_bwd) instead of the forward pass")
    ap.add_argument("--shape", default=None,
                    help="B,H,N,D[,causal] instead of a named workload (bf16, seed 8)")
    ap.add_argument("--record-traffic", default=None, metavar="NCU_CSV",
                    help="store the DRAM bytes of an ncu --csv capture of this workload (one "
                         "forward launch, or one backward step with --bwd) in "
                         "profiles/traffic.json, then exit")
    ap.add_argument("--captured-with", default="",
                    help="the ncu command line of that capture, kept beside the numbers")
    ap.add_argument("--e2e-runs", type=int, default=E2E_RUNS,
                    help="runs that fa_fwd_host cuts a dense batch into for the e2e measurement")
    ap.add_argument("--ref-seconds", type=float, default=90.0,
                    help="seconds of oracle time that --impl reference spreads over its steps")
    ap.add_argument("--no-extras", dest="extras", action="store_false",
                    help="leave out per_config, sustained and the host-link rate (N=1 runs)")
    ap.add_argument("--config-seconds", type=float, default=0.4,
                    help="minimum timed device seconds of each per_config workload")
    ap.add_argument("--sustained-seconds", type=float, default=2.5,
                    help="minimum timed device seconds of the sustained leg")
    ap.add_argument("--cpu-one-core", action="store_true", help=argparse.SUPPRESS)
    args = ap.parse_args(argv)
    if args.cpu_one_core:
        # child of cpu_baseline_one_core: the oracle timing on the first allowed core
        os.sched_setaffinity(0, {min(os.sched_getaffinity(0))})
        from exact_attention_24_gb300.workloads import WORKLOADS
        rec = cpu_baseline(WORKLOADS[args.workload], args.cpu_seconds, one_core=False)
        print(json.dumps(rec), flush=True)
        return 0
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    from exact_attention_24_gb300.workloads import WORKLOADS, Workload
    if args.shape:
        f = [int(x) for x in args.shape.split(",")]
        if len(f) not in (4, 5):
            ap.error("--shape wants B,H,N,D[,causal]")
        causal = bool(f[4]) if len(f) == 5 else False
        name = f"B{f[0]}_H{f[1]}_N{f[2]}_D{f[3]}_bf16" + ("_causal" if causal else "")
        w = Workload(name, f[0], f[1], f[2], f[3], "bf16", causal, 8)
    else:
        w = WORKLOADS[args.workload]
    if args.record_traffic:
        tag = "fa_bwd" if args.bwd else ("fa_simt" if w.dtype == "f32" else "fa_tc")
        e = record_traffic(args.record_traffic, tag, w.name, args.captured_with)
        print(json.dumps({f"{tag}/{w.name}": e}), flush=True)
        return 0
    rank, world, local = dist_env()
    if world != args.gpus:
        world = max(world, 1)

    if args.impl == "reference":
        rec = (bench_reference_bwd if args.bwd else bench_reference)(args, w, rank, world)
        if rec is not None:
            print(json.dumps(rec), flush=True)
        return 0

    import torch
    init_dist(world, "nccl" if torch.cuda.is_available() else "gloo")
    rec = (bench_bwd if args.bwd else bench_ours)(args, w, rank, world, local)
    if rank == 0:
        if world == 1:
            base = cpu_baseline_bwd if args.bwd else cpu_baseline
            rec["cpu_baseline"] = base(w, args.cpu_seconds) if args.cpu_seconds > 0 else None
        print(json.dumps(rec), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
