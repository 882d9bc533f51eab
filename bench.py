#!/usr/bin/env python
"""Benchmark of the selective-scan hot path on B300, one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one selective scan (softplus, discretisation, recurrence, C readout, D skip,
silu gate, final state) over the largest scan workload, b=1, D=2048, L=131072, N=16, bf16
I/O, fp32 state, split into 2048-step chunks joined by the chunk carry, with inputs
resident in HBM. ``value`` is GB/s of algorithmic bytes (every input read once, every
output written once) over all ranks. ``configs`` holds the same measurement for every
other workload: the tiny fp32 scan (0), the Mamba-130M-shaped layer (1), the
Mamba-2.8B-shaped layer (2) and the SSD chunked scan (4, TFLOP/s). Each scan entry carries
the duration of every kernel of the call (CUDA events recorded between the kernels inside
the timed region) and the roofline of the dominant one. Under torchrun each rank runs its
own replica (different seed): the path shards with no collective, so scaling is weak.

``--impl reference`` times the fp64 CPU oracle instead, on bounded samples of the same
workload (rank 0 only), and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "selective-scan GB/s and fraction of B300 HBM peak; SSD TFLOP/s (1 GPU)"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "sm_max_mhz": 2032.0}
SMS = 148
# Per-SM, per-clock rates measured on this B300 by the unit-rate microbenchmark
# (python -m selective_state_space_127_b300.unit_rates): ex2.approx.f32 at 32 per clock per SM,
# packed FP32 FMA at 128 lanes per clock per SM. A delta*B state update needs one ex2 and four
# FP32 lane operations, so both pipes cap it at 32 updates per clock per SM.
UPDATES_PER_CLK_SM = 32.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=3, choices=[1, 2, 3],
                    help="the headline scan workload (default: the largest, b1 D2048 L131072)")
    ap.add_argument("--no-ssd", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-conv", action="store_true", help="skip the conv1d + SiLU prologue measurements")
    ap.add_argument("--no-variants", action="store_true", help="skip the exact-ZOH and reverse measurements")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the scan configs other than the headline")
    ap.add_argument("--seqlen", type=int, default=0,
                    help="shorten the headline workload to this many steps (smaller profiling captures; the "
                         "line then names the shortened workload)")
    return ap.parse_args()


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ work accounting

def scan_bytes(w, batch=None, dim=None, seqlen=None):
    """Algorithmic bytes of one selective scan: x, delta, z read and y written once in the
    I/O dtype; B, C read once; A, D, bias read once (fp32); h_last written once (fp32)."""
    b, d, L, n = batch or w.batch, dim or w.dim, seqlen or w.seqlen, w.dstate
    io = 2 if w.dtype == "bf16" else 4
    per_bld = (3 + (1 if w.gate else 0)) * io       # x, delta, (z) in, y out
    tot = b * L * d * per_bld + 2 * b * L * n * io
    tot += d * n * 4 + d * 4 * (2 if w.d_skip != "none" else 1) + b * d * n * 4
    return tot


def ssd_bytes(w):
    io = 2
    return (2 * w.batch * w.seqlen * w.nheads * w.headdim * io + w.batch * w.seqlen * w.nheads * io
            + 2 * w.batch * w.seqlen * w.dstate * io + 2 * w.nheads * 4
            + w.batch * w.nheads * w.dstate * w.headdim * 4)


def ssd_flops(w):
    """Useful flops of the chunked SSD algorithm: C B^T (causal half, once per batch and
    chunk since B and C are head-shared), masked-block times X (causal half), C times the
    carried state, and the chunk-state update B^T X."""
    nch = (w.seqlen + w.chunk - 1) // w.chunk
    Q, N, P = w.chunk, w.dstate, w.headdim
    cb = w.batch * nch * Q * Q * N                 # 2 * Q*Q/2 * N
    diag = w.batch * w.nheads * nch * Q * Q * P    # 2 * Q*Q/2 * P
    off = w.batch * w.nheads * nch * 2 * Q * N * P
    state = w.batch * w.nheads * nch * 2 * Q * N * P
    return cb + diag + off + state


def ssd_mma_flops(w, block=128):
    """Flops the tensor-core SSD kernel executes: per (batch, head, 128-step block) the dense
    products G = C B^T (2*Q*Q*N), Y = M X (2*Q*Q*P), the hand-off (exp(cum) o C) S_prev
    (2*Q*N*P) and the state product (w o B)^T X (2*Q*N*P)."""
    nblk = (w.seqlen + block - 1) // block
    per = 2 * block * block * w.dstate + 2 * block * block * w.headdim + 4 * block * w.dstate * w.headdim
    return w.batch * w.nheads * nblk * per


def profiled_traffic(kernel_file, summary):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) recorded in a
    profile summary under profiles/, if that summary was taken of the current source of the
    kernel (its sha256 matches); else None."""
    import hashlib
    import re
    if not summary:
        return None
    src = os.path.join(ROOT, "selective_state_space_127_b300", "csrc", kernel_file)
    path = os.path.join(ROOT, "profiles", summary)
    if not (os.path.isfile(src) and os.path.isfile(path)):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*(\d+)\s+source_sha256:\s*([0-9a-f]{64})", text)
    if not m:
        return None
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()
    return int(m.group(1)) if digest == m.group(2) else None


# ------------------------------------------------------------------ clocks during the timed region

class ClockSampler:
    """Samples SM clock and throttle reasons with `nvidia-smi -lms 100` (read-only) while the
    benchmark runs; summary() reports the samples taken inside the marked timed window (or,
    if the window was shorter than the sampling period, those of the whole loaded phase)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        import subprocess
        import torch
        self.rows = []
        self.window = None
        self.err = None
        try:
            uuid = "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", uuid, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception as e:  # reported in the JSON line
            self.proc, self.err = None, str(e)

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 7:
                self.rows.append((time.time(), parts))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=5)

    def summary(self):
        if self.proc is None:
            return {"error": self.err}
        rows = self.rows
        in_window = False
        if self.window:
            inside = [r for r in rows if self.window[0] - 0.05 <= r[0] <= self.window[1] + 0.05]
            if inside:
                rows, in_window = inside, True

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        mhz = [num(r[1][0]) for r in rows if num(r[1][0]) is not None]
        mx = [num(r[1][1]) for r in rows if num(r[1][1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[1][3 + i].lower().startswith("active")})
        watts = [num(r[1][2]) for r in rows if num(r[1][2]) is not None]
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(watts) if watts else None, "samples": len(rows), "in_window": in_window,
                "reasons": reasons, "source": "nvidia-smi, 100 ms",
                **({"nvml_unused": self.nvml_error} if getattr(self, "nvml_error", None) else {})}


class _NvmlLib:
    """The few read-only NVML calls the clock record needs, through ctypes on the driver's
    libnvidia-ml (no Python bindings needed)."""
    CLOCK_SM = 1

    def __init__(self):
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        self._ok(self.lib.nvmlInit_v2())
        f = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self._reasons = f if f is not None else self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    @staticmethod
    def _ok(r):
        if r != 0:
            raise RuntimeError(f"NVML error {r}")

    def handle(self, uuid, index):
        h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) != 0:
            self._ok(self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h)))
        return h

    def sm_mhz(self, h):
        v = ctypes.c_uint()
        self._ok(self.lib.nvmlDeviceGetClockInfo(h, self.CLOCK_SM, ctypes.byref(v)))
        return v.value

    def max_sm_mhz(self, h):
        v = ctypes.c_uint()
        self._ok(self.lib.nvmlDeviceGetMaxClockInfo(h, self.CLOCK_SM, ctypes.byref(v)))
        return v.value

    def watts(self, h):
        v = ctypes.c_uint()
        self._ok(self.lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(v)))
        return v.value / 1000.0

    def reasons(self, h):
        v = ctypes.c_ulonglong()
        self._ok(self._reasons(h, ctypes.byref(v)))
        return v.value

    def shutdown(self):
        self.lib.nvmlShutdown()


class NvmlClockSampler:
    """The same record as ClockSampler from NVML (read-only queries: SM clock, maximum SM clock,
    power draw, active clock-event reasons) every 5 ms in a thread, so that a timed region of a
    few tens of milliseconds still holds several samples."""

    # clock-event reason bits of NVML's public header
    BITS = (("hw_slowdown", 0x8), ("hw_thermal_slowdown", 0x40), ("sw_thermal_slowdown", 0x20),
            ("sw_power_cap", 0x4))

    def __init__(self, device_index, period_s=0.005):
        import torch
        self.nv = _NvmlLib()
        uuid = "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)
        visible = os.environ.get("CUDA_VISIBLE_DEVICES")
        self.h = self.nv.handle(uuid, int(visible.split(",")[device_index]) if visible and
                                visible.split(",")[device_index].isdigit() else device_index)
        self.max_mhz = self.nv.max_sm_mhz(self.h)
        self.rows, self.window, self.period = [], None, period_s
        self.done = threading.Event()
        self.t = threading.Thread(target=self._run, daemon=True)
        self.t.start()

    def _run(self):
        while not self.done.is_set():
            try:
                self.rows.append((time.time(), self.nv.sm_mhz(self.h), self.nv.watts(self.h),
                                  self.nv.reasons(self.h)))
            except Exception:
                pass
            self.done.wait(self.period)

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        self.done.set()
        self.t.join(timeout=5)
        try:
            self.nv.shutdown()
        except Exception:
            pass

    def summary(self):
        rows, in_window = self.rows, False
        if self.window:
            inside = [r for r in rows if self.window[0] <= r[0] <= self.window[1]]
            if inside:
                rows, in_window = inside, True
        reasons = sorted({name for r in rows for name, bit in self.BITS if r[3] & bit})
        mhz = [r[1] for r in rows]
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": self.max_mhz,
                "power_w_max": max(r[2] for r in rows) if rows else None, "samples": len(rows),
                "in_window": in_window, "reasons": reasons, "source": "nvml, 5 ms"}


def clock_sampler(device_index):
    """NVML sampling when the NVML bindings load, else nvidia-smi (the reason is recorded)."""
    try:
        return NvmlClockSampler(device_index)
    except Exception as e:
        c = ClockSampler(device_index)
        c.nvml_error = f"{type(e).__name__}: {e}"[:200]
        return c


# ------------------------------------------------------------------ oracle timing (CPU)

def _oracle_sample(w, target_s, threads=None):
    """Pick a sample (batch rows, channels) of workload w that the oracle finishes in about
    target_s seconds on this host with `threads` threads (default: all), from a probe of one
    channel per thread."""
    import oracle
    from selective_state_space_127_b300.synth import make_scan_inputs, SEED_BASE

    threads = threads or oracle.max_threads()
    probe_d = max(1, min(w.dim, threads))
    inp = make_scan_inputs(1, w.seqlen, probe_d, w.dstate, w.dtype, SEED_BASE + 1, "cpu", w.d_skip, w.gate)
    conv = {k: (oracle.f64(v) if v is not None else None) for k, v in inp.items()}
    t0 = time.perf_counter()
    oracle.ssm_scan_ref(**conv, nthreads=threads)
    probe_s = max(time.perf_counter() - t0, 1e-6)
    chans = max(probe_d, int(probe_d * target_s / probe_s))     # channel-sequences that fit
    rows = max(1, min(w.batch, chans // w.dim))
    d = w.dim if rows > 1 or chans >= w.dim else max(1, chans)
    return rows, d, threads


def _oracle_inputs(w, rows, d):
    import oracle
    from selective_state_space_127_b300.synth import make_scan_inputs, SEED_BASE

    inp = make_scan_inputs(rows, w.seqlen, d, w.dstate, w.dtype, SEED_BASE + 1, "cpu", w.d_skip, w.gate)
    return {k: (oracle.f64(v) if v is not None else None) for k, v in inp.items()}


def time_oracle_scan(w, target_s=12.0, threads=None):
    """Time the fp64 oracle on a bounded sample of workload w (all L steps of some batch rows
    and channels, about target_s seconds) with `threads` threads (default: all). Returns
    (GB/s, seconds, sample, threads)."""
    import oracle

    rows, d, threads = _oracle_sample(w, target_s, threads)
    conv = _oracle_inputs(w, rows, d)
    t0 = time.perf_counter()
    oracle.ssm_scan_ref(**conv, nthreads=threads)
    dt = time.perf_counter() - t0
    nbytes = scan_bytes(w, batch=rows, dim=d)
    return nbytes / dt / 1e9, dt, f"{rows} of {w.batch} batch rows, {d} of {w.dim} channels, all {w.seqlen} steps", threads


# ------------------------------------------------------------------ GPU arm

def _timed(fn, steps, warmup, stream, barrier=None):
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    return e0.elapsed_time(e1) / steps  # ms per step


def _max_over_ranks(v, dev, world):
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], device=dev, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or "unknown"


def scan_phases(w, chunk):
    """The kernels one scan call of workload w launches, as (name, state updates, algorithmic
    bytes) each: one output pass when the sequence is one chunk; else the local pass over all
    chunks but the last (x, delta, B in; chunk end states and sums of dt out), the chunk carry
    (end states in, initial states out) and the output pass (the whole scan's bytes plus the
    initial states read)."""
    io = 2 if w.dtype == "bf16" else 4
    b, L, D, N = w.batch, w.seqlen, w.dim, w.dstate
    nch = (L + chunk - 1) // chunk
    if nch <= 1:
        return [("scan", w.units, scan_bytes(w))]
    Lp1 = L - (L - (nch - 1) * chunk)           # steps of the local pass
    p1_units = b * Lp1 * D * N
    p1_bytes = b * Lp1 * D * 2 * io + b * Lp1 * N * io + (nch - 1) * b * D * (N + 1) * 4 + D * N * 4 + D * 4
    carry_bytes = 2 * nch * b * D * N * 4 + (nch - 1) * b * D * 4 + D * N * 4
    p2_bytes = scan_bytes(w) + nch * b * D * N * 4
    return [("local pass", p1_units, p1_bytes), ("chunk carry", 0, carry_bytes), ("output pass", w.units, p2_bytes)]


def bench_scan(k, steps, warmup, dev, rank, world, barrier, peaks, with_phases=True, seqlen=0):
    """Time scan workload k: `warmup` untimed steps, then `steps` steps between CUDA events on
    the launching stream. With phase events each step records an event before its first
    kernel and after each kernel, so every kernel's average duration inside the timed region
    is known. Returns a result dict (per-rank times reduced by max over ranks)."""
    import torch
    from selective_state_space_127_b300 import ScanCall, binding, ssm_scan_fwd
    from selective_state_space_127_b300.synth import SCAN_WORKLOADS, scan_workload_inputs

    w = SCAN_WORKLOADS[k]
    if seqlen:
        import dataclasses
        w = dataclasses.replace(w, seqlen=seqlen, name=w.name.replace(f"L{w.seqlen}", f"L{seqlen}"))
    inp = scan_workload_inputs(k, device=dev, rank=rank, seqlen=seqlen or None)
    y = torch.empty_like(inp["x"])
    hl = torch.empty(w.batch, w.dim, w.dstate, device=dev, dtype=torch.float32)
    stream = torch.cuda.current_stream(dev)
    call = ScanCall(**inp, out=y, h_last=hl, chunk_len=w.chunk_len)
    from selective_state_space_127_b300.binding import _event_array
    nph = 4
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nph)] for _ in range(steps)] if with_phases else []
    arrays = []
    for row in evs:
        for e in row:
            e.record(stream)
        arrays.append(_event_array(row)[0])
    p = call._p
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    n0 = binding.kernel_launch_count()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    e0.record(stream)
    th0 = time.perf_counter()
    for i in range(steps):
        if with_phases:
            p.phase_events, p.n_phase_events = ctypes.cast(arrays[i], ctypes.POINTER(ctypes.c_void_p)), nph
        call()
    th1 = time.perf_counter()
    e1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if barrier:
        barrier()
    p.phase_events, p.n_phase_events = None, 0
    launches = binding.kernel_launch_count() - n0
    ms = _max_over_ranks(e0.elapsed_time(e1) / steps, dev, world)
    # host time of the binding's one-shot entry point (argument checks, params, C call)
    tb0 = time.perf_counter()
    nb = 20
    for _ in range(nb):
        ssm_scan_fwd(**inp, out=y, h_last=hl, chunk_len=w.chunk_len, workspace=call.workspace)
    tb1 = time.perf_counter()
    torch.cuda.synchronize()
    nbytes = scan_bytes(w)
    gbs = nbytes / (ms * 1e-3) / 1e9
    res = {"workload": w.name, "ms_per_step": round(ms, 5), "steps": steps, "warmup": warmup,
           "gbs": round(gbs * world, 2), "hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
           "hbm_frac_of_8tbs": round(gbs / 8000.0, 4), "algorithmic_bytes": nbytes, "updates": w.units,
           "gupdates_per_s": round(w.units / (ms * 1e-3) / 1e9, 1),
           "host_us_per_call": {"prepared (ScanCall)": round((th1 - th0) / steps * 1e6, 1),
                                "ssm_scan_fwd": round((tb1 - tb0) / nb * 1e6, 1)},
           "gpu_launches": int(launches), "_window": (t_wall0, t_wall1)}
    if with_phases:
        chunk = _chunk_of(w)
        phases = scan_phases(w, chunk)
        kern = []
        for j, (name, units, pbytes) in enumerate(phases):
            dur = sum(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(steps)) / steps
            dur = _max_over_ranks(dur, dev, world)
            kern.append({"kernel": name, "ms": round(dur, 5), "units": units, "algorithmic_bytes": pbytes,
                         "gbs": round(pbytes / (dur * 1e-3) / 1e9, 1) if dur > 0 else None,
                         "gupdates_per_s": round(units / (dur * 1e-3) / 1e9, 1) if dur > 0 and units else None})
        res["kernels"] = kern
        dom = max(kern, key=lambda r: r["ms"])
        mhz = peaks.get("sm_max_mhz", 2032.0)
        alu_peak = UPDATES_PER_CLK_SM * SMS * mhz * 1e6 / 1e9
        achieved = dom["units"] / (dom["ms"] * 1e-3) / 1e9
        res["roofline"] = {"bound": "alu", "achieved": round(achieved, 1), "peak": round(alu_peak, 1),
                           "unit": "Gupdate/s", "frac": round(achieved / alu_peak, 4), "kernel": dom["kernel"],
                           "units_per_launch": dom["units"], "ms_per_launch": dom["ms"],
                           "hbm": {"achieved": dom["gbs"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                   "frac": round(dom["gbs"] / peaks["hbm_gbs"], 4),
                                   "algorithmic_bytes": dom["algorithmic_bytes"]},
                           "traffic": profiled_traffic("scan_fast.cuh", PROFILE_OF.get(k, "")),
                           "peak_basis": f"{UPDATES_PER_CLK_SM:.0f} updates/clk/SM x {SMS} SMs x {mhz:.0f} MHz: "
                                         "one SFU ex2 per update at the measured 32/clk/SM "
                                         "(profiles/unit_rates_b300.md)"}
    del inp, y, hl, call
    return res


def _chunk_of(w):
    """Steps per chunk of workload w's scan as the library picks them (the TMA path rounds the
    requested chunk to a multiple of its 32-step tile; 0 = one chunk for these workloads)."""
    if w.chunk_len:
        return ((w.chunk_len + 31) // 32) * 32
    return ((w.seqlen + 31) // 32) * 32


PROFILE_OF = {1: "scan_fast_b8_D1536_L2048_N16_bf16.md", 3: "scan_fast_b1_D2048_L131072_N16_bf16.md"}


def copy_ceiling(nbytes_in, nbytes_out, dev):
    """Plain pinned host<->device copy bandwidth on this machine (GB/s), the ceiling of the e2e
    number: nbytes_in host->device and nbytes_out device->host, each timed alone."""
    import torch
    hin = torch.empty(nbytes_in, dtype=torch.uint8, pin_memory=True)
    din = torch.empty(nbytes_in, dtype=torch.uint8, device=dev)
    dout = torch.empty(nbytes_out, dtype=torch.uint8, device=dev)
    hout = torch.empty(nbytes_out, dtype=torch.uint8, pin_memory=True)
    res = {}
    for name, (dst, src, n) in (("h2d", (din, hin, nbytes_in)), ("d2h", (hout, dout, nbytes_out))):
        dst.copy_(src, non_blocking=True)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(3):
            dst.copy_(src, non_blocking=True)
        torch.cuda.synchronize()
        res[name + "_gbs"] = round(3 * n / (time.perf_counter() - t0) / 1e9, 2)
    t_serial = nbytes_in / (res["h2d_gbs"] * 1e9) + nbytes_out / (res["d2h_gbs"] * 1e9)
    res["serial_ms_per_step"] = round(t_serial * 1e3, 3)
    # both directions at once on two streams (the link is full duplex): the ceiling of a
    # pipeline whose copies in and out overlap
    s1, s2 = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(3):
        with torch.cuda.stream(s1):
            din.copy_(hin, non_blocking=True)
        with torch.cuda.stream(s2):
            hout.copy_(dout, non_blocking=True)
    torch.cuda.synchronize()
    res["duplex_ms_per_step"] = round((time.perf_counter() - t0) / 3 * 1e3, 3)
    del hin, din, dout, hout
    return res


def run_ours(args):
    import torch
    import torch.distributed as dist
    from selective_state_space_127_b300 import binding, causal_conv1d_fwd, ssd_chunk_scan_fwd, ssm_scan_fwd, \
        ssm_scan_fwd_host
    from selective_state_space_127_b300.synth import (SCAN_WORKLOADS, SSD_WORKLOAD, scan_workload_inputs,
                                                      ssd_workload_inputs)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    barrier = (lambda: dist.barrier(device_ids=[local])) if world > 1 else None
    binding.load_library()
    peaks, peak_src = load_peaks()
    stream = torch.cuda.current_stream()
    clk = clock_sampler(local)
    few = max(3, min(args.steps, 20))

    # the other scan workloads first (they also bring the GPU to its working clock)
    configs = {}
    for k in (0, 1, 2):
        if k == args.workload or args.no_configs:
            continue
        r = bench_scan(k, few, 3, dev, rank, world, barrier, peaks)
        r.pop("_window")
        if k == 0:
            r["note"] = "6 KB problem: launch-latency bound and L2-resident (a correctness config)"
        configs[str(k)] = r

    # the headline: exactly `steps` timed steps after `warmup` untimed ones
    head = bench_scan(args.workload, args.steps, args.warmup, dev, rank, world, barrier, peaks, seqlen=args.seqlen)
    w = SCAN_WORKLOADS[args.workload]
    if args.seqlen:
        import dataclasses
        w = dataclasses.replace(w, seqlen=args.seqlen, name=head["workload"])
    t_w0, t_w1 = head.pop("_window")
    clk.mark(t_w0, t_w1)
    ms = head["ms_per_step"]
    nbytes = head["algorithmic_bytes"]
    gbs_rank = nbytes / (ms * 1e-3) / 1e9
    result = {
        "metric": METRIC, "value": round(gbs_rank * world, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded torch generator on the device)",
        "config": {"workload": w.name, "batch": w.batch, "seqlen": w.seqlen, "dim": w.dim, "dstate": w.dstate,
                   "io_dtype": w.dtype, "state_dtype": "f32", "d_skip": True, "gate": True, "h_last": True,
                   "chunk_len": w.chunk_len,
                   "l2": f"inputs larger than L2 ({nbytes / 1e6:.0f} MB per step > 126 MB); no flush",
                   "parallelism": f"replicas x{world}"},
        "hbm_frac": head["hbm_frac"], "hbm_frac_of_8tbs": head["hbm_frac_of_8tbs"],
        "hbm_peak_gbs": peaks["hbm_gbs"], "peak_source": peak_src,
        "roofline": head["roofline"], "kernels": head["kernels"],
        "host_us_per_call": head["host_us_per_call"],
        "gpu_launches": head["gpu_launches"],
        "host_cpu": {"model": cpu_model(), "cores": len(os.sched_getaffinity(0))},
    }
    configs[str(args.workload)] = {kk: v for kk, v in head.items() if kk not in ("roofline",)}
    configs[str(args.workload)]["roofline"] = head["roofline"]

    if not args.no_ssd:
        sw = SSD_WORKLOAD
        sinp = ssd_workload_inputs(device=dev, rank=rank)
        sy = torch.empty_like(sinp["x"])
        shl = torch.empty(sw.batch, sw.nheads, sw.dstate, sw.headdim, device=dev, dtype=torch.float32)
        sws = binding.new_workspace(binding.WORKSPACE_HEADER_BYTES, dev)

        def sstep():
            ssd_chunk_scan_fwd(**sinp, chunk_size=sw.chunk, out=sy, h_last=shl, workspace=sws)

        ssteps = max(3, min(args.steps, 50))
        sms = _max_over_ranks(_timed(sstep, ssteps, 3, stream, barrier), dev, world)
        fl = ssd_flops(sw)
        tf = fl / (sms * 1e-3) / 1e12
        mma = ssd_mma_flops(sw)
        mma_tf = mma / (sms * 1e-3) / 1e12
        sgbs = ssd_bytes(sw) / (sms * 1e-3) / 1e9
        configs["4"] = {
            "workload": sw.name, "ms_per_step": round(sms, 4), "steps": ssteps,
            "tflops": round(tf * world, 2), "unit": "TFLOP/s", "flops_per_step": fl,
            "flops_basis": "algorithmic: causal halves, C B^T once per (batch, 256-step chunk)",
            "gbs": round(sgbs * world, 1), "hbm_frac": round(sgbs / peaks["hbm_gbs"], 4),
            "hbm_frac_of_8tbs": round(sgbs / 8000.0, 4), "algorithmic_bytes": ssd_bytes(sw),
            "executed_mma": {"flops_per_launch": mma, "tflops": round(mma_tf, 1),
                             "frac_of_bf16_burst": round(mma_tf / peaks["bf16_tflops"], 4)},
            "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": round(tf / peaks["bf16_tflops"], 4),
                         "traffic": profiled_traffic("ssd_tc.cu", "ssd_tc_b4_H64_P64_N128_L4096_bf16.md"),
                         "kernel": "ssd_tc_kernel", "flops_per_launch": fl,
                         "peak_basis": "measured bf16 dense burst (cuBLAS 8192^3); algorithmic flops"}}
        del sinp, sy, shl

    # inputs of workload 1 for the remaining kernel measurements
    w1 = SCAN_WORKLOADS[1]
    inp1 = scan_workload_inputs(1, device=dev, rank=rank)
    y1 = torch.empty_like(inp1["x"])
    hl1 = torch.empty(w1.batch, w1.dim, w1.dstate, device=dev, dtype=torch.float32)
    ws1 = binding.new_workspace(binding.scan_workspace_size(**inp1), dev)
    ms1 = configs["1"]["ms_per_step"] if "1" in configs else None
    nbytes1 = scan_bytes(w1)

    if not args.no_conv:
        # causal conv1d (4 taps) + SiLU: the standalone kernel on 4x workload 1's x (so that its
        # input plus output exceed L2), and the scan of workload 1 with the prologue fused
        K = 4
        gconv = torch.Generator(device=dev).manual_seed(20261202 + 40 + rank)
        cw = torch.randn(w1.dim, K, generator=gconv, device=dev) / K ** 0.5
        cb = 0.1 * torch.randn(w1.dim, generator=gconv, device=dev)
        cx = torch.randn(4 * w1.batch, w1.seqlen, w1.dim, generator=gconv, device=dev).to(inp1["x"].dtype)
        cy = torch.empty_like(cx)
        cws = binding.new_workspace(binding.WORKSPACE_HEADER_BYTES, dev)

        def cstep():
            causal_conv1d_fwd(cx, cw, cb, silu=True, out=cy, workspace=cws)

        csteps = max(3, min(args.steps, 200))
        cms = _max_over_ranks(_timed(cstep, csteps, 3, stream, barrier), dev, world)
        cbytes = 2 * cx.numel() * cx.element_size() + cw.numel() * 4 + cb.numel() * 4
        cgbs = cbytes / (cms * 1e-3) / 1e9
        del cx, cy

        def fstep():
            ssm_scan_fwd(**inp1, out=y1, h_last=hl1, workspace=ws1, conv_weight=cw, conv_bias=cb)

        fms = _max_over_ranks(_timed(fstep, few, 3, stream, barrier), dev, world)
        fbytes = nbytes1 + cw.numel() * 4 + cb.numel() * 4
        result["conv1d"] = {
            "workload": f"causal conv1d K{K} + SiLU, b{4 * w1.batch} L{w1.seqlen} D{w1.dim} {w1.dtype} "
                        "(4x the scan's batch so that in + out > L2)",
            "ms_per_step": round(cms, 4), "steps": csteps, "value": round(cgbs * world, 1), "unit": "GB/s",
            "roofline": {"bound": "hbm", "achieved": round(cgbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(cgbs / peaks["hbm_gbs"], 4), "algorithmic_bytes": cbytes,
                         "traffic": profiled_traffic("conv1d.cu", "conv1d_b32_L2048_D1536_K4_bf16.md"),
                         "kernel": "conv1d_kernel"},
            "fused_scan": {"workload": w1.name + " with the conv1d + SiLU prologue on x",
                           "ms_per_step": round(fms, 4), "gbs": round(fbytes / (fms * 1e-3) / 1e9 * world, 1),
                           "vs_plain_scan": round(fms / ms1, 3) if ms1 else None}}

    if not args.no_variants:
        # the exact-ZOH discretisation and the reverse direction on workload 1 (TMA kernel variants),
        # and the in-tile associative scan (the other algorithm of the same call)
        variants = {}
        kernel_of = {"zoh": "scan_fast_kernel (zoh variant)", "reverse": "scan_fast_kernel (reverse variant)",
                     "assoc_scan": "scan_assoc_kernel (algorithm=assoc)"}
        for name, kw in (("zoh", {"zoh": True}), ("reverse", {"reverse": True}),
                         ("assoc_scan", {"algorithm": "assoc"})):
            def vstep(kw=kw):
                ssm_scan_fwd(**inp1, out=y1, h_last=hl1, workspace=ws1, **kw)
            vms = _max_over_ranks(_timed(vstep, few, 3, stream, barrier), dev, world)
            variants[name] = {"ms_per_step": round(vms, 4), "gbs": round(nbytes1 / (vms * 1e-3) / 1e9 * world, 1),
                              "vs_plain_scan": round(vms / ms1, 3) if ms1 else None,
                              "kernel": kernel_of[name]}
        result["variants"] = dict(workload=w1.name, **variants)

    if not args.no_decode:
        # single-token recurrent step with the state advanced in place, workload 1's shapes
        dinp = {k: (v[:, :1].contiguous() if k in ("x", "delta", "B", "C", "z") else v) for k, v in inp1.items()}
        dstate = torch.zeros(w1.batch, w1.dim, w1.dstate, device=dev, dtype=torch.float32)
        dy = torch.empty_like(dinp["x"])

        def dstep():
            ssm_scan_fwd(**dinp, h0=dstate, h_last=dstate, out=dy)

        # a decode step is launch-bound: capture 32 steps in a CUDA graph and replay it
        for _ in range(3):
            dstep()
        torch.cuda.synchronize()
        per_graph = 32
        graph = torch.cuda.CUDAGraph()
        gstream = torch.cuda.Stream(device=dev)
        gstream.wait_stream(stream)
        with torch.cuda.stream(gstream):
            with torch.cuda.graph(graph, stream=gstream):
                for _ in range(per_graph):
                    dstep()
        torch.cuda.synchronize()
        dsteps = 20
        dms = _max_over_ranks(_timed(graph.replay, dsteps, 3, stream, barrier), dev, world) / per_graph
        state_bytes = 2 * w1.batch * w1.dim * w1.dstate * 4
        io_bytes = scan_bytes(w1, seqlen=1) - w1.batch * w1.dim * w1.dstate * 4
        result["decode"] = {"workload": f"b{w1.batch} D{w1.dim} N{w1.dstate} {w1.dtype}, one token, state in place",
                            "us_per_token": round(dms * 1e3, 3), "steps": dsteps * per_graph,
                            "launch": "CUDA graph of 32 steps through the C ABI",
                            "gbs": round((state_bytes + io_bytes) / (dms * 1e-3) / 1e9 * world, 1),
                            "bytes_per_token": state_bytes + io_bytes}
    del inp1, y1, hl1

    if not args.no_e2e:
        # the headline workload end to end through the C ABI from pinned host buffers
        inp = scan_workload_inputs(args.workload, device=dev, rank=rank, seqlen=args.seqlen or None)
        host = {k: (v.cpu().pin_memory() if v is not None else None) for k, v in inp.items()}
        del inp
        bufs = {}
        ssm_scan_fwd_host(host, device=dev, dev_buffers=bufs, chunk_len=w.chunk_len)
        e2e_steps = max(3, min(args.steps, 5))
        torch.cuda.synchronize()
        if barrier:
            barrier()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            ssm_scan_fwd_host(host, device=dev, dev_buffers=bufs, chunk_len=w.chunk_len)
        e2e_s = _max_over_ranks((time.perf_counter() - t0) / e2e_steps, dev, world)
        h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
        d2h = bufs["_y_host"].numel() * bufs["_y_host"].element_size() + bufs["_h_last_host"].numel() * 4
        del bufs, host
        torch.cuda.empty_cache()
        ceil = copy_ceiling(h2d, d2h, dev)
        result["e2e"] = {"value": round(nbytes / e2e_s / 1e9 * world, 2), "unit": "GB/s",
                         "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                         "ms_per_step": round(e2e_s * 1e3, 3), "steps": e2e_steps,
                         "api": "ssm_scan_fwd_host (pinned host in, pinned host out)",
                         "copy_ceiling": dict(ceil, basis="plain pinned copies of the same bytes: each direction "
                                                          "timed alone (3 copies), then both at once on two "
                                                          "streams"),
                         "frac_of_duplex_copies": round(ceil["duplex_ms_per_step"] / (e2e_s * 1e3), 3)}

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        gbs, secs, sample, threads = time_oracle_scan(w)
        result["cpu_baseline"] = {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                                  "sample": sample, "seconds": round(secs, 2), "cpu": cpu_model()}
        gbs1, secs1, sample1, _ = time_oracle_scan(w, 4.0, threads=1)
        result["cpu_baseline"]["single_thread"] = {"value": round(gbs1, 4), "unit": "GB/s", "cores": 1,
                                                   "sample": sample1, "seconds": round(secs1, 2)}
    time.sleep(0.15)
    clk.stop()
    result["clocks"] = clk.summary()
    result["configs"] = configs

    if world > 1:
        dist.barrier(device_ids=[local])
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(result), flush=True)


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    from selective_state_space_127_b300.synth import SCAN_WORKLOADS

    w = SCAN_WORKLOADS[args.workload]
    # size one step so that warmup + steps stay within about three minutes
    budget = min(10.0, 180.0 / max(1, args.steps + args.warmup))
    rows, d, threads = _oracle_sample(w, budget)
    conv = _oracle_inputs(w, rows, d)
    for _ in range(args.warmup):
        oracle.ssm_scan_ref(**conv, nthreads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.ssm_scan_ref(**conv, nthreads=threads)
    dt = (time.perf_counter() - t0) / args.steps
    nbytes = scan_bytes(w, batch=rows, dim=d)
    gbs = nbytes / dt / 1e9
    sample = f"{rows} of {w.batch} batch rows, {d} of {w.dim} channels, all {w.seqlen} steps (fp64 oracle)"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "sample": sample},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
