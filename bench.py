#!/usr/bin/env python3
"""Benchmark of the row-wise normalization library on one or more GPUs.

Default workload: fused residual-add + RMSNorm, bf16, x and residual
[4096, 4096], w [4096], eps 1e-6 (seeded synthetic inputs).  Metric: achieved
HBM GB/s of algorithmic bytes (read x and residual once, write residual_out
and y once, read w) and us/call.

Timing: inputs are resident in HBM before the timed region; R rotating input
sets whose total size exceeds 3x L2 are used round-robin, so every call reads
cold inputs.  The K steps are captured in CUDA graphs and replayed between two
CUDA events on the launching stream, after W warm-up steps, bracketed by a
barrier and torch.cuda.synchronize(); a short spin kernel queued before the
first event keeps the host's launch latency out of the timed region.  SM
clocks and throttle reasons are sampled (NVML) during the timed region.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl nrm|reference]
"""
from __future__ import annotations

import argparse
import ctypes
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
import torch  # noqa: E402

from row_wise_normalization_reduce_gb300 import workloads as W  # noqa: E402

METRIC = "achieved HBM GB/s (% of GB300 peak) and µs/call, add+RMSNorm 4096x4096 bf16"
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# bytes
# ---------------------------------------------------------------------------
def algorithmic_bytes(w: W.Workload, stats: bool = True) -> int:
    """Bytes an ideal kernel moves per call: every input read once, every output
    written once (parameters and statistics included)."""
    es = torch.tensor([], dtype=w.torch_dtype).element_size()
    if w.op.startswith("bn"):
        c = w.shape[1]
        n = int(np.prod(w.shape))
        if w.op == "bn":      # x, y; gamma, beta; save_mean/rstd; running stats r+w
            return 2 * n * es + 2 * c * es + 2 * c * 4 + 4 * c * 4
        if w.op == "bn_infer":  # x, y; gamma, beta; running stats read
            return 2 * n * es + 2 * c * es + 2 * c * 4
        if w.op == "bn_bwd":  # dy, x, dx; gamma; save_mean/rstd; dgamma, dbeta
            return 3 * n * es + c * es + 4 * c * 4
    rows, n = w.shape
    t = rows * n * es
    if w.op == "ln":
        return 2 * t + 2 * n * es + (2 * rows * 4 if stats else 0)
    if w.op == "rms":
        return 2 * t + n * es + (rows * 4 if stats else 0)
    if w.op == "add_rms":
        return 4 * t + n * es + (rows * 4 if stats else 0)
    if w.op == "softmax":  # x, y (the timed call writes no statistics)
        return 2 * t
    raise ValueError(w.op)


# ---------------------------------------------------------------------------
# clocks (NVML through ctypes; reported as unavailable when NVML cannot be loaded)
# ---------------------------------------------------------------------------
REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
           0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
           0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
           0x100: "display_clock_setting"}


class ClockSampler:
    def __init__(self, device_index: int, period_s: float = 0.005):
        self.period = period_s
        self.samples = []  # (t, sm_mhz, reasons_mask)
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._nvml = None
        self._handle = None
        try:
            nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if nvml.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            props = torch.cuda.get_device_properties(device_index)
            bus = "%08x:%02x:%02x.0" % (props.pci_domain_id, props.pci_bus_id,
                                        props.pci_device_id)
            h = ctypes.c_void_p()
            if nvml.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
                raise OSError("no NVML handle for " + bus)
            mx = ctypes.c_uint()
            if nvml.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self._nvml, self._handle = nvml, h
        except OSError:
            self._nvml = None

    def _poll(self):
        nvml, h = self._nvml, self._handle
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        get_reasons = getattr(nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(nvml, "nvmlDeviceGetCurrentClocksThrottleReasons")
        while not self._stop.is_set():
            ok = nvml.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0
            ok = ok and get_reasons(h, ctypes.byref(rs)) == 0
            if ok:
                self.samples.append((time.perf_counter(), clk.value, rs.value))
            time.sleep(self.period)

    def start(self):
        if self._nvml is None:
            return
        self._stop.clear()
        self._thread = threading.Thread(target=self._poll, daemon=True)
        self._thread.start()

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join()

    def summary(self, t0=None, t1=None):
        if self._nvml is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "source": "unavailable"}
        s = [x for x in self.samples if (t0 is None or x[0] >= t0) and (t1 is None or x[0] <= t1)]
        window = "timed"
        if len(s) < 3:
            s, window = self.samples, "warmup+timed"
        mask = 0
        for _, _, r in s:
            mask |= r
        reasons = [name for bit, name in REASONS.items() if mask & bit and bit != 0x1]
        return {"sm_mhz": statistics.median([c for _, c, _ in s]) if s else None,
                "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(s),
                "window": window, "source": "nvml"}


# ---------------------------------------------------------------------------
# ncu traffic record (profiles/ncu_traffic.json), valid only for unchanged kernels
# ---------------------------------------------------------------------------
# The sources the row kernels (and their plan choice) are built from: a
# traffic record stays valid while none of them changes.
ROW_KERNEL_SOURCES = ("api.cpp", "nrm_device.cuh", "nrm_internal.h", "row_kernels.cuh",
                      "row_pipe.cuh")  # and every rows_*.cu instance file


def csrc_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "row_wise_normalization_reduce_gb300", "csrc")
    inst = sorted(f for f in os.listdir(csrc) if f.startswith("rows_") and f.endswith(".cu"))
    for name in ROW_KERNEL_SOURCES + tuple(inst):
        h.update(name.encode())
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        rec = json.load(open(path)).get(workload)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("csrc_hash") != csrc_hash():
        return None
    return rec.get("dram_bytes_per_launch")


def measured_peak():
    try:
        p = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        return float(p["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
# BatchNorm calls report their plan with the row-plan codes (include/nrm.h,
# nrm_last_plan); name them by what they run.
_BN_PLAN_NAMES = {
    "bn": {"tma": "cluster", "cta": "stream", "generic": "scalar", "persist": "flow"},
    "bn_bwd": {"cta": "stream", "generic": "scalar", "persist": "flow"},
    "bn_infer": {"cta": "flat", "generic": "scalar"},
}


def plan_name(op, kind_name):
    return _BN_PLAN_NAMES.get(op, {}).get(kind_name, kind_name)


class Step:
    """One call of the hot path on rotating, pre-filled device buffers."""

    max_sets = 0  # cap on the rotating input sets (profiling runs), 0: none

    def __init__(self, w: W.Workload, device, l2_bytes: int, hot: bool = False):
        import row_wise_normalization_reduce_gb300 as nrm
        self.nrm = nrm
        self.w = w
        inp = W.make_inputs(w)
        per_set = algorithmic_bytes(w)
        # cold: rotating input sets totalling > 3x L2; hot: one set, reused
        self.nsets = 1 if hot else max(2, int(np.ceil(3 * l2_bytes / per_set)) + 1)
        if Step.max_sets:
            self.nsets = min(self.nsets, Step.max_sets)
        dev = lambda t: t.to(device)  # noqa: E731
        self.params = {k: dev(v) for k, v in inp.items() if k not in ("x", "residual", "dy")}
        self.sets = []
        for i in range(self.nsets):
            s = {"x": dev(inp["x"])}
            if w.op == "add_rms":
                s["residual"] = dev(inp["residual"])
                s["residual_out"] = torch.empty_like(s["x"])
            if w.op == "bn_bwd":
                s["dy"] = dev(inp["dy"])
            s["y"] = torch.empty_like(s["x"])
            rows = inp["x"].shape[0]
            if w.op.startswith("bn"):
                c = w.shape[1]
                s["save_mean"] = torch.empty(c, device=device)
                s["save_rstd"] = torch.empty(c, device=device)
                s["dgamma"] = torch.empty(c, device=device)
                s["dbeta"] = torch.empty(c, device=device)
                s["ws"] = torch.empty(nrm.bn_fwd_train_workspace_size(w.shape[0], c, int(
                    np.prod(w.shape[2:]))), device=device, dtype=torch.uint8)
            else:
                s["rstd"] = torch.empty(rows, device=device)
                if w.op == "ln":
                    s["mean"] = torch.empty(rows, device=device)
            self.sets.append(s)
        self.i = 0
        self.host_inputs = inp
        # kernels per call: one, except the two-stage BatchNorm plans
        self.run(self.sets[0])
        torch.cuda.synchronize()
        kind = nrm.last_plan()[0]
        self.plan = plan_name(w.op, nrm.PLAN_NAMES.get(kind))
        self.launches_per_step = 1
        if w.op in ("bn", "bn_bwd") and kind in (nrm.PLAN_CTA, nrm.PLAN_GENERIC, nrm.PLAN_PERSIST):
            self.launches_per_step = 2

    def __call__(self):
        s = self.sets[self.i % self.nsets]
        self.i += 1
        self.run(s)

    def run(self, s):
        nrm, w, p = self.nrm, self.w, self.params
        if w.op == "add_rms":
            nrm.add_rms_fwd(s["x"], s["residual"], p["w"], w.eps, residual_out=s["residual_out"],
                            out=s["y"], rstd=s["rstd"])
        elif w.op == "ln":
            nrm.ln_fwd(s["x"], p["gamma"], p["beta"], w.eps, out=s["y"], mean=s["mean"],
                       rstd=s["rstd"])
        elif w.op == "rms":
            nrm.rms_fwd(s["x"], p["w"], w.eps, out=s["y"], rstd=s["rstd"])
        elif w.op == "softmax":
            nrm.softmax_fwd(s["x"], out=s["y"])
        elif w.op == "bn":
            nrm.bn_fwd_train(s["x"], p["gamma"], p["beta"], p["running_mean"], p["running_var"],
                             w.eps, w.momentum, out=s["y"], save_mean=s["save_mean"],
                             save_rstd=s["save_rstd"], workspace=s["ws"])
        elif w.op == "bn_infer":
            nrm.bn_fwd_infer(s["x"], p["running_mean"], p["running_var"], p["gamma"], p["beta"],
                             w.eps, out=s["y"])
        else:
            nrm.bn_bwd(s["dy"], s["x"], p["save_mean"], p["save_rstd"], p["gamma"], out=s["y"],
                       dgamma=s["dgamma"], dbeta=s["dbeta"], workspace=s["ws"])


def capture(step: Step, n: int, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(n):
            step()
    return g


def time_graphs(step: Step, k: int, warmup: int, stream, chunk=1000, dist=None):
    """Replay exactly k steps from CUDA graphs; return (seconds, t0, t1)."""
    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    full, rem = divmod(k, chunk)
    g_full = capture(step, chunk, stream) if full else None
    g_rem = capture(step, rem, stream) if rem else None
    g_warm = capture(step, max(warmup, 1), stream)
    torch.cuda.synchronize()
    g_warm.replay()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        # a bounded spin kernel (about 0.1 ms) before ev0, outside the timed
        # region: the graphs are queued before the GPU reaches ev0, so the
        # host's launch latency does not fall between the events
        torch.cuda._sleep(200_000)
        ev0.record(stream)
        for _ in range(full):
            g_full.replay()
        if g_rem is not None:
            g_rem.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    t1 = time.perf_counter()
    if dist is not None:
        dist.barrier()
    return ev0.elapsed_time(ev1) / 1e3, t0, t1


# ---------------------------------------------------------------------------
# per-call timings of one workload (the isolated-call protocol with an L2
# scrub before each call, hot back-to-back calls, and a drained variant of the
# graph replay)
# ---------------------------------------------------------------------------
def _cudart():
    """The CUDA runtime torch already loaded (for cudaMemsetAsync), or None."""
    for name in ("libcudart.so.13", "libcudart.so.12", "libcudart.so"):
        try:
            rt = ctypes.CDLL(name)
            rt.cudaMemsetAsync.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t,
                                           ctypes.c_void_p]
            rt.cudaMemsetAsync.restype = ctypes.c_int
            return rt
        except (OSError, AttributeError):
            continue
    return None


class Scrub:
    """Evicts L2 between calls.  write(): cudaMemsetAsync of 4x L2 bytes on
    the stream (the call then starts with L2 full of dirty lines it must
    write back as it evicts them); read(): a reduction that reads 4x L2 bytes
    (L2 is left holding clean lines only, as after a flush and invalidate)."""

    def __init__(self, device, l2_bytes, stream):
        self.nbytes = 4 * l2_bytes
        self.buf = torch.empty(self.nbytes // 4, dtype=torch.float32, device=device)
        self.buf.zero_()
        self.out = torch.empty((), dtype=torch.float32, device=device)
        self.stream = stream
        self.rt = _cudart()
        self.how = "cudaMemsetAsync" if self.rt is not None else "torch fill (no cudart handle)"

    def write(self):
        if self.rt is not None:
            st = self.rt.cudaMemsetAsync(ctypes.c_void_p(self.buf.data_ptr()), 0, self.nbytes,
                                         ctypes.c_void_p(self.stream.cuda_stream))
            if st != 0:
                raise RuntimeError(f"cudaMemsetAsync failed ({st})")
        else:
            self.buf.fill_(0.0)

    def read(self):
        torch.sum(self.buf, dim=0, out=self.out)


def time_isolated(step, stream, scrub, warm=50, timed=50, reps=5):
    """Section 8(d)'s isolated-call protocol: before every call the L2 is
    scrubbed (outside the events); CUDA events bracket the call alone.
    Median over `timed` calls, median of `reps` repeats; seconds."""
    meds = []
    with torch.cuda.stream(stream):
        for _ in range(reps):
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(timed)]
            # a head start for the GPU (a bounded spin kernel of about 30 ms):
            # every call below is queued before the GPU reaches it, so no
            # host launch gap falls between an event pair
            torch.cuda._sleep(60_000_000)
            for i in range(warm + timed):
                scrub()
                if i >= warm:
                    evs[i - warm][0].record(stream)
                step()
                if i >= warm:
                    evs[i - warm][1].record(stream)
            torch.cuda.synchronize()
            meds.append(statistics.median(a.elapsed_time(b) for a, b in evs) / 1e3)
    return statistics.median(meds)


def time_drained(step, stream, scrub, k=200, reps=5):
    """The graph replay with the write-back of every call inside the timed
    region: L2 is emptied of dirty lines before ev0 (a read scrub), and a read
    scrub after the k calls, before ev1, writes back what the last calls left
    in L2; the time of the same read scrub on a clean L2 is subtracted.
    Median of `reps`; seconds per call."""
    g = capture(step, k, stream)
    out = []
    with torch.cuda.stream(stream):
        for _ in range(reps):
            e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            scrub.read()
            e[0].record(stream)
            scrub.read()          # on a clean L2: the scrub's own time
            e[1].record(stream)
            scrub.read()
            e[2].record(stream)
            g.replay()
            scrub.read()          # writes back the calls' last dirty lines
            e[3].record(stream)
            torch.cuda.synchronize()
            out.append((e[2].elapsed_time(e[3]) - e[0].elapsed_time(e[1])) / 1e3 / k)
    return statistics.median(out)


def target_line(w: W.Workload, device, stream, l2, peak):
    """Every timing of one target workload (graph replay cold and hot,
    isolated calls after a write or a read scrub, drained replay)."""
    b = algorithmic_bytes(w)
    cold = Step(w, device, l2)
    t_graph, _, _ = time_graphs(cold, 2000, 20, stream)
    t_graph /= 2000
    scrub = Scrub(device, l2, stream)
    t_iso_w = time_isolated(cold, stream, scrub.write)
    t_iso_r = time_isolated(cold, stream, scrub.read)
    t_drain = time_drained(cold, stream, scrub)
    plan = cold.plan
    del cold
    torch.cuda.empty_cache()
    hot = Step(w, device, l2, hot=True)
    t_hot, _, _ = time_graphs(hot, 2000, 20, stream)
    t_hot /= 2000
    del hot, scrub
    torch.cuda.empty_cache()

    def entry(t):
        return {"us": round(t * 1e6, 3), "frac": round(b / t / 1e9 / peak, 4),
                "frac8": round(b / t / 1e9 / 8000.0, 4)}

    return {"bytes": b, "plan": plan,
            "graph_cold": entry(t_graph), "graph_hot": entry(t_hot),
            "isolated_cold_memset": entry(t_iso_w), "isolated_cold_clean": entry(t_iso_r),
            "graph_cold_drained": entry(t_drain)}


def time_e2e(w: W.Workload, device, steps: int):
    """Through the public API with host buffers (pinned): per step the step's
    inputs go host -> device and its outputs device -> host inside the timed
    region.  add+RMSNorm uses the C-ABI host entry point add_rms_fwd_host
    (chunked copies overlapped with the kernels); the other operators copy,
    call and copy back on one stream."""
    import row_wise_normalization_reduce_gb300 as nrm
    inp = W.make_inputs(w)
    host = {k: v.pin_memory() for k, v in inp.items()}
    dev = {k: torch.empty_like(v, device=device) for k, v in inp.items()}
    params = [k for k in dev if k not in ("x", "residual")]
    for k in params:
        dev[k].copy_(host[k])
    if w.op == "add_rms":
        outs = {"residual_out": torch.empty_like(dev["x"]), "y": torch.empty_like(dev["x"])}
    else:
        outs = {"y": torch.empty_like(dev["x"])}
    host_out = {k: torch.empty_like(v, device="cpu").pin_memory() for k, v in outs.items()}
    in_keys = ["x"] + (["residual"] if w.op == "add_rms" else [])
    h2d = sum(host[k].numel() * host[k].element_size() for k in in_keys)
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())
    stream = torch.cuda.current_stream(device)

    if w.op == "add_rms":
        # the library's host-memory entry point: chunked copies in both
        # directions overlapped with the kernels, through the C ABI
        ws = nrm.add_rms_fwd_host_workspace(w.shape[1], w.torch_dtype, device)

        def one():
            nrm.add_rms_fwd_host(host["x"], host["residual"], dev["w"], w.eps,
                                 residual_out=host_out["residual_out"], out=host_out["y"],
                                 workspace=ws, synchronize=False)
    else:
        one = None

    def one_device():
        for k in in_keys:
            dev[k].copy_(host[k], non_blocking=True)
        if w.op == "add_rms":
            nrm.add_rms_fwd(dev["x"], dev["residual"], dev["w"], w.eps,
                            residual_out=outs["residual_out"], out=outs["y"])
        elif w.op == "ln":
            nrm.ln_fwd(dev["x"], dev["gamma"], dev["beta"], w.eps, out=outs["y"],
                       want_stats=False)
        elif w.op == "rms":
            nrm.rms_fwd(dev["x"], dev["w"], w.eps, out=outs["y"])
        for k, v in outs.items():
            host_out[k].copy_(v, non_blocking=True)

    if one is None:
        one = one_device
    for _ in range(3):
        one()
    torch.cuda.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(steps):
        one()
    ev1.record(stream)
    torch.cuda.synchronize()
    sec = ev0.elapsed_time(ev1) / 1e3 / steps
    return sec, h2d, d2h


def l2_size(device_index) -> int:
    try:
        return int(torch.cuda.get_device_properties(device_index).L2_cache_size)
    except AttributeError:
        return 126 * 1024 * 1024


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------
def oracle_time(w: W.Workload, rows_sample: int, reps: int, threads: int):
    """Time the CPU oracle on the first rows_sample rows of the workload,
    partitioned by rows over `threads` threads (the oracle code itself unchanged).
    Returns (seconds per rep, bytes per rep)."""
    import concurrent.futures as cf
    import oracle
    orc = oracle.default()
    inp = W.make_inputs(w)
    to_np = (lambda t: t.numpy() if t.dtype == torch.float32
             else t.view(torch.int16).numpy().view(np.uint16))
    dt = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}[w.torch_dtype]
    x = to_np(inp["x"][:rows_sample].contiguous())
    rows = x.shape[0]
    res = to_np(inp["residual"][:rows_sample].contiguous()) if w.op == "add_rms" else None
    prm = {k: to_np(v) for k, v in inp.items() if k not in ("x", "residual")}
    if w.op == "bn":
        # BatchNorm: channels are independent, so they are split over the
        # threads (each thread's channels copied out before the timed region)
        chans = np.array_split(np.arange(x.shape[1]), threads)
        parts = [(np.ascontiguousarray(x[:, c]), c) for c in chans if len(c)]
        f64 = lambda v: v.astype(np.float64)  # noqa: E731

        def work_bn(part):
            xc, c = part
            orc.batchnorm_train(dt, xc, prm["gamma"][c], prm["beta"][c],
                                f64(prm["running_mean"][c]), f64(prm["running_var"][c]),
                                eps=w.eps, momentum=w.momentum)

        with cf.ThreadPoolExecutor(threads) as ex:
            list(ex.map(work_bn, parts))  # warm-up
            times = []
            for _ in range(reps):
                t0 = time.perf_counter()
                list(ex.map(work_bn, parts))
                times.append(time.perf_counter() - t0)
        return statistics.median(times), algorithmic_bytes(w) * rows / w.shape[0]
    chunks = np.array_split(np.arange(rows), threads)

    def work(idx):
        if len(idx) == 0:
            return
        a, b = idx[0], idx[-1] + 1
        if w.op == "add_rms":
            orc.add_rmsnorm(dt, x[a:b], res[a:b], prm["w"], eps=w.eps)
        elif w.op == "ln":
            orc.layernorm(dt, x[a:b], prm["gamma"], prm["beta"], eps=w.eps)
        elif w.op == "rms":
            orc.rmsnorm(dt, x[a:b], prm["w"], eps=w.eps)

    with cf.ThreadPoolExecutor(threads) as ex:
        list(ex.map(work, chunks))  # warm-up
        times = []
        for _ in range(reps):
            t0 = time.perf_counter()
            list(ex.map(work, chunks))
            times.append(time.perf_counter() - t0)
    frac = rows / w.shape[0]
    return statistics.median(times), algorithmic_bytes(w) * frac


# ---------------------------------------------------------------------------
# multi-rank aggregation (one process per GPU; replicas, weak scaling)
# ---------------------------------------------------------------------------
def max_over_ranks(seconds: float, dist=None, device="cpu") -> float:
    """The slowest rank's timed region (every rank gets the same value)."""
    if dist is None:
        return seconds
    t = torch.tensor([seconds], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(world: int, steps: int, bytes_per_step: int, seconds: float) -> float:
    """Whole-job throughput: the bytes every rank moved over the slowest rank's time."""
    return world * steps * bytes_per_step / seconds / 1e9


# ---------------------------------------------------------------------------
def emit(line: dict):
    print(json.dumps(line), flush=True)


def base_line(args, w, world):
    return {"metric": METRIC, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded torch.Generator)"}


def workload_config(w: W.Workload, world: int) -> dict:
    """The workload as both arms name it (identical dicts)."""
    return {"workload": w.name, "shape": list(w.shape), "dtype": w.dtype, "eps": w.eps,
            "parallelism": f"replicas x{world} (rows are independent)",
            "l2": "cold: rotating input sets totalling more than 3x L2, used round-robin"}


def run_reference(args, w, rank, world):
    if rank != 0:
        return
    threads = os.cpu_count() or 1
    # size each step so the whole run stays within about two minutes
    probe_rows = min(w.shape[0], threads)
    t_probe, _ = oracle_time(w, probe_rows, 1, threads)
    budget = 120.0 / (args.steps + args.warmup)
    rows = int(max(1, min(w.shape[0], probe_rows * budget / max(t_probe, 1e-9))))
    if args.warmup:
        oracle_time(w, rows, args.warmup, threads)
    sec, nbytes = oracle_time(w, rows, max(args.steps, 1), threads)
    gbs = nbytes / sec / 1e9
    line = base_line(args, w, world)
    line.update({
        "impl": "reference", "value": gbs, "ms_per_step": sec * 1e3,
        "config": workload_config(w, world),
        "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{rows} of {w.shape[0]} rows per step, fp64 oracle, "
                                   f"rows split over {threads} threads"},
        "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    })
    emit(line)


class StridedLnStep:
    """LayerNorm bf16 4096 x 4096 on a strided view: x is the first 4096
    columns of [4096, 4160] buffers (row stride 4160), y contiguous."""

    name = "ln_bf16_4096x4096_rowstride4160"

    def __init__(self, device, l2_bytes):
        import row_wise_normalization_reduce_gb300 as nrm
        self.nrm = nrm
        w = W.LN_BF16_4096x4096
        self.w = w
        inp = W.make_inputs(w)
        self.bytes = algorithmic_bytes(w, stats=False)
        self.nsets = max(2, int(np.ceil(3 * l2_bytes / self.bytes)) + 1)
        self.g, self.b = inp["gamma"].to(device), inp["beta"].to(device)
        self.sets = []
        for _ in range(self.nsets):
            buf = torch.zeros(4096, 4160, dtype=torch.bfloat16, device=device)
            buf[:, :4096].copy_(inp["x"].to(device))
            self.sets.append((buf[:, :4096], torch.empty(4096, 4096, dtype=torch.bfloat16,
                                                         device=device)))
        self.i = 0
        self()
        torch.cuda.synchronize()
        self.plan = nrm.PLAN_NAMES.get(nrm.last_plan()[0])
        self.launches_per_step = 1

    def __call__(self):
        x, y = self.sets[self.i % self.nsets]
        self.i += 1
        self.nrm.ln_fwd(x, self.g, self.b, self.w.eps, out=y, want_stats=False)


class SyncBnStep:
    """Synchronized BatchNorm training forward through its two library halves
    (partial statistics, then apply with the one part), binary32
    [32, 64, 56, 56]: the single-process cost of the exchange-ready path."""

    name = "sync_bn_train_f32_32x64x56x56_one_part"

    def __init__(self, device, l2_bytes):
        import row_wise_normalization_reduce_gb300 as nrm
        self.nrm = nrm
        w = W.BN_F32_32x64x56x56
        self.w = w
        inp = W.make_inputs(w)
        self.bytes = algorithmic_bytes(w)
        self.nsets = max(2, int(np.ceil(3 * l2_bytes / self.bytes)) + 1)
        self.g, self.b = inp["gamma"].to(device), inp["beta"].to(device)
        self.rm, self.rv = inp["running_mean"].to(device), inp["running_var"].to(device)
        self.sets = [(inp["x"].to(device), torch.empty(w.shape, device=device))
                     for _ in range(self.nsets)]
        c = w.shape[1]
        self.parts = torch.empty(1, c, 3, dtype=torch.float64, device=device)
        self.ws = torch.empty(nrm.bn_fwd_train_workspace_size(w.shape[0], c, int(np.prod(w.shape[2:]))),
                              dtype=torch.uint8, device=device)
        self.sm = torch.empty(c, device=device)
        self.sr = torch.empty(c, device=device)
        self.i = 0
        x, _ = self.sets[0]
        nrm.bn_fwd_partial_stats(x, out=self.parts[0], workspace=self.ws)
        torch.cuda.synchronize()
        # partial statistics in one cluster launch, else two (units and fold)
        one = nrm.last_plan()[0] == nrm.PLAN_TMA
        self()
        torch.cuda.synchronize()
        self.plan = ("cluster-stats" if one else "unit-stats+fold") + "+apply"
        self.launches_per_step = 2 if one else 3

    def __call__(self):
        x, y = self.sets[self.i % self.nsets]
        self.i += 1
        self.nrm.bn_fwd_partial_stats(x, out=self.parts[0], workspace=self.ws)
        self.nrm.bn_fwd_apply_stats(x, self.parts, self.g, self.b, self.rm, self.rv, self.w.eps,
                                    self.w.momentum, out=y, save_mean=self.sm, save_rstd=self.sr)


def secondary(args, device, stream, l2):
    steps = [(w, None) for w in (
        W.LN_BF16_4096x4096, W.RMS_F16_2048x4096, W.LN_BF16_1024x16384, W.BN_F32_32x64x56x56,
        W.LN_F32_64x1024, W.BN_INFER_F32_32x64x56x56, W.BN_BWD_F32_32x64x56x56,
        W.BN_F32_64x64x112x112, W.BN_BWD_F32_64x64x112x112, W.SOFTMAX_F32_128x4096,
        W.SOFTMAX_BF16_4096x4096, W.BN_BF16_32x64x56x56, W.BN_BF16_64x64x112x112)]
    steps += [(None, StridedLnStep), (None, SyncBnStep)]
    out = []
    for w, cls in steps:
        if w is not None:
            st = Step(w, device, l2)
            name, b = w.name, algorithmic_bytes(w)
        else:
            st = cls(device, l2)
            name, b = st.name, st.bytes
        k = 2000
        sec, _, _ = time_graphs(st, k, 20, stream)
        per = sec / k
        peak, _ = measured_peak()
        # compact keys: us per call, fraction of the measured peak and of 8 TB/s
        out.append({"w": name, "us": round(per * 1e6, 3),
                    "frac": round(b / per / 1e9 / peak, 4),
                    "frac8": round(b / per / 1e9 / 8000.0, 4), "plan": st.plan,
                    "launches": st.launches_per_step})
        del st
        torch.cuda.empty_cache()
    return out


def baseline_table(device, stream, l2):
    """One JSON line per workload of the measured table: graph replay cold and
    hot, isolated calls after a memset or read scrub, and the oracle on one
    and on all host cores (the full workload, median of 3)."""
    peak, _ = measured_peak()
    cores = os.cpu_count() or 1
    for w in (W.LN_F32_64x1024, W.RMS_F16_2048x4096, W.ADD_RMS_BF16_4096x4096,
              W.LN_BF16_1024x16384, W.LN_BF16_4096x4096, W.BN_F32_32x64x56x56):
        b = algorithmic_bytes(w)
        cold = Step(w, device, l2)
        t_cold = time_graphs(cold, 2000, 20, stream)[0] / 2000
        scrub = Scrub(device, l2, stream)
        t_iso_w = time_isolated(cold, stream, scrub.write)
        t_iso_r = time_isolated(cold, stream, scrub.read)
        plan = cold.plan
        del cold
        hot = Step(w, device, l2, hot=True)
        t_hot = time_graphs(hot, 2000, 20, stream)[0] / 2000
        del hot, scrub
        torch.cuda.empty_cache()
        c1, _ = oracle_time(w, w.shape[0], 3, 1)
        cn, _ = oracle_time(w, w.shape[0], 3, cores)
        emit({"w": w.name, "bytes": b, "plan": plan, "graph_cold_us": t_cold * 1e6,
              "graph_hot_us": t_hot * 1e6, "isolated_memset_us": t_iso_w * 1e6,
              "isolated_clean_us": t_iso_r * 1e6, "gbs_graph_cold": b / t_cold / 1e9,
              "frac_measured": b / t_cold / 1e9 / peak, "frac_8tbs": b / t_cold / 8e12,
              "oracle_1core_ms": c1 * 1e3, "oracle_allcore_ms": cn * 1e3, "cores": cores})


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="nrm", choices=["nrm", "reference"])
    ap.add_argument("--workload", default=W.ADD_RMS_BF16_4096x4096.name, choices=list(W.BY_NAME))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--sets", type=int, default=0,
                    help="at most this many rotating input sets (for small profiling runs; "
                         "the default keeps them above 3x L2)")
    ap.add_argument("--baseline-table", action="store_true",
                    help="print the measured table of the six workloads (per-call timings, "
                         "oracle on one and on all cores) instead of the bench line")
    ap.add_argument("--no-targets", action="store_true",
                    help="skip the per-call timings of the two 4096x4096 bf16 targets")
    ap.add_argument("--plan", default="auto",
                    help="row-operator plan: auto, generic:T, warp:T:P, cta:T:P or "
                         "tma:T:P:STAGES:GROUPS (for measurements and profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    Step.max_sets = max(0, args.sets)

    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local = int(os.environ.get("LOCAL_RANK", 0))
    w = W.BY_NAME[args.workload]

    if args.impl == "reference":
        run_reference(args, w, rank, world)
        return

    dist = None
    if world > 1:
        import torch.distributed as tdist
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl", device_id=torch.device("cuda", local))
        dist = tdist
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    import row_wise_normalization_reduce_gb300 as nrm
    nrm.lib()
    if args.plan != "auto":
        kind, *nums = args.plan.split(":")
        code = {v: k for k, v in nrm.PLAN_NAMES.items()}[kind]
        nrm.force_plan(code, *[int(v) for v in nums])
    stream = torch.cuda.Stream(device)
    l2 = l2_size(local)
    if args.baseline_table:
        baseline_table(device, stream, l2)
        return

    step = Step(w, device, l2)
    sampler = ClockSampler(local)
    sampler.start()
    sec, t0, t1 = time_graphs(step, args.steps, args.warmup, stream, dist=dist)
    sampler.stop()
    sec = max_over_ranks(sec, dist, device)
    per_step = sec / args.steps
    nbytes = algorithmic_bytes(w)
    value = job_gbs(world, args.steps, nbytes, sec)
    peak, peak_src = measured_peak()
    kernel_gbs = nbytes / (per_step / step.launches_per_step) / 1e9 if step.launches_per_step == 1 \
        else nbytes / per_step / 1e9
    traffic = ncu_traffic(w.name)

    e2e = None
    if not args.no_e2e and not w.op.startswith("bn"):
        es, h2d, d2h = time_e2e(w, device, 20)
        e2e = {"value": world * nbytes / es / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": es * 1e3,
               "path": ("add_rms_fwd_host (C ABI, pinned host buffers, chunked copies "
                        "overlapped with the kernels)") if w.op == "add_rms" else
                       "H2D copy, device call, D2H copy on one stream"}

    sec_lines = None
    if rank == 0 and not args.no_secondary:
        sec_lines = secondary(args, device, stream, l2)

    targets = None
    if rank == 0 and not args.no_targets:
        peak, _ = measured_peak()
        tsampler = ClockSampler(local, period_s=0.02)
        tsampler.start()
        targets = {t.name: target_line(t, device, stream, l2, peak)
                   for t in (W.ADD_RMS_BF16_4096x4096, W.LN_BF16_4096x4096)}
        tsampler.stop()
        ts = tsampler.summary()
        targets["clocks"] = {"sm_mhz": ts["sm_mhz"], "reasons": ts["reasons"]}
        targets["how"] = ("graph_*: K calls replayed from a CUDA graph, per call (cold: rotating "
                          "sets > 3x L2; hot: one set); isolated_*: events around one call after "
                          "a 4x L2 scrub, median of 50, median of 5 repeats (memset: the scrub "
                          "writes, so the call first writes back dirty lines; clean: the scrub "
                          "reads); drained: graph replay plus the write-back of the last calls' "
                          "dirty lines; frac of the measured peak, frac8 of 8 TB/s")

    cpu = None
    if rank == 0 and not args.no_cpu_baseline and not w.op.startswith("bn"):
        rows = w.shape[0]
        cs, cb = oracle_time(w, rows, 3, 1)
        cpu = {"value": cb / cs / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "us_per_call": cs * 1e6,
               "sample": f"the full {rows}-row workload, fp64 oracle, one thread, "
                         f"median of 3 after 1 warm-up"}

    if rank == 0:
        line = base_line(args, w, world)
        line.update({
            "value": value, "ms_per_step": per_step * 1e3, "us_per_call": per_step * 1e6,
            "config": workload_config(w, world),
            "timing": (f"CUDA graphs replaying exactly K calls between CUDA events (a spin "
                       f"kernel queued before the first keeps host launch latency out); "
                       f"{step.nsets} rotating input sets ({step.nsets * nbytes / 1e6:.0f} MB) "
                       f"> L2 ({l2 / 1e6:.0f} MB)"),
            "roofline": {"bound": "hbm", "achieved": kernel_gbs, "peak": peak, "unit": "GB/s",
                         "frac": kernel_gbs / peak, "peak_source": peak_src,
                         "frac_of_nominal_8tbs": kernel_gbs / 8000.0,
                         "algorithmic_bytes_per_launch": nbytes, "traffic": traffic},
            "gpu_launches": args.steps * step.launches_per_step,
            "clocks": sampler.summary(t0, t1),
            "plan": step.plan,
        })
        if e2e is not None:
            line["e2e"] = e2e
        if cpu is not None:
            line["cpu_baseline"] = cpu
        if sec_lines is not None:
            line["secondary"] = sec_lines
        if targets is not None:
            line["targets"] = targets  # last, so the end of the line carries both targets
        emit(line)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
