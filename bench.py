#!/usr/bin/env python3
"""Benchmark of the streaming block-causal hot path on one B300 per rank.

One step = one 160 ms streaming unit: append the unit's K/V slice to the
full-history cache, block-causal attention of the unit's queries against the
whole cache, then the flow-matching Euler steps over the unit's latents --
every call through the C ABI (``streaming_block_causal_flash_b300.ws``).

Prints ONE JSON line (rank 0).  ``value`` is the attention's algorithmic
TFLOP/s over the whole step (4*D*H*sum_i e(i) per unit / step time) summed
over ranks; ``ms_per_step`` is the time of one unit.  See ``--help``.

  python bench.py [--gpus N --steps K --warmup W --workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle, timed on host cores
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from streaming_block_causal_flash_b300.inputs import WORKLOADS, Workload  # noqa: E402

METRIC = "block-causal attn TFLOP/s & µs per 160ms streaming unit (1 B300, vs roofline)"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "unit_640x368"
L2_BYTES = 126 * 1024 * 1024
ATTN_SOURCE = os.path.join(ROOT, "streaming_block_causal_flash_b300", "csrc", "attn_tcgen05.cu")
PROFILES_DIR = os.path.join(ROOT, "profiles")


def traffic_file(workload: str) -> str:
    """The committed ncu summary of one attention launch's DRAM bytes for a workload."""
    return os.path.join(PROFILES_DIR, f"attn_tcgen05_{workload}_traffic.txt")


# ----------------------------------------------------------------- plumbing

def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=[k for k, w in WORKLOADS.items() if w.dtype == "bf16"])
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer measurement")
    ap.add_argument("--no-hbm", action="store_true", help="skip the append/Euler HBM measurement")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="skip the brief measurements of the other workloads (and the full oracle timings)")
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int, device=None):
    if world > 1:
        if device is not None and torch.distributed.get_backend() == "nccl":
            torch.distributed.barrier(device_ids=[device.index])
        else:
            torch.distributed.barrier()


def reduce_over_ranks(local_ms: float, local_flops: float, world: int, device="cpu"):
    """(max step time over ranks, total work over ranks)."""
    if world == 1:
        return local_ms, local_flops
    t = torch.tensor([local_ms], dtype=torch.float64, device=device)
    w = torch.tensor([local_flops], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    torch.distributed.all_reduce(w, op=torch.distributed.ReduceOp.SUM)
    return float(t.item()), float(w.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
            "source": "fallback"}


class _CtypesNvml:
    """The few read-only NVML queries the clock sampler makes, called through
    ctypes on the driver's libnvidia-ml.so.1 (for hosts without the pynvml
    package).  Names and reason bits follow NVML's public header."""

    NVML_CLOCK_SM = 1
    nvmlClocksEventReasonSwPowerCap = 0x4
    nvmlClocksEventReasonHwSlowdown = 0x8
    nvmlClocksEventReasonSwThermalSlowdown = 0x20
    nvmlClocksEventReasonHwThermalSlowdown = 0x40

    def __init__(self):
        import ctypes
        self._c = ctypes
        self._lib = ctypes.CDLL("libnvidia-ml.so.1")

    def _call(self, name, *args):
        rc = getattr(self._lib, name)(*args)
        if rc != 0:
            raise RuntimeError(f"{name} returned NVML error {rc}")

    def nvmlInit(self):
        self._call("nvmlInit_v2")

    def nvmlDeviceGetHandleByPciBusId(self, bus):
        h = self._c.c_void_p()
        self._call("nvmlDeviceGetHandleByPciBusId_v2", self._c.c_char_p(bus.encode()), self._c.byref(h))
        return h

    def nvmlDeviceGetHandleByIndex(self, i):
        h = self._c.c_void_p()
        self._call("nvmlDeviceGetHandleByIndex_v2", self._c.c_uint(i), self._c.byref(h))
        return h

    def _uint(self, name, h, *extra):
        v = self._c.c_uint()
        self._call(name, h, *extra, self._c.byref(v))
        return v.value

    def nvmlDeviceGetClockInfo(self, h, kind):
        return self._uint("nvmlDeviceGetClockInfo", h, self._c.c_int(kind))

    def nvmlDeviceGetMaxClockInfo(self, h, kind):
        return self._uint("nvmlDeviceGetMaxClockInfo", h, self._c.c_int(kind))

    def nvmlDeviceGetPowerUsage(self, h):
        return self._uint("nvmlDeviceGetPowerUsage", h)

    def nvmlDeviceGetCurrentClocksEventReasons(self, h):
        v = self._c.c_ulonglong()
        fn = "nvmlDeviceGetCurrentClocksEventReasons"
        if not hasattr(self._lib, fn):
            fn = "nvmlDeviceGetCurrentClocksThrottleReasons"
        self._call(fn, h, self._c.byref(v))
        return v.value

    nvmlDeviceGetCurrentClocksThrottleReasons = nvmlDeviceGetCurrentClocksEventReasons


class ClockSampler:
    """SM clock and clock-event (throttle) reasons of the GPU while it works.

    A thread polls NVML every 2 ms from start() to stop(); start() also takes
    one snapshot at once and stop() one more, so even a timed region of a few
    milliseconds carries samples.  The host thread that launched the work is
    then blocked in a device synchronisation (the GIL is free), which is when
    the samples are taken.  Falls back to an `nvidia-smi -lms` stream when
    NVML cannot be used."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = (("hw_slowdown", "nvmlClocksEventReasonHwSlowdown"),
               ("hw_thermal_slowdown", "nvmlClocksEventReasonHwThermalSlowdown"),
               ("sw_thermal_slowdown", "nvmlClocksEventReasonSwThermalSlowdown"),
               ("sw_power_cap", "nvmlClocksEventReasonSwPowerCap"))

    def __init__(self, gpu_index: int, period_s: float = 0.002):
        self.gpu = gpu_index
        self.period = period_s
        self.proc = None
        self.thread = None
        self.samples = []
        self.nvml = None
        self.handle = None

    def _nvml_handle(self):
        try:
            import pynvml
        except ImportError:
            pynvml = _CtypesNvml()
        pynvml.nvmlInit()
        try:
            p = torch.cuda.get_device_properties(self.gpu)
            bus = f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
            return pynvml, pynvml.nvmlDeviceGetHandleByPciBusId(bus)
        except Exception:
            return pynvml, pynvml.nvmlDeviceGetHandleByIndex(self.gpu)

    def _sample(self):
        nv, h = self.nvml, self.handle
        sm = nv.nvmlDeviceGetClockInfo(h, nv.NVML_CLOCK_SM)
        mx = nv.nvmlDeviceGetMaxClockInfo(h, nv.NVML_CLOCK_SM)
        try:
            mask = nv.nvmlDeviceGetCurrentClocksEventReasons(h)
        except Exception:
            mask = nv.nvmlDeviceGetCurrentClocksThrottleReasons(h)
        try:
            watts = nv.nvmlDeviceGetPowerUsage(h) / 1000.0
        except Exception:
            watts = None
        reasons = [name for name, attr in self.REASONS if mask & getattr(nv, attr, 0)]
        self.samples.append((float(sm), float(mx), reasons, watts))

    def start(self):
        import threading
        self.samples = []
        self.nvml_error = None
        try:
            self.nvml, self.handle = self._nvml_handle()
            self._sample()
        except Exception as e:     # noqa: BLE001 -- any NVML failure: use nvidia-smi
            self.nvml = None
            self.nvml_error = f"{type(e).__name__}: {e}"[:200]
        if self.nvml is not None:
            self.stop_flag = threading.Event()

            def loop():
                while not self.stop_flag.wait(self.period):
                    try:
                        self._sample()
                    except Exception:
                        break
            self.thread = threading.Thread(target=loop, daemon=True)
            self.thread.start()
            return
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.nvml is not None:
            self.stop_flag.set()
            self.thread.join(timeout=5)
            try:
                self._sample()
            except Exception:
                pass
            sms = [x[0] for x in self.samples]
            reasons = sorted({r for x in self.samples for r in x[2]})
            watts = [x[3] for x in self.samples if x[3] is not None]
            return {"sm_mhz": statistics.median(sms) if sms else None,
                    "sm_max_mhz": max(x[1] for x in self.samples) if self.samples else None,
                    "sm_mhz_min": min(sms) if sms else None,
                    "power_w_median": round(statistics.median(watts), 1) if watts else None,
                    "reasons": reasons, "samples": len(sms),
                    "source": f"NVML every {self.period * 1e3:.0f} ms plus snapshots at start and stop"}
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sms, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxes.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sms) if sms else None,
                "sm_max_mhz": max(maxes) if maxes else None,
                "reasons": sorted(reasons), "samples": len(sms), "source": "nvidia-smi -lms 100",
                "nvml_error": self.nvml_error}


def clock_normalised(ms: float, clk: dict):
    """ms x median SM MHz (thousands of SM cycles), to compare runs at different clocks."""
    if not clk or not clk.get("sm_mhz"):
        return None
    return round(ms * clk["sm_mhz"], 1)


def source_digest(path: str) -> str:
    """sha256[:16] of the kernel source's code: // comments, blank lines and
    trailing spaces removed, so that a comment edit keeps recorded counters."""
    code = []
    with open(path, encoding="utf-8") as f:
        for line in f:
            line = line.split("//", 1)[0].rstrip()
            if line:
                code.append(line)
    return hashlib.sha256("\n".join(code).encode()).hexdigest()[:16]


def recorded_traffic(workload: str = DEFAULT_WORKLOAD):
    """DRAM bytes per attention launch from the workload's committed ncu
    summary, or None when there is none or the kernel source changed since
    its counters were taken."""
    path = traffic_file(workload)
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if ":" in line:
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("kernel_source_sha256_16") != source_digest(ATTN_SOURCE):
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ----------------------------------------------------------- the workload

def attention_flops(offsets: np.ndarray, rows: np.ndarray, heads: int, head_dim: int) -> float:
    """4*D*H*sum_i e(i): QK^T and PV over the visible keys of each query row."""
    offs = np.asarray(offsets, dtype=np.int64)
    blk = np.searchsorted(offs, rows, side="right") - 1
    e = offs[blk + 1]
    return 4.0 * head_dim * heads * float(e.sum())


class UnitSession:
    """Device state for streaming units of one workload: the full-history
    cache (history units resident), and per-unit inputs."""

    def __init__(self, w: Workload, device, host_only=False):
        self.w = w
        self.sizes = w.unit_sizes()
        self.offsets_all = w.offsets()
        self.cap = w.capacity()
        H, D = w.heads, w.head_dim
        T_hist = int(self.offsets_all[w.history_units])
        k = torch.zeros(H, self.cap, D, dtype=torch.bfloat16)
        v = torch.zeros(H, self.cap, D, dtype=torch.bfloat16)
        for h in range(H):
            if w.history_units:
                k[h, :T_hist] = w.head_timeline("k", h, w.history_units, self.sizes)
                v[h, :T_hist] = w.head_timeline("v", h, w.history_units, self.sizes)
        self.k_host, self.v_host = k, v
        self.units = list(range(w.history_units, w.n_units))
        # per new unit: Q, KV slice, velocities, eps
        self.q_host = {u: w.token_major("q", u, self.sizes) for u in self.units}
        self.kv_host = {u: (w.token_major("k", u, self.sizes), w.token_major("v", u, self.sizes))
                        for u in self.units}
        self.vel_host = {u: [w.velocity_input(u, s) for s in range(w.euler_steps)] for u in self.units}
        self.eps_host = {u: w.eps(u) for u in self.units}
        if host_only:
            return
        self.device = device
        self.k = k.to(device)
        self.v = v.to(device)
        self.q = {u: t.to(device) for u, t in self.q_host.items()}
        self.kv = {u: (a.to(device), b.to(device)) for u, (a, b) in self.kv_host.items()}
        self.vel = {u: [t.to(device) for t in ts] for u, ts in self.vel_host.items()}
        self.z = {u: self.eps_host[u].to(device) for u in self.units}
        self.offs_dev = {u: torch.from_numpy(self.offsets_all[:u + 2].astype(np.int32)).to(device)
                         for u in self.units}
        q_max = max(self.sizes[u] for u in self.units)
        self.out = torch.empty(q_max, H, D, dtype=torch.bfloat16, device=device)
        from streaming_block_causal_flash_b300 import ws
        need = max(ws.ws_block_causal_attn_workspace_size(self.sizes[u], int(self.offsets_all[u + 1]), H, D)
                   for u in self.units)
        self.workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=device)
        self.split = need > 0

    def unit_flops(self, u: int) -> float:
        offs = self.offsets_all[:u + 2]
        rows = np.arange(int(offs[-2]), int(offs[-1]))
        return attention_flops(offs, rows, self.w.heads, self.w.head_dim)

    def launches_per_step(self) -> int:
        return 1 + 1 + (1 if self.split else 0) + self.w.euler_steps


def run_unit(sess: UnitSession, u: int, stream, ev=None):
    """append -> attention -> Euler steps for unit u, all on `stream`."""
    from streaming_block_causal_flash_b300 import ws
    w = sess.w
    n = sess.sizes[u]
    offs = sess.offsets_all[:u + 2]
    k_new, v_new = sess.kv[u]
    if ev is not None:
        ev[0].record(stream)
    ws.ws_kv_append(k_new, v_new, sess.k, sess.v, int(offs[-2]), stream=stream)
    if ev is not None:
        ev[1].record(stream)
    ws.ws_block_causal_attn(sess.q[u], sess.k, sess.v, sess.out[:n], offs, sess.offs_dev[u],
                            workspace=sess.workspace, stream=stream)
    if ev is not None:
        ev[2].record(stream)
    z = sess.z[u]
    for s in range(w.euler_steps):
        ws.ws_fm_euler_step(z, sess.vel[u][s], 1.0 / w.euler_steps, stream=stream)
    if ev is not None:
        ev[3].record(stream)


# ------------------------------------------------------------- native arm

def time_native(args, sess: UnitSession, device, world, clocks=None):
    stream = torch.cuda.current_stream(device)
    units = sess.units
    K, W = args.steps, args.warmup
    for i in range(W):
        run_unit(sess, units[i % len(units)], stream)
    torch.cuda.synchronize(device)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world, device)
    torch.cuda.synchronize(device)
    if clocks is not None:
        clocks.start()
    start.record(stream)
    flops = 0.0
    for i in range(K):
        u = units[i % len(units)]
        run_unit(sess, u, stream, evs[i])
        flops += sess.unit_flops(u)
    stop.record(stream)
    torch.cuda.synchronize(device)
    clk = clocks.stop() if clocks is not None else None
    barrier(world, device)
    total_ms = start.elapsed_time(stop)
    append_ms = [e[0].elapsed_time(e[1]) for e in evs]
    attn_ms = [e[1].elapsed_time(e[2]) for e in evs]
    euler_ms = [e[2].elapsed_time(e[3]) for e in evs]
    unit_ms = [e[0].elapsed_time(e[3]) for e in evs]
    return total_ms, flops, append_ms, attn_ms, euler_ms, unit_ms, clk


def time_e2e(args, sess: UnitSession, device):
    """Same step through the public API with host buffers: every step copies
    its inputs in from pinned host memory and reads its results (O and z)
    back, inside the timed region.

    Pipelined, as a streaming deployment runs it: two device buffer sets;
    the inputs of unit k+1 go up on one copy stream and the results of unit
    k-1 come back on another while unit k computes (buffer reuse guarded by
    CUDA events).  The plain serial figure (copy in, compute, copy out, one
    step after another) is reported beside it."""
    from streaming_block_causal_flash_b300 import ws
    compute = torch.cuda.current_stream(device)
    up, down = torch.cuda.Stream(device), torch.cuda.Stream(device)
    w = sess.w
    u = sess.units[0]
    n = sess.sizes[u]
    offs = sess.offsets_all[:u + 2]
    pin = lambda t: t.contiguous().pin_memory()  # noqa: E731
    h_in = [pin(sess.q_host[u]), pin(sess.kv_host[u][0]), pin(sess.kv_host[u][1]),
            pin(sess.eps_host[u])] + [pin(t) for t in sess.vel_host[u]]
    h_out = [(torch.empty(n, w.heads, w.head_dim, dtype=torch.bfloat16).pin_memory(),
              torch.empty_like(h_in[3]).pin_memory()) for _ in range(2)]
    d_in = [[torch.empty(t.shape, dtype=t.dtype, device=device) for t in h_in] for _ in range(2)]
    d_out = [torch.empty(n, w.heads, w.head_dim, dtype=torch.bfloat16, device=device) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in h_in)
    d2h = sum(t.numel() * t.element_size() for t in h_out[0])

    def compute_step(b, st):
        q, k, v, z, *vel = d_in[b]
        ws.ws_kv_append(k, v, sess.k, sess.v, int(offs[-2]), stream=st)
        ws.ws_block_causal_attn(q, sess.k, sess.v, d_out[b], offs, sess.offs_dev[u],
                                workspace=sess.workspace, stream=st)
        for s_ in range(w.euler_steps):
            ws.ws_fm_euler_step(z, vel[s_], 1.0 / w.euler_steps, stream=st)

    def serial_step():
        for d, h in zip(d_in[0], h_in):
            d.copy_(h, non_blocking=True)
        compute_step(0, compute)
        h_out[0][0].copy_(d_out[0], non_blocking=True)
        h_out[0][1].copy_(d_in[0][3], non_blocking=True)

    steps = max(10, min(args.steps, 100))
    for _ in range(3):
        serial_step()
    torch.cuda.synchronize(device)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(compute)
    for _ in range(steps):
        serial_step()
    b.record(compute)
    torch.cuda.synchronize(device)
    serial_ms = a.elapsed_time(b) / steps

    def pipelined(nsteps, timed):
        up_done = [torch.cuda.Event() for _ in range(nsteps)]
        comp_done = [torch.cuda.Event() for _ in range(nsteps)]
        down_done = [torch.cuda.Event() for _ in range(nsteps)]
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(compute)
        up.wait_event(start)

        def upload(i):
            with torch.cuda.stream(up):
                if i >= 2:
                    up.wait_event(down_done[i - 2])     # set i%2 free: read back, so computed
                for d, h in zip(d_in[i % 2], h_in):
                    d.copy_(h, non_blocking=True)
                up_done[i].record(up)

        upload(0)
        for i in range(nsteps):
            if i + 1 < nsteps:
                upload(i + 1)
            compute.wait_event(up_done[i])
            compute_step(i % 2, compute)
            comp_done[i].record(compute)
            with torch.cuda.stream(down):
                down.wait_event(comp_done[i])
                h_out[i % 2][0].copy_(d_out[i % 2], non_blocking=True)
                h_out[i % 2][1].copy_(d_in[i % 2][3], non_blocking=True)
                down_done[i].record(down)
        compute.wait_event(down_done[nsteps - 1])
        stop.record(compute)
        torch.cuda.synchronize(device)
        return start.elapsed_time(stop) / nsteps

    pipelined(4, False)
    ms = pipelined(steps, True)
    flops = sess.unit_flops(u)
    return {"value": round(flops / (ms * 1e-3) / 1e12, 3), "unit": UNIT,
            "ms_per_step": round(ms, 4), "steps": steps,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "method": "pipelined: inputs of unit k+1 uploaded and results of unit k-1 read back on "
                      "copy streams while unit k computes; every step moves its own inputs and results",
            "serial_ms_per_step": round(serial_ms, 4),
            "serial_value": round(flops / (serial_ms * 1e-3) / 1e12, 3)}


def graph_time_us(launch, reps: int, device) -> float:
    """Mean device time of one launch among `reps` back-to-back launches,
    captured once in a CUDA graph and replayed between two CUDA events (no
    host launch overhead, no event between kernels)."""
    launch(0, torch.cuda.current_stream(device))           # first call outside capture
    torch.cuda.synchronize(device)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(reps):
            launch(i, torch.cuda.current_stream(device))
    stream = torch.cuda.current_stream(device)
    g.replay()
    torch.cuda.synchronize(device)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    g.replay()
    b.record(stream)
    torch.cuda.synchronize(device)
    return a.elapsed_time(b) * 1e3 / reps


def time_hbm_kernels(sess: UnitSession, device, peaks):
    """Append and Euler alone, as back-to-back launches replayed from a CUDA
    graph, rotating buffer sets whose total is 3x larger than L2 so every
    launch streams from HBM."""
    from streaming_block_causal_flash_b300 import ws
    w = sess.w
    H, D = w.heads, w.head_dim
    u = sess.units[0]
    n = sess.sizes[u]
    slice_bytes = n * H * D * 2
    nsets = max(4, int(3 * L2_BYTES // (4 * slice_bytes)) + 1)
    ks = [torch.randn(n, H, D, device=device).to(torch.bfloat16) for _ in range(nsets)]
    vs = [torch.randn(n, H, D, device=device).to(torch.bfloat16) for _ in range(nsets)]
    cap_sets = max(1, sess.cap // n - 1)

    def append(i, st):
        ws.ws_kv_append(ks[i % nsets], vs[i % nsets], sess.k, sess.v, (i % cap_sets) * n, stream=st)

    us = graph_time_us(append, 8 * nsets, device)
    byts = 4.0 * slice_bytes
    out = {"append": {"us": round(us, 2), "bytes": int(byts), "gbs": round(byts / us / 1e3, 1),
                      "frac_hbm": round(byts / us / 1e3 / peaks["hbm_gbs"], 3)}}
    # The ceiling for one standalone launch that moves this many bytes: a
    # plain device-to-device copy (cudaMemcpyAsync) of the same 2 x slice
    # bytes (read once, written once), timed the same way.
    src = [torch.empty(2 * slice_bytes, dtype=torch.uint8, device=device) for _ in range(nsets)]
    dst = [torch.empty(2 * slice_bytes, dtype=torch.uint8, device=device) for _ in range(nsets)]

    def copy(i, st):
        with torch.cuda.stream(st):
            dst[(i + 1) % nsets].copy_(src[i % nsets], non_blocking=True)

    us_c = graph_time_us(copy, 8 * nsets, device)
    out["same_size_copy"] = {"us": round(us_c, 2), "bytes": int(byts), "gbs": round(byts / us_c / 1e3, 1),
                             "frac_hbm": round(byts / us_c / 1e3 / peaks["hbm_gbs"], 3),
                             "what": "one device-to-device cudaMemcpyAsync of the K+V slice bytes"}
    out["append"]["frac_of_same_size_copy"] = round(us_c / us, 3)
    del ks, vs, src, dst
    nl = w.latent_tokens * w.latent_channels
    per = nl * (4 + 2 + 4)
    zsets = max(4, int(3 * L2_BYTES // per) + 1)
    zs = [torch.randn(nl, device=device) for _ in range(zsets)]
    vls = [torch.randn(nl, device=device).to(torch.bfloat16) for _ in range(zsets)]

    def euler(i, st):
        ws.ws_fm_euler_step(zs[i % zsets], vls[i % zsets], 0.25, stream=st)

    us = graph_time_us(euler, 8 * zsets, device)
    out["euler"] = {"us": round(us, 2), "bytes": int(per), "gbs": round(per / us / 1e3, 1),
                    "frac_hbm": round(per / us / 1e3 / peaks["hbm_gbs"], 3)}
    vcs = [torch.randn(nl, device=device).to(torch.bfloat16) for _ in range(zsets)]

    def euler_cfg(i, st):
        ws.ws_fm_euler_cfg_step(zs[i % zsets], vls[i % zsets], vcs[(i + 1) % zsets], 3.0, 0.25, stream=st)

    us = graph_time_us(euler_cfg, 8 * zsets, device)
    per_cfg = nl * (4 + 2 + 2 + 4)
    out["euler_cfg"] = {"us": round(us, 2), "bytes": int(per_cfg), "gbs": round(per_cfg / us / 1e3, 1),
                        "frac_hbm": round(per_cfg / us / 1e3 / peaks["hbm_gbs"], 3)}
    out["method"] = (f"back-to-back launches replayed from a CUDA graph, mean per launch; rotating "
                     f"{nsets} (append) / {zsets} (Euler) buffer sets, 3x L2 in total; "
                     f"peak = {peaks['source']} HBM copy bandwidth")
    return out


def time_attn_side(sess: UnitSession, device, peaks, reps: int = 20):
    """ws_block_causal_attn_side for the unit (history from the cache, the
    unit's own K/V from its slice buffers), graph-replayed back to back."""
    from streaming_block_causal_flash_b300 import ws
    u = sess.units[0]
    n = sess.sizes[u]
    offs = sess.offsets_all[:u + 2]
    k_side, v_side = sess.kv[u]

    def call(i, st):
        ws.ws_block_causal_attn_side(sess.q[u], sess.k, sess.v, k_side, v_side, sess.out[:n], offs,
                                     sess.offs_dev[u], workspace=sess.workspace, stream=st)

    def plain(i, st):
        ws.ws_block_causal_attn(sess.q[u], sess.k, sess.v, sess.out[:n], offs, sess.offs_dev[u],
                                workspace=sess.workspace, stream=st)

    us_plain = graph_time_us(plain, reps, device)
    us = graph_time_us(call, reps, device)
    achieved = sess.unit_flops(u) / (us * 1e-6) / 1e12
    return {"us": round(us, 1), "achieved": round(achieved, 2), "unit": "TFLOP/s",
            "frac": round(achieved / peaks["bf16_tflops"], 4),
            "plain_call_us": round(us_plain, 1),
            "method": f"{reps} calls replayed from a CUDA graph; plain_call_us: ws_block_causal_attn "
                      f"timed the same way"}


def time_fused_unit(sess: UnitSession, device, reps: int = 20, rounds: int = 4,
                    rest_s: float = 0.5):
    """The unit step with the append fused into the attention (one
    ws_block_causal_attn_side call that reads the unit's K/V from its slice
    and commits them to the cache from shared memory; then the Euler steps)
    against the plain step (append, attention, Euler steps).  Both
    graph-replayed in alternation, the order swapped every round and the GPU
    left idle before each replay, so that neither always runs on the hotter
    GPU; the best round of each."""
    from streaming_block_causal_flash_b300 import ws
    u = sess.units[0]
    n = sess.sizes[u]
    offs = sess.offsets_all[:u + 2]
    k_side, v_side = sess.kv[u]

    def fused(i, st):
        ws.ws_block_causal_attn_side(sess.q[u], sess.k, sess.v, k_side, v_side, sess.out[:n], offs,
                                     sess.offs_dev[u], workspace=sess.workspace, commit=True, stream=st)
        for s_ in range(sess.w.euler_steps):
            ws.ws_fm_euler_step(sess.z[u], sess.vel[u][s_], 1.0 / sess.w.euler_steps, stream=st)

    def plain(i, st):
        run_unit(sess, u, st)

    best = {"plain": float("inf"), "fused": float("inf")}
    for r in range(rounds):
        for name in (("plain", "fused") if r % 2 == 0 else ("fused", "plain")):
            time.sleep(rest_s)
            best[name] = min(best[name], graph_time_us(plain if name == "plain" else fused, reps,
                                                       device))
    flops = sess.unit_flops(u)
    return {"fused_us_per_unit": round(best["fused"], 1), "plain_us_per_unit": round(best["plain"], 1),
            "fused_value": round(flops / (best["fused"] * 1e-6) / 1e12, 3), "unit": UNIT,
            "method": f"{reps} unit steps per CUDA graph, fused and plain replayed in alternation "
                      f"(order swapped each round, {rest_s} s idle before each), best of {rounds}"}


def time_unit_graph(sess: UnitSession, device, reps: int = 50):
    """The whole unit step (append, attention, Euler steps) captured once in a
    CUDA graph and replayed: per-unit latency without host launch overhead."""
    u = sess.units[0]

    def step(i, st):
        run_unit(sess, u, st)

    us = graph_time_us(step, reps, device)
    return {"us_per_unit": round(us, 1), "value": round(sess.unit_flops(u) / (us * 1e-6) / 1e12, 3),
            "unit": UNIT, "method": f"{reps} unit steps captured in one CUDA graph, replayed once"}


# ------------------------------------------------------------ oracle arms

def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def host_cpu() -> dict:
    """The host the oracle runs on: CPU model and the cores this process may use."""
    model = "unknown"
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    try:
        affinity = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        affinity = os.cpu_count() or 1
    return {"cpu_model": model, "affinity_cores": affinity}


def oracle_unit_sample(sess: UnitSession, u: int, n_rows: int, heads=None):
    """Time the oracle on a row sample of unit u; returns (seconds, flops)."""
    from oracle import block_causal as bc
    w = sess.w
    offs = sess.offsets_all[:u + 2]
    lo, hi = int(offs[-2]), int(offs[-1])
    idx = np.unique(np.linspace(0, hi - lo - 1, n_rows).astype(np.int64))
    heads = list(range(w.heads)) if heads is None else heads
    e = int(offs[-1])
    key = (u, tuple(heads))
    cache = getattr(sess, "_f32_cache", None)
    if cache is None or cache[0] != key:
        # host-side data preparation (not timed): bf16 -> fp32, with unit u appended
        k = sess.k_host[heads, :e].float().numpy()
        v = sess.v_host[heads, :e].float().numpy()
        k_new, v_new = sess.kv_host[u]
        k[:, lo:hi] = k_new[:, heads].transpose(0, 1).float().numpy()
        v[:, lo:hi] = v_new[:, heads].transpose(0, 1).float().numpy()
        sess._f32_cache = (key, k, v)
    _, k, v = sess._f32_cache
    q = sess.q_host[u][idx][:, heads].float().numpy()
    t0 = time.perf_counter()
    bc.attention_rows(q, lo + idx, k, v, offs)
    dt = time.perf_counter() - t0
    flops = attention_flops(offs, lo + idx, len(heads), w.head_dim)
    return dt, flops, idx.size, len(heads)


def oracle_step_rest(sess: UnitSession, u: int):
    """Oracle Euler steps over the unit's full latents; returns seconds."""
    from oracle import flow_matching as fm
    z = sess.eps_host[u].numpy()
    vel = [t.float().numpy() for t in sess.vel_host[u]]
    t0 = time.perf_counter()
    for s in range(sess.w.euler_steps):
        z = fm.euler_step(z, vel[s], 1.0 / sess.w.euler_steps)
    return time.perf_counter() - t0


REFERENCE_ROWS = 64


def cpu_baseline(sess: UnitSession):
    u = sess.units[0]
    n_rows = REFERENCE_ROWS
    dt, flops, rows, heads = oracle_unit_sample(sess, u, n_rows)
    return {"value": round(flops / dt / 1e12, 6), "unit": UNIT, "cores": blas_threads(),
            "kind": "oracle", **host_cpu(),
            "sample": f"fp64 numpy oracle, block-causal attention of {rows} evenly spaced query rows x "
                      f"{heads} heads of unit {u} against {int(sess.offsets_all[u + 1])} keys "
                      f"({flops / 1e9:.1f} GFLOP in {dt:.2f} s)"}


def _timed(fn):
    t0 = time.perf_counter()
    out = fn()
    return time.perf_counter() - t0, out


def oracle_append_euler(sess: UnitSession, u: int):
    """The oracle's full KV append of unit u's slice into the session's cache
    (a bit copy; 16-bit views of the bf16 bytes) and its full Euler steps over
    the unit's latents: seconds for each."""
    from oracle import kv_cache as kc
    k16 = sess.k_host.view(torch.int16).numpy()
    v16 = sess.v_host.view(torch.int16).numpy()
    kn, vn = (t.view(torch.int16).numpy() for t in sess.kv_host[u])
    dt_app, _ = _timed(lambda: kc.kv_append(k16, v16, kn, vn, int(sess.offsets_all[u])))
    return dt_app, oracle_step_rest(sess, u)


def oracle_full(sess: UnitSession):
    """The oracle timed in full where that takes seconds, on the machine's host
    cores: every attention row of the tiny fp32 and 192x336 workloads, and the
    append and Euler steps of the bench unit and the 192x336 unit.  The long
    session's unit has the bench unit's shapes (its append copies a larger
    cache; the oracle's append copies its whole cache, so its time scales
    with the capacity) and the prefill's bulk append is timed on 8 of its 128
    units -- both said so in the entries."""
    from oracle import block_causal as bc
    out = {}
    # tiny fp32: the full prefill and the per-block incremental calls
    w = WORKLOADS["tiny_fp32"]
    offs = w.offsets()
    k = torch.stack([w.head_timeline("k", 0, w.n_units)]).double().numpy()
    v = torch.stack([w.head_timeline("v", 0, w.n_units)]).double().numpy()
    q = w.head_timeline("q", 0, w.n_units).double().numpy()[:, None, :]
    dt_p, _ = _timed(lambda: bc.block_causal_attention(q, k, v, offs))
    dt_i, _ = _timed(lambda: [bc.unit_attention(q[int(offs[b]):int(offs[b + 1])], k[:, :int(offs[b + 1])],
                                                 v[:, :int(offs[b + 1])], offs[:b + 2])
                              for b in range(len(offs) - 1)])
    out["tiny_fp32"] = {"prefill_s": round(dt_p, 4), "incremental_8_blocks_s": round(dt_i, 4)}
    # 192x336: every row of the unit's attention, plus its append and Euler steps
    s2 = UnitSession(WORKLOADS["unit_192x336"], None, host_only=True)
    u2 = s2.units[0]
    dt_a, fl, rows, heads = oracle_unit_sample(s2, u2, s2.sizes[u2])
    dt_app2, dt_eu2 = oracle_append_euler(s2, u2)
    out["unit_192x336"] = {"attention_s": round(dt_a, 3), "attention_tflops": round(fl / dt_a / 1e12, 6),
                           "rows": rows, "heads": heads, "append_s": round(dt_app2, 4),
                           "euler_4_steps_s": round(dt_eu2, 4)}
    del s2
    u = sess.units[0]
    dt_app, dt_eu = oracle_append_euler(sess, u)
    out.setdefault(sess.w.name, {}).update({"append_s": round(dt_app, 4), "euler_steps_s": round(dt_eu, 4),
                                            "cache_rows": int(sess.cap)})
    out["long_session_640x368"] = {"note": f"same slice and latent shapes as {sess.w.name}: its Euler "
                                           f"steps take the time above; its append copies a cache of "
                                           f"{WORKLOADS['long_session_640x368'].capacity()} rows instead of "
                                           f"{sess.cap}"}
    # prefill: the bulk append of 8 units (all heads) into a cache of 8 units
    wp = WORKLOADS["prefill_128x932"]
    sizes = wp.unit_sizes()[:8]
    kn = wp.token_major_range("k", 0, 8, sizes).view(torch.int16).numpy()
    vn = wp.token_major_range("v", 0, 8, sizes).view(torch.int16).numpy()
    from oracle import kv_cache as kc
    cache = np.zeros((wp.heads, kn.shape[0], wp.head_dim), dtype=np.int16)
    dt_b, _ = _timed(lambda: kc.kv_append(cache, cache, kn, vn, 0))
    out["prefill_128x932"] = {"bulk_append_8_units_s": round(dt_b, 4),
                              "extrapolated_128_units_s": round(dt_b * 16, 3),
                              "note": "bulk append timed on 8 of the 128 units; the 128-unit figure is "
                                      "that time x 16, an estimate"}
    return out


def prefill_cpu_baseline(w: Workload, q_h, k_h, v_h, offs, n_rows: int = 64, n_heads: int = 8):
    """The oracle on a bounded sample of the prefill: n_rows evenly spaced
    query rows x the first n_heads heads, each against its visible keys."""
    from oracle import block_causal as bc
    T = int(offs[-1])
    rows = np.unique(np.linspace(0, T - 1, n_rows).astype(np.int64))
    heads = list(range(min(n_heads, w.heads)))
    e_max = int(offs[np.searchsorted(offs, rows.max(), side="right")])
    k = k_h[:e_max, heads].transpose(0, 1).float().numpy()
    v = v_h[:e_max, heads].transpose(0, 1).float().numpy()
    q = q_h[rows][:, heads].float().numpy()
    dt, _ = _timed(lambda: bc.attention_rows(q, rows, k, v, offs))
    flops = attention_flops(offs, rows, len(heads), w.head_dim)
    return {"value": round(flops / dt / 1e12, 6), "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
            **host_cpu(),
            "sample": f"fp64 numpy oracle, block-causal attention of {rows.size} evenly spaced query rows "
                      f"x {len(heads)} heads of the {T}-token prefill against their visible keys "
                      f"({flops / 1e9:.1f} GFLOP in {dt:.2f} s)"}


def reference_arm(args, rank, world):
    if rank != 0:
        return None
    w = WORKLOADS[args.workload]
    if w.prefill:
        raise SystemExit("--impl reference times the oracle on the streaming-unit workloads only")
    sess = UnitSession(w, None, host_only=True)
    u = sess.units[0]
    n = sess.sizes[u]
    # Each step is one measured run of the oracle on a named, bounded sample
    # of the unit: its attention for n_rows evenly spaced query rows x every
    # head.  value and ms_per_step are that measurement, nothing scaled.  A
    # long run (more than 60 steps) takes a quarter of the rows per step so
    # that it still ends within a few minutes.
    n_rows = REFERENCE_ROWS if args.steps + args.warmup <= 60 else REFERENCE_ROWS // 4
    times, flops_s, rows = [], 0.0, 0
    for i in range(args.warmup + args.steps):
        dt_attn, flops_s, rows, nh = oracle_unit_sample(sess, u, n_rows)
        if i >= args.warmup:
            times.append(dt_attn * 1e3)
    ms = statistics.mean(times)
    value = flops_s / (ms * 1e-3) / 1e12
    euler_ms = oracle_step_rest(sess, u) * 1e3
    cores = blas_threads()
    sample = (f"per step: fp64 numpy oracle, block-causal attention of {rows} evenly spaced query rows x "
              f"{w.heads} heads of unit {u} against {int(sess.offsets_all[u + 1])} keys "
              f"({flops_s / 1e9:.1f} GFLOP)")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, sess, u),
            "step_sample": sample,
            "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cores, "kind": "oracle",
                             **host_cpu(), "sample": sample},
            "extrapolated": {"unit_ms": round(ms * (n / rows) + euler_ms, 1),
                             "what": f"the sample's time scaled to the unit's {n} query rows, plus "
                                     f"{w.euler_steps} oracle Euler steps over the full latents "
                                     f"({euler_ms:.1f} ms, measured once): an estimate, not a measurement"},
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def workload_config(w: Workload, sess: UnitSession, u: int):
    offs = sess.offsets_all[:u + 2]
    return {"workload": w.name, "heads": w.heads, "head_dim": w.head_dim,
            "q_len": int(offs[-1] - offs[-2]), "kv_len": int(offs[-1]),
            "history_units": w.history_units, "new_units": w.new_units,
            "euler_steps": w.euler_steps, "latent": [w.latent_tokens, w.latent_channels],
            "cache_capacity_tokens": sess.cap,
            "l2": "inputs larger than L2: every step reads the full K/V cache "
                  f"({2 * w.heads * int(offs[-1]) * w.head_dim * 2 / 1e9:.2f} GB)"}


# ------------------------------------------------------------ prefill arm

def prefill_main(args, w: Workload, device, rank, world, peaks):
    line = prefill_measure(args.steps, args.warmup, w, device, rank, world, peaks,
                           with_e2e=not args.no_e2e,
                           with_cpu=not args.no_cpu_baseline and world == 1 and rank == 0)
    if rank == 0:
        print(json.dumps(line), flush=True)
    barrier(world, device)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def prefill_measure(K: int, W: int, w: Workload, device, rank, world, peaks, with_e2e=True,
                    with_cpu=False):
    """One step = the session prefill: bulk KV append of all T tokens, then
    full-sequence block-causal attention over them (every call through the C
    ABI).  Returns the bench line."""
    from streaming_block_causal_flash_b300 import ws
    sizes = w.unit_sizes()
    offs = w.offsets()
    T, H, D = int(offs[-1]), w.heads, w.head_dim
    q_h = w.token_major_range("q", 0, w.n_units, sizes)
    k_h = w.token_major_range("k", 0, w.n_units, sizes)
    v_h = w.token_major_range("v", 0, w.n_units, sizes)
    q, k_new, v_new = q_h.to(device), k_h.to(device), v_h.to(device)
    kc = torch.empty(H, T, D, dtype=torch.bfloat16, device=device)
    vc = torch.empty_like(kc)
    out = torch.empty_like(q)
    offs_dev = torch.from_numpy(offs.astype(np.int32)).to(device)
    flops = attention_flops(offs, np.arange(T), H, D)
    stream = torch.cuda.current_stream(device)

    def step(ev=None, st=stream, src=(q, k_new, v_new), dst=out):
        if ev is not None:
            ev[0].record(st)
        ws.ws_kv_append(src[1], src[2], kc, vc, 0, stream=st)
        if ev is not None:
            ev[1].record(st)
        ws.ws_block_causal_prefill(src[0], kc, vc, dst, offs, offs_dev, stream=st)
        if ev is not None:
            ev[2].record(st)

    for _ in range(W):
        step()
    torch.cuda.synchronize(device)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(K)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(device.index)
    clocks.start()
    barrier(world, device)
    torch.cuda.synchronize(device)
    start.record(stream)
    for i in range(K):
        step(evs[i])
    stop.record(stream)
    torch.cuda.synchronize(device)
    barrier(world, device)
    clk = clocks.stop()
    code, info = ws.ws_get_device_error()
    if code != 0:
        raise SystemExit(f"device error word set during the timed region: {info:#x}")
    local_ms = start.elapsed_time(stop) / K
    max_ms, total_flops = reduce_over_ranks(local_ms, flops * K, world, device)
    value = total_flops / (max_ms * 1e-3 * K) / 1e12
    attn_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    append_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    achieved = flops / (attn_ms * 1e-3) / 1e12
    line = {"metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": W, "ms_per_step": round(max_ms, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic: seeded N(0,1)*0.5 bf16 Q/K/V",
            "config": {"workload": w.name, "heads": H, "head_dim": D, "tokens": T,
                       "units": w.n_units, "attention_tflop": round(flops / 1e12, 3),
                       "l2": f"inputs larger than L2 (K/V {2 * H * T * D * 2 / 1e9:.2f} GB)"},
            "roofline": {"bound": "tensor", "achieved": round(achieved, 2),
                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": round(achieved / peaks["bf16_tflops"], 4),
                         "traffic": recorded_traffic(w.name),
                         "kernel": "attn_tc_bf16_kernel, prefill mode (one ws_block_causal_prefill call)",
                         "frac_of_sustained_peak": round(achieved / peaks["bf16_tflops_sustained"], 4)},
            "gpu_launches": 2 * K, "clocks": clk,
            "kernels_ms_mean": {"kv_append_bulk": round(append_ms, 4), "block_causal_prefill": round(attn_ms, 4)}}
    if with_e2e and rank == 0:
        hq, hk, hv = q_h.pin_memory(), k_h.pin_memory(), v_h.pin_memory()
        ho = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        dq, dk, dv, do = torch.empty_like(q), torch.empty_like(k_new), torch.empty_like(v_new), torch.empty_like(out)
        reps = max(3, min(K, 10))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            dq.copy_(hq, non_blocking=True)
            dk.copy_(hk, non_blocking=True)
            dv.copy_(hv, non_blocking=True)
            step(src=(dq, dk, dv), dst=do)
            ho.copy_(do, non_blocking=True)
        b.record(stream)
        torch.cuda.synchronize(device)
        e_ms = a.elapsed_time(b) / reps
        line["e2e"] = {"value": round(flops / (e_ms * 1e-3) / 1e12, 3), "unit": UNIT,
                       "ms_per_step": round(e_ms, 3), "steps": reps,
                       "h2d_bytes_per_step": int(3 * q.numel() * 2), "d2h_bytes_per_step": int(out.numel() * 2)}
    if with_cpu:
        line["cpu_baseline"] = prefill_cpu_baseline(w, q_h, k_h, v_h, offs)
    del q, k_new, v_new, kc, vc, out
    return line


def measure_unit_brief(name: str, device, peaks, steps: int = 10, warmup: int = 3):
    """The unit step of another streaming workload, measured compactly so
    that one bench line covers every configuration: per-step CUDA-event
    times (each of the workload's new units in turn), the attention call's
    TFLOP/s and roofline fraction, clocks, and the graph-replayed step."""
    w = WORKLOADS[name]
    sess = UnitSession(w, device)
    n_units = len(sess.units)
    K = max(steps, n_units)
    args = argparse.Namespace(steps=K, warmup=min(warmup, K))
    clocks = ClockSampler(device.index)
    total_ms, flops, append_ms, attn_ms, euler_ms, unit_ms, clk = time_native(args, sess, device, 1, clocks)
    per_attn = statistics.mean(sess.unit_flops(sess.units[i % n_units]) for i in range(K))
    achieved = per_attn / (statistics.mean(attn_ms) * 1e-3) / 1e12
    out = {"config": workload_config(w, sess, sess.units[0]), "steps": K,
           "ms_per_step": round(total_ms / K, 4),
           "value": round(flops / (total_ms * 1e-3) / 1e12, 3), "unit": UNIT,
           "per_unit_ms": {"mean": round(statistics.mean(unit_ms), 4),
                           "p50": round(statistics.median(unit_ms), 4), "max": round(max(unit_ms), 4),
                           "min": round(min(unit_ms), 4), "units": n_units},
           "kernels_ms_mean": {"kv_append": round(statistics.mean(append_ms), 4),
                               "block_causal_attn": round(statistics.mean(attn_ms), 4),
                               "fm_euler_steps": round(statistics.mean(euler_ms), 4)},
           "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"],
                        "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4)},
           "clocks": clk}
    if n_units == 1:
        out["graph"] = time_unit_graph(sess, device)
    del sess
    torch.cuda.empty_cache()
    return out


def measure_other_workloads(device, peaks, exclude: str):
    """Brief measurements of every bf16 workload but the line's own."""
    res = {}
    # streaming units first, the prefill (which heats the GPU most) last
    order = sorted(WORKLOADS.items(), key=lambda kv: kv[1].prefill)
    for name, w in order:
        if w.dtype != "bf16" or name == exclude:
            continue
        if w.prefill:
            line = prefill_measure(2, 1, w, device, 0, 1, peaks, with_e2e=False, with_cpu=True)
            res[name] = {k: line[k] for k in ("config", "value", "unit", "ms_per_step", "roofline", "clocks",
                                              "kernels_ms_mean", "cpu_baseline")}
            res[name]["steps"] = 2
        else:
            res[name] = measure_unit_brief(name, device, peaks)
        torch.cuda.empty_cache()
    return res


# --------------------------------------------------------------------- main

def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if args.impl == "reference":
        init_dist(world, "gloo")
        line = reference_arm(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        if world > 1:
            torch.distributed.destroy_process_group()
        return 0

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the hot path has no CPU fallback)")
    from streaming_block_causal_flash_b300 import build as ws_build
    from streaming_block_causal_flash_b300 import ws
    ws_build.build()
    ws.load()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    init_dist(world, "nccl")
    peaks = load_peaks()
    w = WORKLOADS[args.workload]
    if w.prefill:
        return prefill_main(args, w, device, rank, world, peaks)
    sess = UnitSession(w, device)
    clocks = ClockSampler(local)
    total_ms, flops, append_ms, attn_ms, euler_ms, unit_ms, clk = time_native(
        args, sess, device, world, clocks)
    code, info = ws.ws_get_device_error()
    if code != 0:
        raise SystemExit(f"device error word set during the timed region: {info:#x}")
    K = args.steps
    local_ms = total_ms / K
    max_ms, total_flops = reduce_over_ranks(local_ms, flops, world, device)
    value = total_flops / (max_ms * 1e-3 * K) / 1e12

    # roofline of the dominant call (attention: main kernel + combine)
    attn_avg_ms = statistics.mean(attn_ms)
    u0 = sess.units[0]
    per_launch = statistics.mean(sess.unit_flops(sess.units[i % len(sess.units)]) for i in range(K))
    achieved = per_launch / (attn_avg_ms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                "traffic": recorded_traffic(w.name),
                "kernel": "attn_tc_bf16_kernel (+ attn_combine_kernel) = one ws_block_causal_attn call",
                "peak_source": f"{peaks['source']} bf16 burst (MEASURED_PEAKS.json)"
                if peaks["source"] == "measured" else "fallback 1.8 PFLOP/s (no MEASURED_PEAKS.json)",
                "frac_of_sustained_peak": round(achieved / peaks["bf16_tflops_sustained"], 4)}
    per_unit = {"mean": round(statistics.mean(unit_ms), 4), "p50": round(statistics.median(unit_ms), 4),
                "max": round(max(unit_ms), 4), "min": round(min(unit_ms), 4),
                "units": len(sess.units),
                "what": "device time of each timed step (append + attention + Euler steps of one "
                        "unit, CUDA events on the launching stream); the steps cycle over the "
                        f"workload's {len(sess.units)} new unit(s)"}
    if len(sess.units) > 1:
        per_unit["by_unit_mean"] = {str(u): round(statistics.mean(
            unit_ms[i] for i in range(K) if sess.units[i % len(sess.units)] == u), 4)
            for u in sess.units if any(sess.units[i % len(sess.units)] == u for i in range(K))}
    line = {"metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": round(max_ms, 4),
            "us_per_unit": round(max_ms * 1e3, 1), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic: seeded N(0,1)*0.5 bf16 Q/K/V, N(0,1) latents and velocities",
            "config": workload_config(w, sess, u0), "roofline": roofline,
            "gpu_launches": sess.launches_per_step() * K, "clocks": clk,
            "kernels_ms_mean": {"kv_append": round(statistics.mean(append_ms), 4),
                                "block_causal_attn": round(attn_avg_ms, 4),
                                "fm_euler_steps": round(statistics.mean(euler_ms), 4)},
            "per_unit_ms": per_unit,
            "attn_ms_x_sm_mhz": clock_normalised(attn_avg_ms, clk)}
    if not args.no_e2e:
        e2e = time_e2e(args, sess, device)
        e_ms, e_flops = reduce_over_ranks(e2e["ms_per_step"], sess.unit_flops(sess.units[0]), world, device)
        e2e["value"] = round(e_flops / (e_ms * 1e-3) / 1e12, 3)
        e2e["ms_per_step"] = round(e_ms, 4)
        line["e2e"] = e2e
    if rank == 0:
        if not args.no_hbm:
            line["hbm_kernels"] = time_hbm_kernels(sess, device, peaks)
            line["graph"] = time_unit_graph(sess, device)
            line["attn_side"] = time_attn_side(sess, device, peaks)
            line["graph_fused_commit"] = time_fused_unit(sess, device)
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_baseline(sess)
            if not args.no_other_workloads:
                line["cpu_baseline"]["oracle_full"] = oracle_full(sess)
        if not args.no_other_workloads and world == 1:
            line["workloads"] = measure_other_workloads(device, peaks, w.name)
        print(json.dumps(line), flush=True)
    barrier(world, device)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
