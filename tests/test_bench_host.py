"""Host-side logic of bench.py: the FLOP count, the over-ranks reduction
(world size 2 on gloo), argument defaults and the traffic bookkeeping."""
import os

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import bench
from oracle import block_causal as bc


def test_attention_flops_counts_visible_pairs():
    offsets = np.array([0, 3, 3, 8, 12])
    mask = bc.visibility_mask(offsets)
    rows = np.arange(12)
    assert bench.attention_flops(offsets, rows, heads=3, head_dim=16) == 4 * 16 * 3 * mask.sum()
    last = np.arange(8, 12)       # the newest unit sees every key
    assert bench.attention_flops(offsets, last, 1, 128) == 4 * 128 * 4 * 12


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    ms, work = bench.reduce_over_ranks(1.0 + rank, 10.0 * (rank + 1), world)
    q.put((rank, ms, work))
    torch.distributed.destroy_process_group()


def test_reduce_over_ranks_takes_max_time_and_total_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for _, ms, work in res:
        assert ms == 2.0 and work == 30.0


def test_default_arguments_are_the_unit_640x368_bench():
    a = bench.parse_args([])
    assert a.gpus == 1 and a.warmup >= 3 and a.workload == "unit_640x368" and a.impl == "native"


def test_recorded_traffic_is_null_when_kernel_changed(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "PROFILES_DIR", str(tmp_path))
    f = tmp_path / "attn_tcgen05_unit_640x368_traffic.txt"
    f.write_text("dram_bytes_per_launch: 123\nkernel_source_sha256_16: deadbeef\n")
    assert bench.recorded_traffic() is None
    f.write_text(f"dram_bytes_per_launch: 123\nkernel_source_sha256_16: {bench.source_digest(bench.ATTN_SOURCE)}\n")
    assert bench.recorded_traffic() == 123.0
    assert bench.recorded_traffic("long_session_640x368") is None


def test_clock_sampler_without_nvidia_smi(monkeypatch):
    def boom(*a, **k):
        raise OSError("no nvidia-smi")
    monkeypatch.setattr(bench.subprocess, "Popen", boom)
    s = bench.ClockSampler(0)
    s.start()
    assert s.stop()["samples"] == 0


def test_reference_arm_under_torchrun_two_ranks(tmp_path):
    """bench.py --impl reference launched like the multi-GPU arm (torchrun,
    two ranks, gloo on CPU): rank 0 prints exactly one JSON line for the
    oracle, the other rank exits 0 without output."""
    import json
    import socket
    import subprocess
    import sys
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        port = sock.getsockname()[1]
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(root, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--workload", "unit_192x336"]
    import time
    t0 = time.time()
    res = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=root)
    wall = time.time() - t0
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["cpu_baseline"]["affinity_cores"] >= 1 and line["cpu_baseline"]["cpu_model"]
    # the step time is a measurement of the named sample: it fits in the run
    assert line["ms_per_step"] * (line["steps"] + line["warmup"]) / 1e3 < wall
    assert line["cpu_baseline"]["value"] == line["value"] and "step_sample" in line


def test_clock_sampler_reads_nvml_snapshots_and_reasons(monkeypatch):
    """With NVML available the sampler records a snapshot at start and stop
    (so a timed region of a few milliseconds still carries samples) and
    reports the median SM clock, the maximum and the active reasons."""
    import sys
    import types
    import time

    clocks = iter([1900, 1950, 2000] + [2000] * 10000)
    fake = types.SimpleNamespace(
        NVML_CLOCK_SM=1,
        nvmlClocksEventReasonHwSlowdown=0x8, nvmlClocksEventReasonHwThermalSlowdown=0x40,
        nvmlClocksEventReasonSwThermalSlowdown=0x20, nvmlClocksEventReasonSwPowerCap=0x4,
        nvmlInit=lambda: None,
        nvmlDeviceGetHandleByPciBusId=lambda bus: "h",
        nvmlDeviceGetHandleByIndex=lambda i: "h",
        nvmlDeviceGetClockInfo=lambda h, kind: next(clocks),
        nvmlDeviceGetMaxClockInfo=lambda h, kind: 2032,
        nvmlDeviceGetCurrentClocksEventReasons=lambda h: 0x4,
        nvmlDeviceGetPowerUsage=lambda h: 900000,
    )
    monkeypatch.setitem(sys.modules, "pynvml", fake)
    s = bench.ClockSampler(0, period_s=0.001)
    s.start()
    time.sleep(0.01)
    out = s.stop()
    assert out["samples"] >= 2
    assert out["sm_max_mhz"] == 2032 and out["reasons"] == ["sw_power_cap"]
    assert 1900 <= out["sm_mhz"] <= 2000 and out["power_w_median"] == 900.0
    assert bench.clock_normalised(2.0, out) == round(2.0 * out["sm_mhz"], 1)
    assert bench.clock_normalised(2.0, {"sm_mhz": None}) is None


def test_oracle_timing_suite_and_prefill_sample_on_the_cpu():
    """The full oracle timings and the prefill's sampled oracle baseline run on
    the host alone and report what they timed."""
    from streaming_block_causal_flash_b300.inputs import Workload
    sess = bench.UnitSession(bench.WORKLOADS["unit_192x336"], None, host_only=True)
    full = bench.oracle_full(sess)
    assert full["tiny_fp32"]["prefill_s"] > 0 and full["unit_192x336"]["rows"] == 264
    assert full["unit_192x336"]["heads"] == 24 and full["unit_192x336"]["append_s"] > 0
    assert "estimate" in full["prefill_128x932"]["note"]
    w = Workload("p", seed=5, heads=2, head_dim=128, dtype="bf16", std=0.5, video_tokens=100,
                 audio_tokens=0, text_tokens=0, history_units=0, new_units=6, latent_tokens=1,
                 latent_channels=8, euler_steps=0, prefill=True)
    sizes = w.unit_sizes()
    q, k, v = (w.token_major_range(n, 0, w.n_units, sizes) for n in ("q", "k", "v"))
    cb = bench.prefill_cpu_baseline(w, q, k, v, w.offsets(), n_rows=16, n_heads=2)
    assert cb["kind"] == "oracle" and cb["value"] > 0 and "16 evenly spaced" in cb["sample"]
