#!/usr/bin/env python3
"""Benchmark of the FFD decode-attention step (one kernel: stages 1-3 and the split merge) on GB300.

Default workload: the Qwen2.5-7B-shaped decode step (batch 4, 28 query / 4 KV heads, 128K
context, S=64, L=1024, delta=5), seeded synthetic inputs, N=1. Prints ONE JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

value = algorithmic HBM bytes of one step / device time of one step (GB/s): all 2-bit
thumbnails (48 B per token and KV head) + int8 residual and bf16 V of the kept blocks (392 B per
kept token and KV head) + q, output, seq_lens and block table. Inputs are resident in HBM and
larger than L2, so no flush is needed between steps. N > 1 runs one rank per GPU, each on its own
sequences (weak scaling, no collective on the data path).

--impl reference times the CPU oracle (test infrastructure, fp64) on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn µs/step & achieved HBM GB/s vs 8 TB/s roofline, 32K–256K ctx"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0
L2_BYTES = 129 * 1000 ** 2
THUMB_B = 48          # bytes per token and KV head: 32 code bytes + 4 fp16 scales + 4 fp16 zeros
REFINE_B = 136 + 256  # int8 residual + 4 fp16 residual scales + bf16 V
DENSE_B = 512         # bf16 K + V
LAUNCHES_PER_DECODE = 1  # one cooperative kernel: stage 1, stages 2/3, split merge
# the committed ncu summary of each schedule's kernel, and the sources its hash covers
PROFILES = {0: os.path.join(ROOT, "profiles", "ffd_main_kernel_qwen2.5-7b_128k.txt"),
            1: os.path.join(ROOT, "profiles", "ffd_sparse_kernel_qwen2.5-7b_128k_peaked.txt")}


SCHEDULES = {"fused": 0, "scan-refine": 1}  # FFD_SCHEDULE_FUSED, FFD_SCHEDULE_SCAN_REFINE
SCHEDULE_NAMES = {v: k for k, v in SCHEDULES.items()}


def pick_schedule(a, ffd, total_blocks: int, kept_blocks: int) -> int:
    """--schedule auto: the library's suggestion from the kept blocks of a first (untimed) step,
    as a serving loop would take it from the previous step; else the named schedule."""
    if a.schedule == "auto":
        return ffd.ffd_suggest_schedule(total_blocks, kept_blocks)
    return SCHEDULES[a.schedule]


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def args_parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000,
                    help="timed steps (the default keeps the timed region near 0.5 s)")
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=2, help="workload id 0..4")
    ap.add_argument("--delta", type=float, default=None)
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the peaked-attention variant and the CPU baseline")
    ap.add_argument("--schedule", choices=["auto", "fused", "scan-refine"], default="auto",
                    help="order of the decode step's work (FFD_SCHEDULE_*; same results); auto: "
                         "ffd_suggest_schedule from a first untimed step's keep mask")
    ap.add_argument("--peaked", action="store_true",
                    help="measure the peaked-attention inputs (sink shift and needles in score "
                         "units) as the primary workload")
    ap.add_argument("--sweep", metavar="MD",
                    help="instead of the benchmark line: time every workload (literal and peaked, "
                         "each delta) next to the dense kernel, one JSON line per case, and "
                         "write a markdown table to MD")
    return ap.parse_args(argv)


# ------------------------------------------------------------------------------------------- #
# Byte accounting (algorithmic, per step)                                                      #
# ------------------------------------------------------------------------------------------- #

def kept_tokens(seq_lens, keep_mask) -> int:
    """Valid tokens inside kept blocks, summed over (sequence, KV head)."""
    total = 0
    B, Hkv, maxb = keep_mask.shape
    for b in range(B):
        n = int(seq_lens[b])
        nb = (n + 63) // 64
        if nb == 0:
            continue
        sizes = np.full(nb, 64, np.int64)
        sizes[-1] = n - 64 * (nb - 1)
        total += int((keep_mask[b, :, :nb].astype(np.int64) * sizes[None]).sum())
    return total


def step_bytes(w, seq_lens, max_blocks, kept) -> dict:
    tok_heads = int(np.sum(seq_lens)) * w.num_kv_heads
    q = w.batch * w.num_q_heads * 128 * 2
    out = w.batch * w.num_q_heads * 128 * 4
    meta = 4 * w.batch + 4 * w.batch * max_blocks
    thumbs = THUMB_B * tok_heads
    refine = REFINE_B * kept
    return {"thumbs": thumbs, "refine": refine, "q": q, "out": out, "meta": meta,
            "step": thumbs + refine + q + out + meta,
            "main_kernel": thumbs + refine + q + out + meta,  # the step is this one kernel
            "dense_step": DENSE_B * tok_heads + q + out + meta,
            "token_heads": tok_heads}


def unit_bytes(w, seq_lens, keep_mask, units) -> int:
    """Algorithmic bytes of a subset of (sequence, KV head) units (CPU-baseline sample)."""
    G = w.num_q_heads // w.num_kv_heads
    total = 0
    for (b, h) in units:
        n = int(seq_lens[b])
        nb = (n + 63) // 64
        sizes = np.full(nb, 64, np.int64)
        if nb:
            sizes[-1] = n - 64 * (nb - 1)
        kept = int((keep_mask[b, h, :nb].astype(np.int64) * sizes).sum())
        total += THUMB_B * n + REFINE_B * kept + G * 128 * (2 + 4)
    return total


# ------------------------------------------------------------------------------------------- #
# Multi-rank plumbing                                                                          #
# ------------------------------------------------------------------------------------------- #

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max_sum(elapsed_ms: float, nbytes: float, backend_device="cpu"):
    """Max of the per-rank times and sum of the per-rank bytes over the process group (a no-op
    without one). Returns (max_ms, total_bytes)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return elapsed_ms, nbytes
    t = torch.tensor([elapsed_ms], dtype=torch.float64, device=backend_device)
    b = torch.tensor([nbytes], dtype=torch.float64, device=backend_device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t.item()), float(b.item())


def rank_seed(base: int, rank: int) -> int:
    """Each rank decodes its own sequences: rank 0 keeps the workload's seed."""
    return base + 7919 * rank


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device])
        else:
            dist.barrier()


# ------------------------------------------------------------------------------------------- #
# Clocks                                                                                       #
# ------------------------------------------------------------------------------------------- #

LEAD_CYCLES = 400_000  # device cycles of the pre-timing delay (~0.2 ms at 2 GHz)


class NvmlPoller:
    """Reads the SM clock and the clock-event (throttle) reasons through NVML (the driver's
    libnvidia-ml, read-only queries) every `period_s` on a thread, between start() and stop().
    The driver's timed regions can be a few milliseconds long, far shorter than nvidia-smi's
    sampling period; NVML answers in microseconds. Unavailable NVML leaves `ok` False."""
    SM_CLOCK = 1
    BITS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
            0x4: "sw_power_cap", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_index: int, period_s: float = 2.5e-4, pci_bus_id: str | None = None):
        import ctypes
        self.period = period_s
        self.samples = []
        self.ok = False
        self._stop = threading.Event()
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            # the CUDA device by its PCI address (NVML numbers every GPU of the machine, CUDA
            # only the visible ones); by index when the address is unknown
            found = pci_bus_id is not None and nv.nvmlDeviceGetHandleByPciBusId_v2(
                pci_bus_id.encode(), ctypes.byref(self.h)) == 0
            if not found and nv.nvmlDeviceGetHandleByIndex_v2(
                    ctypes.c_uint(gpu_index), ctypes.byref(self.h)) != 0:
                return
            self.reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self.nv, self.ct = nv, ctypes
            mx = ctypes.c_uint()
            self.max_mhz = float(mx.value) if nv.nvmlDeviceGetMaxClockInfo(
                self.h, self.SM_CLOCK, ctypes.byref(mx)) == 0 else None
            self.ok = True
        except (OSError, AttributeError):
            self.ok = False

    def _sample(self):
        c, r = self.ct.c_uint(), self.ct.c_ulonglong()
        if self.nv.nvmlDeviceGetClockInfo(self.h, self.SM_CLOCK, self.ct.byref(c)) != 0:
            return
        if self.reasons_fn(self.h, self.ct.byref(r)) != 0:
            return
        self.samples.append((float(c.value), int(r.value)))

    def _loop(self):
        while not self._stop.is_set():
            self._sample()
            time.sleep(self.period)

    def start(self):
        if self.ok:
            self.thread = threading.Thread(target=self._loop, daemon=True)
            self.thread.start()

    def stop(self):
        if self.ok:
            self._stop.set()
            self.thread.join(timeout=2)
            self._sample()  # one reading right after the region ends

    def summary(self):
        if not self.samples:
            return None
        reasons = sorted({name for _, r in self.samples for bit, name in self.BITS.items()
                          if r & bit})
        return {"sm_mhz": statistics.median(c for c, _ in self.samples),
                "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(self.samples), "window": "timed",
                "source": f"NVML every {self.period * 1e3:g} ms during the timed steps"}


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, pci_bus_id: str | None = None):
        self.gpu = gpu_index
        self.pci = pci_bus_id
        self.samples = []
        self.proc = None
        self.t_on = self.t_off = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20", "-i", self.pci or str(self.gpu)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        # nvidia-smi's start-up (driver queries, seconds on a fresh machine) must not overlap the
        # timed region: wait for its first sample (at most 15 s)
        t_end = time.time() + 15.0
        while not self.samples and time.time() < t_end and self.proc.poll() is None:
            time.sleep(0.01)

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark_on(self):
        self.t_on = time.time()
        self.nvml = NvmlPoller(self.gpu, pci_bus_id=self.pci)
        self.nvml.start()

    def mark_off(self):
        self.nvml.stop()
        self.t_off = time.time()

    def stop(self) -> dict:
        fast = self.nvml.summary() if getattr(self, "nvml", None) is not None else None
        smi = self._stop_smi()
        if fast and fast["samples"] >= 3:
            fast["nvidia_smi"] = smi
            return fast
        return smi

    def _stop_smi(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "note": "nvidia-smi unavailable"}
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        rows = []
        for ts, line in self.samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9], parts[4]))
            except ValueError:
                continue
        window = [r for r in rows if self.t_on and self.t_on <= r[0] <= (self.t_off or 1e30)]
        which = "timed"
        if len(window) < 3:
            window, which = rows, "warmup+timed+after"
        if not window:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in window for i, v in enumerate(r[3])
                          if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[1] for r in window),
                "sm_max_mhz": max(r[2] for r in window), "reasons": reasons,
                "samples": len(window), "window": which,
                "source": "nvidia-smi every 20 ms"}


# ------------------------------------------------------------------------------------------- #
# GPU arm                                                                                      #
# ------------------------------------------------------------------------------------------- #

def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0}, "fallback"


MAIN_KERNEL_SOURCES = {
    0: ("decode.cu", "stage1.cuh", "scan.cuh", "splitkv.cuh", "common.cuh", "ptx.cuh"),
    1: ("sparse.cu", "stage1.cuh", "scan.cuh", "splitkv.cuh", "common.cuh", "ptx.cuh")}


def main_kernel_sha256(schedule: int = 0):
    """SHA-256 over the sources a schedule's kernel is compiled from, in a fixed order."""
    h = hashlib.sha256()
    for name in MAIN_KERNEL_SOURCES[schedule]:
        with open(os.path.join(ROOT, "sparse_quantized_attention_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profile_traffic(schedule: int = 0, workload: str | None = None):
    # workload: words that the summary's workload line must contain (name and input kind)
    """DRAM bytes per launch of the schedule's kernel from the committed ncu summary, if the
    kernel source has not changed since the counters were taken and the summary is of this
    workload (else None)."""
    try:
        text = open(PROFILES[schedule]).read()
    except OSError:
        return None, None
    fields = dict(line.split(":", 1) for line in text.splitlines() if ":" in line)
    have_wl = fields.get("workload", "")
    if workload is not None and not all(part in have_wl for part in workload.split()):
        return None, "the committed capture is of another workload"
    want = fields.get("source_sha256", "").strip()
    have = main_kernel_sha256(schedule)
    if want != have:
        return None, "kernel changed since the ncu capture"
    try:
        return float(fields["dram_bytes_per_launch"].split()[0]), fields.get("workload", "").strip()
    except (KeyError, ValueError):
        return None, None


def pci_bus_id(torch, index: int) -> str | None:
    """PCI address of a CUDA device in NVML's form (domain:bus:device.function)."""
    try:
        p = torch.cuda.get_device_properties(index)
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except (AttributeError, RuntimeError):
        return None


def run_ours(a, rank, world, local):
    import torch

    import ffd_synth
    import sparse_quantized_attention_gb300 as ffd

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    w = ffd_synth.WORKLOADS[a.workload]
    delta = a.delta if a.delta is not None else w.deltas[0]
    inp = ffd_synth.make_inputs(w, seed=rank_seed(w.seed, rank),
                                signal_scale=ffd_synth.peaked_scale() if a.peaked else 1.0)
    G = w.num_q_heads // w.num_kv_heads
    sm = float(np.float32(1.0 / math.sqrt(128.0)))

    def upload(i):
        bf = lambda x: torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(  # noqa
            torch.bfloat16).to(dev)
        return {"q": bf(i.q_bits), "k": bf(i.k_bits), "v": bf(i.v_bits),
                "seq_lens": torch.from_numpy(i.seq_lens).to(dev),
                "block_table": torch.from_numpy(i.block_table).to(dev)}

    d = upload(inp)
    P, Hkv = d["k"].shape[0], d["k"].shape[1]
    qc = ffd.alloc_quantized_cache(P, Hkv, device=dev)
    stream = torch.cuda.current_stream(dev)

    # a0: quantisation of the whole cache (precondition of the step, timed on its own)
    ffd.ffd_quantize_keys(d["k"], qc)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    ffd.ffd_quantize_keys(d["k"], qc)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    quant_ms = e0.elapsed_time(e1)
    quant_bytes = P * Hkv * 64 * (256 + 32 + 8 + 8 + 128 + 8)

    params = ffd.make_params(w.batch, w.num_q_heads, w.num_kv_heads, P, inp.max_blocks,
                             sink=w.sink, local=w.local, delta=delta, sm_scale=sm)
    ws = ffd.alloc_workspace(params, device=dev)
    out = torch.empty((w.batch, w.num_q_heads, 128), dtype=torch.float32, device=dev)
    mask = torch.zeros((w.batch, w.num_kv_heads, inp.max_blocks), dtype=torch.uint8, device=dev)

    def step(keep=None):
        ffd.ffd_decode_attention(params, d["q"], qc, d["v"], d["seq_lens"], d["block_table"],
                                 out, ws, keep_mask=keep)

    step(mask)
    if ffd.ffd_get_error(ws) != 0:
        raise RuntimeError("device error during the first decode step")
    keep = mask.cpu().numpy()
    kept = kept_tokens(inp.seq_lens, keep)
    nb_total = int(sum((int(n) + 63) // 64 for n in inp.seq_lens)) * w.num_kv_heads
    kept_blocks = int(keep.sum())
    by = step_bytes(w, inp.seq_lens, inp.max_blocks, kept)
    params.schedule = pick_schedule(a, ffd, nb_total, kept_blocks)

    # timed region: W warm-up steps, then exactly K steps between barriers + syncs
    clocks = ClockSampler(local, pci_bus_id(torch, local))
    clocks.start()
    for _ in range(a.warmup):
        step()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    barrier(local)
    torch.cuda.synchronize(dev)
    clocks.mark_on()
    # a short device-side delay (a bounded clock spin, about 0.2 ms) queued ahead of the start
    # event, so that the first timed launch is already enqueued when the device reaches it: the
    # events then measure device time only (the host's launch cost is in the end-to-end figure)
    # one event between consecutive launches: the per-launch durations (median, p10, p90) and
    # their sum, the timed region
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(a.steps + 1)]
    torch.cuda._sleep(LEAD_CYCLES)
    evs[0].record(stream)
    for i in range(a.steps):
        step()
        evs[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    clocks.mark_off()
    barrier(local)
    torch.cuda.synchronize(dev)
    clock_info = clocks.stop()
    total_ms = evs[0].elapsed_time(evs[-1])
    per_launch_us = np.array([evs[i].elapsed_time(evs[i + 1]) * 1e3 for i in range(a.steps)])
    if ffd.ffd_get_error(ws) != 0:
        raise RuntimeError("device error during the timed steps")

    max_ms, all_bytes = reduce_max_sum(total_ms, by["step"] * a.steps,
                                       backend_device=dev if world > 1 else "cpu")
    ms_per_step = max_ms / a.steps
    value = all_bytes / a.steps / (ms_per_step * 1e-3) / 1e9

    aux_steps = max(3, min(a.steps, 200))  # the secondary rows: enough launches to average
    # e2e through the public API with pinned host buffers: q, seq_lens and the block table
    # packed in one pinned buffer (one host-to-device copy), the output read back (one
    # device-to-host copy), every step, inside the timed region
    qb = inp.q_bits.view(np.uint8).reshape(-1)
    sb = inp.seq_lens.view(np.uint8).reshape(-1)
    bb = inp.block_table.view(np.uint8).reshape(-1)
    o_s = (qb.size + 255) // 256 * 256
    o_b = o_s + (sb.size + 255) // 256 * 256
    h2d = o_b + bb.size
    hin = torch.zeros(h2d, dtype=torch.uint8).pin_memory()
    hin[:qb.size] = torch.from_numpy(qb)
    hin[o_s:o_s + sb.size] = torch.from_numpy(sb)
    hin[o_b:] = torch.from_numpy(bb)
    din = torch.empty(h2d, dtype=torch.uint8, device=dev)
    eq = din[:qb.size].view(torch.bfloat16).view(d["q"].shape)
    es = din[o_s:o_s + sb.size].view(torch.int32)
    eb = din[o_b:].view(torch.int32).view(d["block_table"].shape)
    hout = torch.empty(out.shape, dtype=torch.float32).pin_memory()
    d2h = hout.numel() * 4

    def e2e_step():
        din.copy_(hin, non_blocking=True)
        ffd.ffd_decode_attention(params, eq, qc, d["v"], es, eb, out, ws)
        hout.copy_(out, non_blocking=True)

    for _ in range(a.warmup):
        e2e_step()
    torch.cuda.synchronize(dev)
    barrier(local)
    t0.record(stream)
    for _ in range(aux_steps):
        e2e_step()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    stream_ms, _ = reduce_max_sum(t0.elapsed_time(t1), 0.0,
                                  backend_device=dev if world > 1 else "cpu")
    if not torch.equal(hout, out.cpu()):
        raise RuntimeError("end-to-end output differs from the device-resident step")
    # the headline e2e: host wall clock, every step waiting for its output on the host (a caller
    # that needs the result before its next step), so launch and copy latencies all count
    torch.cuda.synchronize(dev)
    barrier(local)
    w0 = time.perf_counter()
    for _ in range(aux_steps):
        e2e_step()
        stream.synchronize()
    w1 = time.perf_counter()
    e2e_ms, e2e_bytes = reduce_max_sum((w1 - w0) * 1e3, by["step"] * aux_steps,
                                       backend_device=dev if world > 1 else "cpu")
    e2e_value = e2e_bytes / aux_steps / (e2e_ms / aux_steps * 1e-3) / 1e9

    # a5: the in-library dense bf16 flash-decode on the same inputs
    wsd = ffd.alloc_workspace(params, dense=True, device=dev)
    outd = torch.empty_like(out)
    dense_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    dsteps = max(3, min(aux_steps, 50))
    for _ in range(3):
        ffd.ffd_dense_decode(params, d["q"], d["k"], d["v"], d["seq_lens"], d["block_table"],
                             outd, wsd)
    torch.cuda.synchronize(dev)
    dense_ev[0].record(stream)
    for _ in range(dsteps):
        ffd.ffd_dense_decode(params, d["q"], d["k"], d["v"], d["seq_lens"], d["block_table"],
                             outd, wsd)
    dense_ev[1].record(stream)
    torch.cuda.synchronize(dev)
    dense_ms = dense_ev[0].elapsed_time(dense_ev[1]) / dsteps

    # append-time quantisation of one token per sequence (the last one, rewritten with its own
    # key and value so the cache stays as it is), then append + decode captured once in a CUDA
    # graph and replayed: the decode loop's step without host launch overhead
    last = [(int(inp.block_table[b, (int(n) - 1) // 64]), (int(n) - 1) % 64)
            for b, n in enumerate(inp.seq_lens)]
    k_new = torch.stack([d["k"][pg, :, r] for pg, r in last]).contiguous()
    v_new = torch.stack([d["v"][pg, :, r] for pg, r in last]).contiguous()
    positions = (d["seq_lens"] - 1).contiguous()

    def append():
        ffd.ffd_append_kv(k_new, v_new, positions, d["block_table"], qc, d["v"])

    for _ in range(3):
        append()
    torch.cuda.synchronize(dev)
    app_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    app_ev[0].record(stream)
    for _ in range(50):
        append()
    app_ev[1].record(stream)
    torch.cuda.synchronize(dev)
    append_us = app_ev[0].elapsed_time(app_ev[1]) / 50 * 1e3

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        append()
        step()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize(dev)
    app_ev[0].record(stream)
    for _ in range(aux_steps):
        graph.replay()
    app_ev[1].record(stream)
    torch.cuda.synchronize(dev)
    graph_us = app_ev[0].elapsed_time(app_ev[1]) / aux_steps * 1e3
    if ffd.ffd_get_error(ws) != 0:
        raise RuntimeError("device error during the graph-captured steps")

    peaks, peak_src = measured_peaks()
    # a step is one launch of the main kernel: this rank's events around its K back-to-back steps
    # give the kernel's average launch duration (the launch gaps included)
    main_avg = total_ms / a.steps
    achieved = by["main_kernel"] / (main_avg * 1e-3) / 1e9
    traffic, traffic_note = profile_traffic(params.schedule,
                                            w.name + (" peaked" if a.peaked else " literal"))
    result = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(ms_per_step, 5),
        "us_per_step": round(ms_per_step * 1e3, 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name + ("-peaked" if a.peaked else ""), "batch": w.batch,
                   "num_q_heads": w.num_q_heads,
                   "num_kv_heads": w.num_kv_heads, "context": w.seq_len, "sink": w.sink,
                   "local": w.local, "delta": delta, "page": 64, "head_dim": 128,
                   "schedule": SCHEDULE_NAMES[params.schedule],
                   "l2": (f"inputs larger than L2 ({by['step'] / 1e6:.0f} MB read per step vs "
                          f"{L2_BYTES / 1e6:.0f} MB L2), no flush"
                          if by["step"] > 2 * L2_BYTES else
                          f"no flush: {by['step'] / 1e6:.0f} MB read per step against "
                          f"{L2_BYTES / 1e6:.0f} MB of L2, so back-to-back steps may find part "
                          f"of it in L2 (secondary_peaked times this workload launch by launch "
                          f"after an L2 flush)"),
                   "parallelism": "single GPU" if world == 1 else
                   f"replicas x{world} (own sequences per rank)"},
        "roofline": {"bound": "hbm",
                     "kernel": "ffd " + {0: "fused", 1: "scan-then-refine"}[params.schedule] +
                               " (stages 1-3, merge)",
                     "achieved": round(achieved, 1), "peak": peaks.get("hbm_gbs"),
                     "peak_source": f"{peak_src} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_src == "measured" else "fallback 6.8 TB/s",
                     "unit": "GB/s", "frac": round(achieved / peaks.get("hbm_gbs"), 4),
                     "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
                     "traffic": traffic, "traffic_note": traffic_note,
                     "algorithmic_bytes_per_launch": by["main_kernel"],
                     "kernel_us": round(main_avg * 1e3, 2),
                     "kernel_timing": "CUDA events on the launching stream between the K timed "
                                      "steps, one launch each",
                     "per_launch_us": {
                         "median": round(float(np.median(per_launch_us)), 2),
                         "p10": round(float(np.percentile(per_launch_us, 10)), 2),
                         "p90": round(float(np.percentile(per_launch_us, 90)), 2)}},
        "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "us_per_step": round(e2e_ms / aux_steps * 1e3, 2),
                "steps": aux_steps,
                "timing": "host wall clock (perf_counter) around copy in + decode + copy out + "
                          "stream synchronize, every step",
                "stream_us_per_step": round(stream_ms / aux_steps * 1e3, 2),
                "stream_timing": "CUDA events on the stream around the same steps issued back "
                                 "to back (no per-step synchronize)"},
        "gpu_launches": LAUNCHES_PER_DECODE * a.steps,
        "clocks": clock_info,
        "ffd": {"needed_bytes_per_step": by["step"], "kept_blocks": kept_blocks,
                "total_blocks": nb_total,
                "sparsity": round(1 - kept_blocks / max(1, nb_total), 4),
                "kept_token_fraction": round(kept / max(1, by["token_heads"]), 4),
                "effective_kv_tokens_per_s": round(float(np.sum(inp.seq_lens)) /
                                                   (ms_per_step * 1e-3), 1),
                "frac_of_nominal_8tbs": round(value / world / NOMINAL_HBM_GBS, 4)},
        "rows": {"quantize_us": round(quant_ms * 1e3, 2),
                 "quantize_gbs": round(quant_bytes / (quant_ms * 1e-3) / 1e9, 1),
                 "dense_us": round(dense_ms * 1e3, 2),
                 "dense_gbs": round(by["dense_step"] / (dense_ms * 1e-3) / 1e9, 1),
                 "speedup_vs_dense": round(dense_ms / ms_per_step, 3),
                 "append_us": round(append_us, 2),
                 "graph_append_decode_us": round(graph_us, 2)},
    }

    if not a.no_secondary and not a.peaked and rank == 0 and world == 1:
        result["secondary_peaked"] = peaked_variant(a, w, delta, dev, ffd, torch, upload,
                                                    dense_ms)
        result["cpu_baseline"] = cpu_baseline(w, inp, keep, delta, sm)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return result


def peaked_variant(a, w, delta, dev, ffd, torch, upload, dense_ms):
    """Same shapes with the sink shift and needle magnitude stated in score units: attention is
    concentrated, most blocks fall below m~ - delta and the stream is mostly thumbnails."""
    import ffd_synth
    inp = ffd_synth.make_inputs(w, signal_scale=ffd_synth.peaked_scale())
    d = upload(inp)
    P, Hkv = d["k"].shape[0], d["k"].shape[1]
    qc = ffd.alloc_quantized_cache(P, Hkv, device=dev)
    ffd.ffd_quantize_keys(d["k"], qc)
    sm = float(np.float32(1.0 / math.sqrt(128.0)))
    params = ffd.make_params(w.batch, w.num_q_heads, w.num_kv_heads, P, inp.max_blocks,
                             sink=w.sink, local=w.local, delta=delta, sm_scale=sm)
    ws = ffd.alloc_workspace(params, device=dev)
    out = torch.empty((w.batch, w.num_q_heads, 128), dtype=torch.float32, device=dev)
    mask = torch.zeros((w.batch, w.num_kv_heads, inp.max_blocks), dtype=torch.uint8, device=dev)
    ffd.ffd_decode_attention(params, d["q"], qc, d["v"], d["seq_lens"], d["block_table"], out,
                             ws, keep_mask=mask)
    keep = mask.cpu().numpy()
    kept = kept_tokens(inp.seq_lens, keep)
    by = step_bytes(w, inp.seq_lens, inp.max_blocks, kept)
    nb_total = int(sum((int(n) + 63) // 64 for n in inp.seq_lens)) * w.num_kv_heads
    stream = torch.cuda.current_stream(dev)
    # The peaked step reads about an L2's worth of bytes (all thumbnails and the few kept blocks),
    # so launches issued back to back would find part of them in L2: every launch of this
    # variant is timed alone with L2 emptied first by READING a buffer twice its size (a written
    # buffer would leave dirty lines whose write-back then lands inside the timed launch).
    flush = torch.zeros(2 * L2_BYTES // 8, dtype=torch.int64, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(fn, reps=20):
        """Mean of the middle 80 % of `reps` launches of fn, each after an L2 flush (us)."""
        for _ in range(3):
            fn()
        ts = []
        for _ in range(reps):
            flush.sum()
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ts.append(e0.elapsed_time(e1) * 1e3)
        ts.sort()
        k = len(ts) // 10
        return sum(ts[k:len(ts) - k]) / (len(ts) - 2 * k)

    psteps = max(10, min(a.steps, 200))
    by_schedule = {}
    for sched in (0, 1):  # both schedules, then the chosen one is the variant's figure
        params.schedule = sched
        by_schedule[SCHEDULE_NAMES[sched]] = timed(
            lambda: ffd.ffd_decode_attention(params, d["q"], qc, d["v"], d["seq_lens"],
                                             d["block_table"], out, ws), reps=psteps) * 1e-3
    chosen = pick_schedule(a, ffd, nb_total, int(keep.sum()))
    params.schedule = chosen
    ms = by_schedule[SCHEDULE_NAMES[chosen]]

    # the delta sweep: sparsity and step time of the Top-delta rule
    sweep = []
    for dl in (2.0, 5.0, 7.0, 10.0, math.inf):
        pd = ffd.make_params(w.batch, w.num_q_heads, w.num_kv_heads, P, inp.max_blocks,
                             sink=w.sink, local=w.local, delta=dl, sm_scale=sm)
        mk = torch.zeros_like(mask)
        ffd.ffd_decode_attention(pd, d["q"], qc, d["v"], d["seq_lens"], d["block_table"], out,
                                 ws, keep_mask=mk)
        pd.schedule = pick_schedule(a, ffd, nb_total, int(mk.sum()))
        us = timed(lambda: ffd.ffd_decode_attention(pd, d["q"], qc, d["v"], d["seq_lens"],
                                                    d["block_table"], out, ws))
        sweep.append({"delta": dl if math.isfinite(dl) else "inf", "us": round(us, 2),
                      "schedule": SCHEDULE_NAMES[pd.schedule],
                      "sparsity": round(1 - int(mk.sum()) / nb_total, 4)})
    # the comparison selectors on the same thumbnails: Top-k at the budget Top-delta used (its
    # mean kept non-forced blocks per unit), Top-p at p = 0.9 and 0.99; select + attention
    sws = ffd.alloc_select_workspace(params, device=dev)
    smask = torch.zeros_like(mask)
    forced_total = sum(forced_count(int(n), w.sink, w.local) for n in inp.seq_lens) * w.num_kv_heads
    k_budget = max(0, round((int(keep.sum()) - forced_total) / (w.batch * w.num_kv_heads)))
    selectors = {}
    for name, sel, budget in (("top_k", ffd.SELECT_TOPK, float(k_budget)),
                              ("top_p_0.9", ffd.SELECT_TOPP, 0.9),
                              ("top_p_0.99", ffd.SELECT_TOPP, 0.99)):
        def select():
            ffd.ffd_select_blocks(params, sel, budget, d["q"], qc, d["seq_lens"],
                                  d["block_table"], smask, sws)

        def attend():
            ffd.ffd_decode_attention_masked(params, d["q"], qc, d["v"], d["seq_lens"],
                                            d["block_table"], smask, out, ws)
        select()
        t_sel = timed(select)
        t_att = timed(attend)
        # the selector's own roofline: it streams every thumbnail record once (the per-block
        # statistics it writes and the mask are small beside them)
        sel_gbs = nb_total * 3072 / (t_sel * 1e-6) / 1e9
        selectors[name] = {"budget": budget, "select_us": round(t_sel, 2),
                           "select_thumbnail_gbs": round(sel_gbs, 1),
                           "select_frac_of_measured_copy_peak": round(
                               sel_gbs / measured_peaks()[0]["hbm_gbs"], 3),
                           "attention_us": round(t_att, 2),
                           "step_us": round(t_sel + t_att, 2),
                           "sparsity": round(1 - int(smask.sum()) / nb_total, 4)}
    if ffd.ffd_get_error(ws) != 0 or ffd.ffd_get_error(sws) != 0:
        raise RuntimeError("device error in the selector comparison")
    # run-time termination (ART) over the Top-delta mask: one CTA walks each (sequence, KV head)
    # unit; thresholds 0 use every kept block (compare with the fused step's stage 3)
    aws = ffd.alloc_art_workspace(params, device=dev)
    used = torch.zeros((w.batch, w.num_kv_heads), dtype=torch.int32, device=dev)
    aout = torch.empty_like(out)
    ffd.ffd_decode_attention_masked(params, d["q"], qc, d["v"], d["seq_lens"], d["block_table"],
                                    mask, out, ws)
    art = []
    for tau, phi, pat in ((0.0, 0.0, 1), (1e-3, 1e-4, 2), (1e-2, 1e-3, 2)):
        def run_art():
            ffd.ffd_art_attention(params, tau, phi, pat, d["q"], qc, d["v"], d["seq_lens"],
                                  d["block_table"], aout, aws, keep_in=mask, blocks_used=used)
        run_art()
        t_art = timed(run_art, reps=5)
        art.append({"tau": tau, "phi": phi, "patience": pat, "us": round(t_art, 2),
                    "mean_blocks_used": round(float(used.float().mean()), 1),
                    "max_abs_vs_all_kept": float((aout - out).abs().max())})
    if ffd.ffd_get_error(aws) != 0:
        raise RuntimeError("device error in the ART comparison")
    del d, qc
    return {"signal_scale": round(ffd_synth.peaked_scale(), 4), "us_per_step": round(ms * 1e3, 2),
            "timing": "every launch alone, L2 emptied before it by reading a buffer twice its "
                      "size; mean of the middle 80 % of the launches",
            "schedule": SCHEDULE_NAMES[chosen],
            "us_per_step_by_schedule": {k: round(v * 1e3, 2) for k, v in by_schedule.items()},
            "delta_sweep": sweep, "selectors": selectors, "art": art,
            "needed_bytes_per_step": by["step"], "gbs": round(by["step"] / (ms * 1e-3) / 1e9, 1),
            "sparsity": round(1 - int(keep.sum()) / nb_total, 4),
            "speedup_vs_dense": round(dense_ms / ms, 3),
            "effective_kv_tokens_per_s": round(float(np.sum(inp.seq_lens)) / (ms * 1e-3), 1)}


def forced_count(n, sink, local):
    """Blocks of a length-n sequence that hold a sink or local token."""
    nb = (n + 63) // 64
    return sum(1 for c in range(nb)
               if any(j < sink or j >= n - local for j in range(64 * c, min(n, 64 * c + 64))))


def cpu_baseline(w, inp, keep, delta, sm):
    """The CPU oracle as it stands, on the host cores, over a bounded sample of the same step's
    (sequence, KV head) units. Quantisation (a precondition of the step) is not timed."""
    import oracle
    qk = oracle.quantize(inp.k_bits)
    units = [(b, h) for b in range(w.batch) for h in range(w.num_kv_heads)]
    cores = oracle.default_threads()
    # bound the sample to about 10-30 s of CPU work: ~3e-8 s per (token, head, query head)
    G = w.num_q_heads // w.num_kv_heads
    per_unit = [3e-8 * int(inp.seq_lens[b]) * G * 128 / 64 for (b, h) in units]
    sample, cost = [], 0.0
    for u, c in zip(units, per_unit):
        if cost > 30.0 and sample:
            break
        sample.append(u)
        cost += c
    t = time.time()
    oracle.decode(inp.q_bits, inp.seq_lens, inp.block_table, qk, inp.v_bits, sink=w.sink,
                  local=w.local, delta=delta, sm_scale=sm, units=sample, threads=cores)
    dt = time.time() - t
    nbytes = unit_bytes(w, inp.seq_lens, keep, sample)
    return {"value": round(nbytes / dt / 1e9, 4), "unit": UNIT, "cores": min(cores, len(sample)),
            "kind": "oracle", "seconds": round(dt, 3),
            "sample": f"{len(sample)} of {len(units)} (sequence, KV head) units of one step "
                      f"({nbytes / 1e6:.1f} MB algorithmic)"}


# ------------------------------------------------------------------------------------------- #
# Reference arm: the CPU oracle                                                                #
# ------------------------------------------------------------------------------------------- #

def run_reference(a):
    import ffd_synth
    import oracle
    w = ffd_synth.WORKLOADS[a.workload]
    delta = a.delta if a.delta is not None else w.deltas[0]
    inp = ffd_synth.make_inputs(w)
    sm = float(np.float32(1.0 / math.sqrt(128.0)))
    qk = oracle.quantize(inp.k_bits)
    cores = oracle.default_threads()
    units = [(b, h) for b in range(w.batch) for h in range(w.num_kv_heads)]
    full_lens = inp.seq_lens.astype(np.int64)

    def run(sample, lens, threads):
        return oracle.decode(inp.q_bits, lens, inp.block_table, qk, inp.v_bits, sink=w.sink,
                             local=w.local, delta=delta, sm_scale=sm, units=sample,
                             threads=threads)

    # Each step decodes a bounded sample of the step's (sequence, KV head) units: up to one unit
    # per host core, over the first n' tokens of each sequence (n' = the full length unless the
    # whole --steps K --warmup W run would exceed about 150 s). Calibrate on one unit.
    per_step_units = max(1, min(len(units), cores))
    steps_total = a.warmup + a.steps
    budget_s = 150.0
    n_probe = int(min(full_lens.max(), 16384))
    t = time.time()
    run(units[:1], np.minimum(full_lens, n_probe).astype(np.int32), 1)
    per_token = max(1e-9, (time.time() - t) / max(1, n_probe))
    waves = math.ceil(per_step_units / cores)
    n_cap = int(budget_s / steps_total / waves / per_token)
    n_cap = max(1024, min(int(full_lens.max()), n_cap))
    lens = np.minimum(full_lens, n_cap).astype(np.int32)
    times, nbytes_list = [], []
    for s in range(steps_total):
        sample = [units[(s * per_step_units + k) % len(units)] for k in range(per_step_units)]
        t = time.time()
        res = run(sample, lens, cores)
        dt = time.time() - t
        if s >= a.warmup:
            times.append(dt)
            nbytes_list.append(unit_bytes(w, lens, res.mask, sample))
    total_t = sum(times)
    value = sum(nbytes_list) / total_t / 1e9
    prefix = ("whole sequences" if n_cap >= full_lens.max() else
              f"the first {n_cap} tokens of each sequence")
    sample_desc = (f"{per_step_units} of {len(units)} (sequence, KV head) units per step, "
                   f"rotating, {prefix}; fp64 oracle on {min(cores, per_step_units)} host "
                   f"threads")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": round(total_t / a.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch, "num_q_heads": w.num_q_heads,
                       "num_kv_heads": w.num_kv_heads, "context": w.seq_len, "sink": w.sink,
                       "local": w.local, "delta": delta},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT,
                             "cores": min(cores, per_step_units), "kind": "oracle",
                             "sample": sample_desc},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_sweep(a):
    """Every workload, literal and peaked inputs, each of its deltas: the decode step timed one
    launch at a time with L2 emptied in between by a read of twice its size (the 32K workload's
    cache fits in L2), next to the dense kernel on the same inputs."""
    import torch

    import ffd_synth
    import sparse_quantized_attention_gb300 as ffd

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    peaks, _ = measured_peaks()
    # L2 is emptied between launches by READING a buffer twice its size: a written buffer would
    # leave up to an L2's worth of dirty lines whose write-back then lands inside the next timed
    # launch
    flush = torch.zeros(2 * L2_BYTES // 8, dtype=torch.int64, device=dev)
    sm = float(np.float32(1.0 / math.sqrt(128.0)))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(fn, reps=30):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(reps):
            flush.sum()
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            ts.append(e0.elapsed_time(e1) * 1e3)
        return float(np.median(ts))

    rows = []
    for wid, w in sorted(ffd_synth.WORKLOADS.items()):
        dense_us = None
        for label, scale in (("literal", 1.0), ("peaked", ffd_synth.peaked_scale())):
            inp = ffd_synth.make_inputs(w, signal_scale=scale)
            bf = lambda x: torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(  # noqa
                torch.bfloat16).to(dev)
            d = {"q": bf(inp.q_bits), "k": bf(inp.k_bits), "v": bf(inp.v_bits),
                 "sl": torch.from_numpy(inp.seq_lens).to(dev),
                 "bt": torch.from_numpy(inp.block_table).to(dev)}
            P, Hkv = d["k"].shape[0], d["k"].shape[1]
            qc = ffd.alloc_quantized_cache(P, Hkv, device=dev)
            ffd.ffd_quantize_keys(d["k"], qc)
            out = torch.empty((w.batch, w.num_q_heads, 128), dtype=torch.float32, device=dev)
            mask = torch.zeros((w.batch, Hkv, inp.max_blocks), dtype=torch.uint8, device=dev)
            if dense_us is None:
                pdn = ffd.make_params(w.batch, w.num_q_heads, Hkv, P, inp.max_blocks,
                                      sink=w.sink, local=w.local, delta=5.0, sm_scale=sm)
                wsd = ffd.alloc_workspace(pdn, dense=True, device=dev)
                dense_us = timed(lambda: ffd.ffd_dense_decode(pdn, d["q"], d["k"], d["v"], d["sl"],
                                                              d["bt"], out, wsd))
            for delta in w.deltas:
                p = ffd.make_params(w.batch, w.num_q_heads, Hkv, P, inp.max_blocks, sink=w.sink,
                                    local=w.local, delta=delta, sm_scale=sm)
                ws = ffd.alloc_workspace(p, device=dev)
                ffd.ffd_decode_attention(p, d["q"], qc, d["v"], d["sl"], d["bt"], out, ws,
                                         keep_mask=mask)
                if ffd.ffd_get_error(ws) != 0:
                    raise RuntimeError(f"device error on workload {wid}")
                keep = mask.cpu().numpy()
                kept = kept_tokens(inp.seq_lens, keep)
                by = step_bytes(w, inp.seq_lens, inp.max_blocks, kept)
                nb_total = int(sum((int(n) + 63) // 64 for n in inp.seq_lens)) * Hkv
                us_by = {}
                for sched in (0, 1):
                    p.schedule = sched
                    us_by[SCHEDULE_NAMES[sched]] = timed(
                        lambda: ffd.ffd_decode_attention(p, d["q"], qc, d["v"], d["sl"], d["bt"],
                                                         out, ws))
                p.schedule = pick_schedule(a, ffd, nb_total, int(keep.sum()))
                us = us_by[SCHEDULE_NAMES[p.schedule]]
                # ART over the same mask with no termination (every kept block, one CTA per
                # unit walking its blocks in sequence): the unit that keeps the most sets the time
                aws = ffd.alloc_art_workspace(p, device=dev)
                used = torch.zeros((w.batch, Hkv), dtype=torch.int32, device=dev)
                art_us = timed(lambda: ffd.ffd_art_attention(
                    p, 0.0, 0.0, 1, d["q"], qc, d["v"], d["sl"], d["bt"], out, aws,
                    keep_in=mask, blocks_used=used))
                art_max = int(used.max())
                if ffd.ffd_get_error(aws) != 0:
                    raise RuntimeError(f"device error in ART on workload {wid}")
                gbs = by["step"] / (us * 1e-6) / 1e9
                row = {"workload": w.name, "inputs": label, "delta": delta,
                       "batch": w.batch, "heads": f"{w.num_q_heads}/{Hkv}",
                       "context": int(np.max(inp.seq_lens)), "us_per_step": round(us, 2),
                       "schedule": SCHEDULE_NAMES[p.schedule],
                       "us_fused": round(us_by["fused"], 2),
                       "us_scan_refine": round(us_by["scan-refine"], 2),
                       "kv_tokens_per_s": round(float(np.sum(inp.seq_lens)) / (us * 1e-6), 1),
                       "sparsity": round(1 - int(keep.sum()) / max(1, nb_total), 4),
                       "needed_mb": round(by["step"] / 1e6, 1), "gbs": round(gbs, 1),
                       "frac_of_measured": round(gbs / peaks["hbm_gbs"], 3),
                       "frac_of_8tbs": round(gbs / NOMINAL_HBM_GBS, 3),
                       "dense_us": round(dense_us, 2),
                       "speedup_vs_dense": round(dense_us / us, 2),
                       "art_us": round(art_us, 1), "art_max_blocks": art_max,
                       "art_us_per_block": round(art_us / max(1, art_max), 2)}
                rows.append(row)
                print(json.dumps(row), flush=True)
            del d, qc
            torch.cuda.empty_cache()
    with open(a.sweep, "w") as f:
        f.write("| workload | inputs | delta | context | us/step | schedule | fused us | "
                "scan-refine us | KV tokens/s | sparsity | "
                "needed MB | GB/s | of measured copy peak | of 8 TB/s | dense us | speedup | "
                "ART us (all kept) | ART blocks (max unit) | ART us/block |\n")
        f.write("|---|---|---|---|---|---|---|---|---|---|---|---|---|---|---|---|---|---|---|\n")
        for r in rows:
            f.write(f"| {r['workload']} | {r['inputs']} | {r['delta']:g} | {r['context']} | "
                    f"{r['us_per_step']} | {r['schedule']} | {r['us_fused']} | "
                    f"{r['us_scan_refine']} | {r['kv_tokens_per_s']:.3g} | {r['sparsity']} | "
                    f"{r['needed_mb']} | {r['gbs']} | {r['frac_of_measured']} | "
                    f"{r['frac_of_8tbs']} | {r['dense_us']} | {r['speedup_vs_dense']} | "
                    f"{r['art_us']} | {r['art_max_blocks']} | {r['art_us_per_block']} |\n")
    return rows


def free_port() -> int:
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def launch_command(nprocs: int, argv, script: str | None = None) -> list:
    """torchrun command that starts `nprocs` ranks of `script` (this file by default) on this
    node, rendezvous on 127.0.0.1."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
            f"--nproc-per-node={nprocs}", "--master-addr", "127.0.0.1",
            f"--master-port={free_port()}", script or os.path.abspath(__file__), *argv]


def self_launch(nprocs: int, argv, script: str | None = None) -> int:
    """Run the job as `nprocs` ranks (one per GPU) when started without a launcher: the ranks'
    output (rank 0 prints the JSON line) goes to this process's stdout and stderr."""
    log(f"starting {nprocs} ranks with torch.distributed.run")
    return subprocess.run(launch_command(nprocs, argv, script)).returncode


def main(argv=None):
    raw = list(sys.argv[1:] if argv is None else argv)
    a = args_parse(raw)
    if a.sweep:
        run_sweep(a)
        return 0
    if a.gpus > 1 and "WORLD_SIZE" not in os.environ:
        return self_launch(a.gpus, raw)
    rank, world, local = dist_env()
    if a.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(a)), flush=True)
        return 0
    if world != a.gpus:
        log(f"warning: --gpus {a.gpus} but WORLD_SIZE={world}; using WORLD_SIZE")
    result = run_ours(a, rank, world, local)
    if rank == 0:
        print(json.dumps(result), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
