#!/usr/bin/env python3
"""Benchmark of the fused q-norm / RoPE / KV-quant / paged-insert step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload stress]
    python bench.py --impl reference ...      # the CPU oracle on a bounded sample

A step is one pass of the whole fused step (one launch) over one batch: by default
the "stress" workload, 131072 tokens x 128 q heads (q is 17.2 GB of bf16), FP8 cache
of 2048 x 64 slots.  Inputs are resident in HBM before the timed region; q is far
larger than the 129 MB L2, so no flush is needed between steps (q is rewritten in
place; every step moves the same bytes).  Rank 0 prints one JSON line.

For N > 1 (torchrun, one rank per GPU) every rank runs its own independent batch of
the same shape (seed offset by rank): weak scaling, no collective on the data path;
the timed region is bracketed by barriers and the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402
from synth import configs  # noqa: E402

METRIC = "HBM GB/s (% of warm copy ceiling) and tokens/s, fused qnorm-rope-kv-insert"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0


# ------------------------------------------------------------------ distributed glue

def dist_env():
    """(rank, world_size, local_rank) from torchrun's environment (1 process: 0, 1, 0)."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_workload(wl: configs.Workload, rank: int) -> configs.Workload:
    """Rank r's independent batch: the same shape, seed offset by 1000 * r."""
    if rank == 0:
        return wl
    name = f"{wl.name}@rank{rank}"
    configs._POSITIONS.setdefault(name, configs._POSITIONS[wl.name])
    configs._SLOTS.setdefault(name, configs._SLOTS[wl.name])
    return dataclasses.replace(wl, name=name, seed=wl.seed + 1000 * rank)


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int, device=None) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ measurement helpers

KERNEL_SOURCES = tuple("kv_norm_rope_gb300/csrc/" + f for f in (
    "qnorm_rope_kv_insert.cu", "rowmath.cuh", "convert.cuh", "fastdiv.h", "launch.h",
    "launch_status.h", "bounds.cuh", "bounds_range.h"))


def kernel_fingerprint() -> str:
    """16 hex digits identifying the code of the kernel sources: comments and
    whitespace are dropped before hashing, so a comment edit does not orphan the
    figures profiled on that code (sha256 over the files' sha256s)."""
    import hashlib
    import re
    digests = ""
    for f in KERNEL_SOURCES:
        text = open(os.path.join(ROOT, f)).read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        digests += hashlib.sha256(" ".join(text.split()).encode()).hexdigest()
    return hashlib.sha256(digests.encode()).hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM read + write bytes per launch from the committed ncu summary of this
    workload, or None when there is none or the kernel changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"qnorm_rope_kv_insert_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    fp = traffic = None
    for line in text.splitlines():
        if "Kernel sources fingerprint" in line and "`" in line:
            fp = line.split("`")[1]
        if line.startswith("traffic_bytes_per_launch:"):
            traffic = int(line.split(":")[1])
    return traffic if fp == kernel_fingerprint() else None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples every 100 ms while running."""

    FIELDS = ("timestamp,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id: str | None):
        self.bus_id = bus_id
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        self.out = os.fdopen(fd, "w")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        time.sleep(0.25)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.out.close()
        with open(self.path) as f:
            lines = f.readlines()
        os.remove(self.path)
        return summarise_clocks(lines, self.bus_id)


def summarise_clocks(lines, bus_id: str | None) -> dict:
    """Median SM clock, max SM clock and the active throttle reasons of nvidia-smi
    CSV samples (the fields of ClockSampler), keeping only the GPU with `bus_id`."""
    rows = []
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 9:
            continue
        if bus_id and bus_id.lower() not in parts[1].lower():
            continue
        try:
            rows.append((float(parts[2]), float(parts[3]), parts[5:9]))
        except ValueError:
            continue
    if not rows:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = sorted({n for _, _, flags in rows for n, fl in zip(names, flags)
                      if fl.lower() == "active"})
    return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
            "reasons": reasons, "samples": len(rows)}


def self_check(per_gpu_gbs: float, achieved_gbs: float, copy_1g: float, copy_512m: float) -> dict:
    """A kernel cannot move its bytes faster than a plain device-to-device copy of the
    same run; more than 5% above it means the timed work is not what was counted.
    Reported, and warned about on stderr, rather than fatal."""
    ceiling = max(copy_1g, copy_512m)
    worst = max(per_gpu_gbs, achieved_gbs) / ceiling
    ok = worst <= 1.05
    if not ok:
        print(f"bench self-check: {worst:.3f} x the in-run copy ceiling ({ceiling:.0f} GB/s)",
              file=sys.stderr)
    return {"ok": ok, "over_copy_ceiling": round(worst, 4)}


def bus_id_of(device_index: int) -> str | None:
    import torch
    p = torch.cuda.get_device_properties(device_index)
    try:
        return f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}"
    except AttributeError:
        return None


def copy_ceiling_gbs(dev, nbytes: int) -> float:
    """Warm device-to-device copy: read + write bytes / time, median of 10 after 3 warm-ups."""
    import torch
    a = torch.empty(nbytes // 2, dtype=torch.bfloat16, device=dev)
    b = torch.empty_like(a)
    a.fill_(1.0)
    for _ in range(3):
        b.copy_(a)
    torch.cuda.synchronize(dev)
    times = []
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        b.copy_(a)
        e1.record()
        e1.synchronize()
        times.append(e0.elapsed_time(e1) / 1e3)
    del a, b
    return 2 * nbytes / statistics.median(times) / 1e9


# ------------------------------------------------------------------ inputs on the device

OPS = ("fused", "prenorm", "kv_only", "gather", "mxfp8", "indexer", "indexer_gather")
IO_OF_OP = {
    "fused": "bf16 q, kv in; bf16 q, FP8 (e4m3 + ue8m0 + bf16) or bf16 cache rows out",
    "prenorm": "bf16 q, normalised kv in; bf16 q, FP8 cache rows out",
    "kv_only": "bf16 kv in; FP8 or bf16 cache rows out",
    "gather": "FP8 cache rows in; bf16 rows out",
    "mxfp8": "bf16 x, residual in; bf16 residual, e4m3 codes, swizzled ue8m0 scales out",
    "indexer": "bf16 indexer K [T, 128] in; e4m3 codes + fp32 power-of-two scale rows out",
    "indexer_gather": "indexer cache rows in; contiguous e4m3 [T, 128] + fp32 [T] out",
}
MXFP8_HIDDEN = 7168
VARIANTS = {"auto": 0, "small": 1, "stream": 2, "half": 4}


class DeviceBatch:
    """One workload resident in HBM.  q and kv are drawn on the device by a seeded
    torch generator (N(0,1), the workload's heavy tail, rounded to bf16); positions,
    slots, the weight and the cos/sin table come from ``synth``.  ``op`` "kv_only"
    holds no q."""

    def __init__(self, wl: configs.Workload, dev, op: str = "fused", variant: int = 0,
                 hidden: int = MXFP8_HIDDEN):
        import torch
        self.variant = variant
        if op in ("kv_only", "gather", "mxfp8", "indexer", "indexer_gather"):
            wl = dataclasses.replace(wl, H=0)
        self.wl = wl
        self.op = op
        self.dev = dev
        g = torch.Generator(device=dev)
        g.manual_seed(wl.seed * 7919 + 17)
        self.q = self._normal((wl.T, wl.H, 512), g)
        self.kv = self._normal((wl.T, 512), g) if not op.startswith("indexer") else None
        self.positions_np = wl.positions()
        self.slots_np = wl.slot_mapping()
        self.w = torch.from_numpy(configs.weight_bits(wl).view(np.int16)).view(torch.bfloat16).to(dev)
        self.pos = torch.from_numpy(self.positions_np).to(dev)
        self.slots = torch.from_numpy(self.slots_np).to(dev)
        self.cs = torch.from_numpy(configs.cos_sin(wl)).to(dev)
        self.cache = torch.zeros(configs.cache_bytes(wl), dtype=torch.uint8, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.bytes = configs.algorithmic_bytes(wl, self.positions_np, self.slots_np)
        if op == "prenorm":
            self.bytes -= 1024  # no weight read
        if op == "mxfp8":
            # activation rows [T, hidden]: x, residual (in place), gamma, codes, scales
            import kv_norm_rope_gb300 as k
            n = self.hidden = hidden
            self.x = self._normal((wl.T, n), g)
            self.res = self._normal((wl.T, n), g)
            self.gamma = self._normal((n,), g)
            self.codes = torch.empty((wl.T, n), dtype=torch.uint8, device=dev)
            self.mx_scales = torch.empty(k.mxfp8_scale_bytes(wl.T, n), dtype=torch.uint8,
                                         device=dev)
            self.bytes = wl.T * n * (2 + 2 + 2 + 1) + self.mx_scales.numel() + 2 * n
        if op.startswith("indexer"):
            # indexer K rows [T, 128] and their paged cache (132 bytes per slot)
            import kv_norm_rope_gb300 as k
            self.k = self._normal((wl.T, 128), g)
            self.idx_cache = torch.zeros(k.indexer_cache_bytes(wl.num_blocks, wl.block_size),
                                         dtype=torch.uint8, device=dev)
            valid = int((self.slots_np >= 0).sum())
            self.bytes = wl.T * 8 + valid * (256 + 132)
            if op == "indexer_gather":
                k.indexer_k_quant_insert(self.k, self.slots, self.idx_cache, wl.num_blocks,
                                         wl.block_size)
                del self.k
                self.k_out = torch.empty((wl.T, 128), dtype=torch.uint8, device=dev)
                self.scale_out = torch.empty(wl.T, dtype=torch.float32, device=dev)
                self.bytes = wl.T * (8 + 132) + valid * 132
        if op == "gather":
            if wl.store != "fp8":
                raise ValueError("the reader reads FP8 caches")
            import kv_norm_rope_gb300 as k
            k.kv_norm_rope_insert(k.STORE_FP8, self.kv, self.w, self.pos, self.cs, self.slots,
                                  self.cache, wl.num_blocks, wl.block_size, wl.eps)
            del self.kv
            self.out = torch.empty((wl.T, 512), dtype=torch.bfloat16, device=dev)
            valid = int((self.slots_np >= 0).sum())
            self.bytes = wl.T * (8 + 1024) + valid * 584

    def _normal(self, shape, g):
        import torch
        wl = self.wl
        out = torch.empty(shape, dtype=torch.bfloat16, device=self.dev)
        flat = out.view(-1)
        chunk = 1 << 28
        for i in range(0, flat.numel(), chunk):
            n = min(chunk, flat.numel() - i)
            x = torch.randn(n, generator=g, device=self.dev, dtype=torch.float32)
            if wl.tail_frac > 0:
                u = torch.rand(n, generator=g, device=self.dev, dtype=torch.float32)
                x = torch.where(u < wl.tail_frac, x * wl.tail_mult, x)
            flat[i:i + n] = x.to(torch.bfloat16)
            del x
        return out

    def call(self, lib, stream_handle: int):
        """(C-ABI function, argument tuple) of one step of this batch's op."""
        wl = self.wl
        if self.op == "mxfp8":
            return lib.dsv4_add_gemma_rmsnorm_mxfp8, (
                self.x.data_ptr(), self.res.data_ptr(), self.gamma.data_ptr(), wl.T, self.hidden,
                wl.eps, self.res.data_ptr(), self.codes.data_ptr(), self.mx_scales.data_ptr(),
                stream_handle)
        if self.op == "indexer":
            return lib.dsv4_indexer_k_quant_insert, (
                self.k.data_ptr(), self.slots.data_ptr(), self.idx_cache.data_ptr(), wl.num_blocks,
                wl.block_size, wl.T, self.err.data_ptr(), stream_handle)
        if self.op == "indexer_gather":
            return lib.dsv4_indexer_k_gather, (
                self.idx_cache.data_ptr(), wl.num_blocks, wl.block_size, self.slots.data_ptr(),
                wl.T, self.k_out.data_ptr(), self.scale_out.data_ptr(), self.err.data_ptr(),
                stream_handle)
        if self.op == "gather":
            return lib.dsv4_dequant_gather, (
                self.cache.data_ptr(), wl.num_blocks, wl.block_size, self.slots.data_ptr(), wl.T,
                self.out.data_ptr(), self.err.data_ptr(), stream_handle)
        if self.op in ("kv_only", "prenorm") and self.variant:
            # the general entry, for an explicit launch variant
            return lib.dsv4_insert_ex, (
                0 if wl.store == "fp8" else 1, self.variant, 1 if self.op == "kv_only" else 0,
                self.q.data_ptr() if wl.H else None, self.kv.data_ptr(), self.w.data_ptr(),
                self.pos.data_ptr(), self.cs.data_ptr(), wl.max_position, self.slots.data_ptr(),
                self.cache.data_ptr(), wl.num_blocks, wl.block_size, wl.T, wl.H, wl.eps,
                self.err.data_ptr(), stream_handle)
        if self.op == "kv_only":
            return lib.dsv4_kv_norm_rope_insert, (
                0 if wl.store == "fp8" else 1, self.kv.data_ptr(), self.w.data_ptr(),
                self.pos.data_ptr(), self.cs.data_ptr(), wl.max_position, self.slots.data_ptr(),
                self.cache.data_ptr(), wl.num_blocks, wl.block_size, wl.T, wl.eps,
                self.err.data_ptr(), stream_handle)
        if self.op == "prenorm":
            if wl.store != "fp8":
                raise ValueError("the pre-normalised entry stores FP8 rows")
            return lib.dsv4_qnorm_rope_kv_rope_quant_insert, (
                self.q.data_ptr(), self.kv.data_ptr(), self.pos.data_ptr(), self.cs.data_ptr(),
                wl.max_position, self.slots.data_ptr(), self.cache.data_ptr(), wl.num_blocks,
                wl.block_size, wl.T, wl.H, wl.eps, self.err.data_ptr(), stream_handle)
        if self.variant:
            return lib.dsv4_insert_ex, (
                0 if wl.store == "fp8" else 1, self.variant, 1, self.q.data_ptr(),
                self.kv.data_ptr(), self.w.data_ptr(), self.pos.data_ptr(), self.cs.data_ptr(),
                wl.max_position, self.slots.data_ptr(), self.cache.data_ptr(), wl.num_blocks,
                wl.block_size, wl.T, wl.H, wl.eps, self.err.data_ptr(), stream_handle)
        fn = (lib.dsv4_qnorm_rope_kv_quant_insert if wl.store == "fp8"
              else lib.dsv4_qnorm_rope_kv_bf16_insert)
        return fn, (self.q.data_ptr(), self.kv.data_ptr(), self.w.data_ptr(), self.pos.data_ptr(),
                    self.cs.data_ptr(), wl.max_position, self.slots.data_ptr(),
                    self.cache.data_ptr(), wl.num_blocks, wl.block_size, wl.T, wl.H, wl.eps,
                    self.err.data_ptr(), stream_handle)


def graph_flushed_us(op, dev, flush, n: int = 50, reps: int = 7) -> float:
    """Device time of op(stream) without the host's launch latency: a CUDA graph of
    n (L2 flush, op) pairs replayed and timed with events, minus a graph of the n
    flushes alone, divided by n (median of `reps` replays)."""
    import torch

    def timed(with_op: bool) -> float:
        s = torch.cuda.Stream(dev)
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(s):
            if with_op:
                op(s)  # warm outside the capture
            torch.cuda.synchronize(dev)
            with torch.cuda.graph(g, stream=s):
                for i in range(n):
                    flush.fill_(i & 0xFF)
                    if with_op:
                        op(s)
        torch.cuda.synchronize(dev)
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize(dev)
            ts.append(e0.elapsed_time(e1) * 1e3 / n)
        return statistics.median(ts)

    return timed(True) - timed(False)


def graph_device_us(batch: DeviceBatch, lib, dev, flush, n: int = 50, reps: int = 7) -> float:
    """Device time of one launch of the batch's step (graph_flushed_us)."""
    def launch(s):
        fn, a = batch.call(lib, s.cuda_stream)
        fn(*a)
    return graph_flushed_us(launch, dev, flush, n, reps)


def graph_copy_us(nbytes: int, dev, flush, n: int = 50, reps: int = 7) -> dict:
    """The same measurement for moving nbytes / 2 bytes from one device buffer to
    another (nbytes read and written in total), two ways: a device-to-device memcpy,
    and an elementwise kernel (bitwise not of int32, one read and one write of each
    word).  What moving the step's bytes costs at this size, with the same launch,
    flush and L2 state around it."""
    import torch
    words = max(4, (nbytes // 2) // 16 * 4)
    src = torch.ones(words, dtype=torch.int32, device=dev)
    dst = torch.empty(words, dtype=torch.int32, device=dev)
    out = {"memcpy_us": graph_flushed_us(lambda s: dst.copy_(src), dev, flush, n, reps),
           "elementwise_us": graph_flushed_us(lambda s: torch.bitwise_not(src, out=dst), dev,
                                              flush, n, reps)}
    del src, dst
    return out


def graph_warm_us(batch: DeviceBatch, lib, dev, n: int = 50, reps: int = 7) -> float:
    """Device time of one launch run back to back with no flush in between (a CUDA
    graph of n launches, median of `reps` replays, divided by n): the inputs stay in L2
    where they fit, as when the step follows the kernel that produced them."""
    import torch
    s = torch.cuda.Stream(dev)
    g = torch.cuda.CUDAGraph()
    fn, a = batch.call(lib, s.cuda_stream)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(s):
        fn(*a)
        torch.cuda.synchronize(dev)
        with torch.cuda.graph(g, stream=s):
            for _ in range(n):
                fn(*a)
    torch.cuda.synchronize(dev)
    ts = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize(dev)
        ts.append(e0.elapsed_time(e1) * 1e3 / n)
    return statistics.median(ts)


def entry(lib, store: str):
    return (lib.dsv4_qnorm_rope_kv_quant_insert if store == "fp8"
            else lib.dsv4_qnorm_rope_kv_bf16_insert)


def known_answer_check() -> str:
    """The tiny workload against the oracle at the parity bar (before and after timing)."""
    from tests import harness
    rep = harness.check(configs.TINY)
    return "pass" if rep.ok else f"FAIL: {rep}"


# ------------------------------------------------------------------ end to end

def _cpulist(text: str) -> list:
    """'0-3,8,10-11' -> [0, 1, 2, 3, 8, 10, 11]"""
    out = []
    for part in text.strip().split(","):
        if not part:
            continue
        a, _, b = part.partition("-")
        out += list(range(int(a), int(b or a) + 1))
    return out


def _ranges(cpus) -> str:
    cpus = sorted(cpus)
    out, i = [], 0
    while i < len(cpus):
        j = i
        while j + 1 < len(cpus) and cpus[j + 1] == cpus[j] + 1:
            j += 1
        out.append(str(cpus[i]) if i == j else f"{cpus[i]}-{cpus[j]}")
        i = j + 1
    return ",".join(out)


def numa_nodes() -> dict:
    """CPU list of every NUMA node that has CPUs ({} where sysfs has no node info)."""
    nodes = {}
    base = "/sys/devices/system/node"
    try:
        names = os.listdir(base)
    except OSError:
        return nodes
    for n in names:
        if n.startswith("node") and n[4:].isdigit():
            try:
                cpus = _cpulist(open(os.path.join(base, n, "cpulist")).read())
            except OSError:
                continue
            if cpus:
                nodes[int(n[4:])] = cpus
    return nodes


def gpu_numa_node(device_index: int):
    """The NUMA node sysfs gives the GPU's PCI function (None if unknown or -1)."""
    import torch
    p = torch.cuda.get_device_properties(device_index)
    try:
        bdf = f"{p.pci_domain_id:04x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
        node = int(open(f"/sys/bus/pci/devices/{bdf}/numa_node").read())
    except (AttributeError, OSError, ValueError):
        return None
    return node if node >= 0 else None


def pages_by_node(ptr: int) -> dict:
    """Resident pages per NUMA node of the mapping that holds address ptr, from
    /proc/self/numa_maps ({} if unknown)."""
    try:
        lines = open("/proc/self/numa_maps").read().splitlines()
    except OSError:
        return {}
    best, best_start = None, -1
    for line in lines:
        start = int(line.split()[0], 16)
        if best_start < start <= ptr:
            best, best_start = line, start
    if best is None:
        return {}
    out = {}
    for f in best.split()[2:]:
        if f.startswith("N") and "=" in f and f[1:f.index("=")].isdigit():
            out[int(f[1:f.index("=")])] = int(f.split("=")[1])
    return out


_SYS_SET_MEMPOLICY = {"aarch64": 237, "x86_64": 238}


def prefer_node(node) -> bool:
    """Ask the kernel to place this thread's new pages on `node` (MPOL_PREFERRED), or
    back to the default policy for None.  False where the call is unavailable."""
    import ctypes
    import platform
    nr = _SYS_SET_MEMPOLICY.get(platform.machine())
    if nr is None:
        return False
    libc = ctypes.CDLL(None, use_errno=True)
    if node is None:
        return libc.syscall(nr, 0, None, 0) == 0
    if not 0 <= node < 64:
        return False
    mask = ctypes.c_ulong(1 << node)
    return libc.syscall(nr, 1, ctypes.byref(mask), 65) == 0


def link_ceilings(host, devbuf, dev, reps: int = 3, chunks: int = 8) -> dict:
    """Pinned host <-> device copy rates of the same buffers in this run (GB/s, best of
    reps): host->device, device->host, and both at once (chunk c of the first half goes
    up on one stream while chunk c of the second half comes down on another, as the
    e2e step interleaves its copies; GB/s counts both directions)."""
    import torch
    n = host.numel()
    half = n // 2
    nbytes = n * host.element_size()
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    cut = np.linspace(0, half, chunks + 1).astype(np.int64)

    def best(fn, moved):
        ts = []
        for _ in range(reps):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize(dev)
            ts.append(time.perf_counter() - t0)
        return round(moved / min(ts) / 1e9, 1)

    def both():
        for c in range(chunks):
            a, b = int(cut[c]), int(cut[c + 1])
            with torch.cuda.stream(s1):
                devbuf[a:b].copy_(host[a:b], non_blocking=True)
            with torch.cuda.stream(s2):
                host[half + a:half + b].copy_(devbuf[half + a:half + b], non_blocking=True)

    h2d = best(lambda: devbuf.copy_(host, non_blocking=True), nbytes)
    d2h = best(lambda: host.copy_(devbuf, non_blocking=True), nbytes)
    bidir = best(both, nbytes)
    return {"h2d_gbs": h2d, "d2h_gbs": d2h, "both_gbs": bidir, "bytes": nbytes,
            "how": f"pinned q buffer <-> device q, best of {reps} each; 'both': {chunks} chunks "
                   f"of the first half up on one stream while the second half's come down on "
                   f"another"}


def e2e_run(batch: DeviceBatch, lib, steps: int, chunks: int = 16):
    """Same metric through the C ABI with host buffers: per step, token chunks of q, kv,
    positions and slots go host->device from pinned memory, the kernel runs on each chunk,
    and q plus the cache come back device->host into separate pinned output buffers.
    Uploads, kernels and downloads run on three streams with per-chunk events.  The
    device buffers are double-buffered by step (step k uses set k % 2), so an upload
    waits only for the download of the same chunk two steps back and a step's first
    kernel only for the cache download two steps back: both directions of the host link
    stay busy across step boundaries.  Returns (GB/s, h2d bytes, d2h bytes, seconds per
    step, link ceilings, placement)."""
    import torch
    wl = batch.wl
    dev = batch.dev
    # pinned buffers on the GPU's own NUMA node where sysfs names one (the host link
    # runs through that node's memory); the placement found is reported either way
    gnode = gpu_numa_node(dev.index if dev.index is not None else 0)
    nodes = numa_nodes()
    preferred = gnode in nodes and prefer_node(gnode)
    try:
        q_in = torch.empty((wl.T, wl.H, 512), dtype=torch.bfloat16, pin_memory=True)
        q_out = torch.empty((wl.T, wl.H, 512), dtype=torch.bfloat16, pin_memory=True)
        kv_h = torch.empty((wl.T, 512), dtype=torch.bfloat16, pin_memory=True)
        pos_h = torch.from_numpy(batch.positions_np).pin_memory()
        sl_h = torch.from_numpy(batch.slots_np).pin_memory()
        cache_h = torch.empty(batch.cache.numel(), dtype=torch.uint8, pin_memory=True)
    finally:
        if preferred:
            prefer_node(None)
    q_in.copy_(batch.q)
    kv_h.copy_(batch.kv)
    allowed = sorted(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else []
    placement = {"gpu_numa_node": gnode, "preferred_node_for_pinned": bool(preferred),
                 "pinned_q_pages_by_node": pages_by_node(q_in.data_ptr()),
                 "process_cpus": _ranges(allowed),
                 "cpu_nodes": {n: _ranges(c) for n, c in sorted(nodes.items())}}
    ceilings = link_ceilings(q_in.view(-1), batch.q.view(-1), dev)
    fn = entry(lib, wl.store)
    sets = [(batch.q, batch.kv, batch.pos, batch.slots, batch.cache),
            (torch.empty_like(batch.q), torch.empty_like(batch.kv), torch.empty_like(batch.pos),
             torch.empty_like(batch.slots), torch.zeros_like(batch.cache))]
    s_in, s_k, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    bounds = np.linspace(0, wl.T, chunks + 1).astype(np.int64)
    h2d = q_in.numel() * 2 + kv_h.numel() * 2 + pos_h.numel() * 8 + sl_h.numel() * 8
    d2h = q_out.numel() * 2 + cache_h.numel()
    downloaded = [[None] * chunks, [None] * chunks]  # per set and chunk: its q is back
    cache_read = [None, None]                       # per set: its cache image is back

    def step(k):
        q, kv, pos, sl, cache = sets[k % 2]
        done = downloaded[k % 2]
        for c in range(chunks):
            a, b = int(bounds[c]), int(bounds[c + 1])
            if done[c] is not None:
                s_in.wait_event(done[c])  # the chunk's buffer was read out two steps back
            with torch.cuda.stream(s_in):
                q[a:b].copy_(q_in[a:b], non_blocking=True)
                kv[a:b].copy_(kv_h[a:b], non_blocking=True)
                pos[a:b].copy_(pos_h[a:b], non_blocking=True)
                sl[a:b].copy_(sl_h[a:b], non_blocking=True)
                up = torch.cuda.Event()
                up.record(s_in)
            s_k.wait_event(up)
            if c == 0 and cache_read[k % 2] is not None:
                s_k.wait_event(cache_read[k % 2])  # this set's cache was read out two steps back
            st = fn(q[a:b].data_ptr(), kv[a:b].data_ptr(), batch.w.data_ptr(), pos[a:b].data_ptr(),
                    batch.cs.data_ptr(), wl.max_position, sl[a:b].data_ptr(), cache.data_ptr(),
                    wl.num_blocks, wl.block_size, b - a, wl.H, wl.eps, batch.err.data_ptr(),
                    s_k.cuda_stream)
            if st != 0:
                raise RuntimeError(f"launch failed with status {st}")
            ran = torch.cuda.Event()
            ran.record(s_k)
            s_out.wait_event(ran)
            with torch.cuda.stream(s_out):
                q_out[a:b].copy_(q[a:b], non_blocking=True)
                done[c] = torch.cuda.Event()
                done[c].record(s_out)
        with torch.cuda.stream(s_out):
            cache_h.copy_(cache, non_blocking=True)
            cache_read[k % 2] = torch.cuda.Event()
            cache_read[k % 2].record(s_out)

    step(0)
    step(1)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for i in range(steps):
        step(i)
    torch.cuda.synchronize(dev)
    dt = (time.perf_counter() - t0) / steps
    # the link ceilings again, right after: the host link is shared with the
    # node's other GPUs and CPU jobs, so both measurements bracket the e2e run
    after = link_ceilings(q_in.view(-1), batch.q.view(-1), dev)
    ceilings = {"before": ceilings, "after": after,
                "both_gbs": max(ceilings["both_gbs"], after["both_gbs"])}
    del sets
    return batch.bytes / dt / 1e9, h2d, d2h, dt, ceilings, placement


def e2e_host_resident(batch: DeviceBatch, lib, steps: int):
    """The same metric through the C ABI with every per-token buffer in pinned host
    memory: q (rewritten in place), kv, positions, slots and the cache live on the
    host and the kernel reads and writes them over NVLink-C2C (pinned host memory is
    addressable from the GPU at the same address); only the cos/sin table, the weight
    and the error word stay on the device.  No copy engine is involved, so nothing
    serialises the two directions of the link.  Returns (GB/s, h2d bytes, d2h bytes,
    seconds per step)."""
    import torch
    wl = batch.wl
    dev = batch.dev
    gnode = gpu_numa_node(dev.index if dev.index is not None else 0)
    preferred = gnode in numa_nodes() and prefer_node(gnode)
    try:
        q_h = torch.empty((wl.T, wl.H, 512), dtype=torch.bfloat16, pin_memory=True)
        kv_h = torch.empty((wl.T, 512), dtype=torch.bfloat16, pin_memory=True)
        pos_h = torch.from_numpy(batch.positions_np).pin_memory()
        sl_h = torch.from_numpy(batch.slots_np).pin_memory()
        cache_h = torch.zeros(batch.cache.numel(), dtype=torch.uint8, pin_memory=True)
    finally:
        if preferred:
            prefer_node(None)
    q_h.copy_(batch.q)
    kv_h.copy_(batch.kv)
    fn = entry(lib, wl.store)
    s = torch.cuda.Stream(dev)
    call = (q_h.data_ptr(), kv_h.data_ptr(), batch.w.data_ptr(), pos_h.data_ptr(),
            batch.cs.data_ptr(), wl.max_position, sl_h.data_ptr(), cache_h.data_ptr(),
            wl.num_blocks, wl.block_size, wl.T, wl.H, wl.eps, batch.err.data_ptr(), s.cuda_stream)
    for _ in range(2):
        if fn(*call) != 0:
            raise RuntimeError("host-resident launch failed")
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(steps):
        fn(*call)
    torch.cuda.synchronize(dev)
    dt = (time.perf_counter() - t0) / steps
    valid = int((batch.slots_np >= 0).sum())
    h2d = q_h.numel() * 2 + kv_h.numel() * 2 + pos_h.numel() * 8 + sl_h.numel() * 8
    d2h = q_h.numel() * 2 + valid * (584 if wl.store == "fp8" else 1024)
    return batch.bytes / dt / 1e9, h2d, d2h, dt


# ------------------------------------------------------------------ CPU oracle timing

class OracleSample:
    """Tokens [t0, t0 + n) of a workload, generated once on the host, for timing the
    oracle: all q heads and the KV row of each token, cache writes included."""

    def __init__(self, wl: configs.Workload, n_tokens: int, t0: int = 0):
        t1 = min(wl.T, t0 + n_tokens)
        self.wl = wl
        self.q = configs.q_bits(wl, t0, t1).reshape(t1 - t0, wl.H, 512)
        self.kv = configs.kv_bits(wl, t0, t1).reshape(t1 - t0, 512)
        self.pos = wl.positions()[t0:t1]
        self.sl = wl.slot_mapping()[t0:t1]
        self.w = configs.weight_bits(wl)
        self.cs = configs.cos_sin(wl)
        self.n = t1 - t0
        self.bytes = (self.n * (2 * wl.H * 1024 + 1024 + 16) + int((self.sl >= 0).sum()) *
                      (584 if wl.store == "fp8" else 1024) + int(np.unique(self.pos).size) * 256
                      + 1024)

    def run(self, n_threads: int = 0) -> float:
        """Seconds for one oracle pass over the sample (on a fresh copy of q)."""
        import oracle
        wl = self.wl
        q = self.q.copy()
        cache = np.zeros(configs.cache_bytes(wl), np.uint8)
        start = time.perf_counter()
        oracle.qnorm_rope_kv_insert(wl.store, q, self.kv, self.w, self.pos, self.cs, self.sl,
                                    cache, wl.num_blocks, wl.block_size, wl.eps,
                                    n_threads=n_threads)
        return time.perf_counter() - start


def _sample_tokens_for(wl: configs.Workload, seconds: float) -> int:
    """Tokens the oracle processes in about `seconds` on all host cores."""
    probe = OracleSample(wl, 128)
    probe.run()  # warm (thread start-up, page faults)
    per_tok = max(probe.run() / probe.n, 1e-7)
    return int(max(1, min(wl.T, seconds / per_tok)))


def cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it (x86 "model name"; on Arm the
    implementer and part numbers), else the machine type."""
    import platform
    try:
        info = open("/proc/cpuinfo").read()
    except OSError:
        return platform.machine()
    for key in ("model name", "Model"):
        for line in info.splitlines():
            if line.startswith(key) and ":" in line:
                return line.split(":", 1)[1].strip()
    fields = {}
    for line in info.splitlines():
        if ":" in line:
            k, v = (x.strip() for x in line.split(":", 1))
            fields.setdefault(k, v)
    if "CPU implementer" in fields:
        return (f"{platform.machine()} implementer {fields['CPU implementer']} "
                f"part {fields.get('CPU part', '?')}")
    return platform.machine()


def cpu_baseline(wl: configs.Workload, seconds: float = 2.0):
    cores = os.cpu_count() or 1
    sample = OracleSample(wl, _sample_tokens_for(wl, seconds))
    dt = sample.run()
    return {"value": round(sample.bytes / dt / 1e9, 4), "unit": "GB/s", "cores": cores,
            "cpu": cpu_model(), "kind": "oracle",
            "sample": f"first {sample.n} tokens of {wl.name} ({wl.T}x{wl.H}), all heads + KV "
                      f"rows, {dt:.1f} s on {cores} threads",
            "tokens_per_s": round(sample.n / dt, 1)}


# ------------------------------------------------------------------ arms

def run_reference(args):
    """The oracle, as it stands, on the host cores: each step is one pass over a bounded
    token sample of the workload, sized so warm-up + steps take about two minutes."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    wl = configs.WORKLOADS[args.workload]
    cores = os.cpu_count() or 1
    n = _sample_tokens_for(wl, 120.0 / max(1, args.steps + args.warmup))
    sample = OracleSample(wl, n)
    times = []
    for i in range(args.warmup + args.steps):
        dt = sample.run()
        if i >= args.warmup:
            times.append(dt)
    mean = statistics.mean(times)
    value = sample.bytes / mean / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(mean * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "T": wl.T, "H": wl.H, "store": wl.store,
                       "step_sample_tokens": sample.n},
            "tokens_per_s": round(sample.n / mean, 1),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                             "cpu": cpu_model(), "kind": "oracle",
                             "sample": f"first {sample.n} tokens of {wl.name} per step, all "
                                       f"heads + KV rows"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def other_configs(lib, dev, names, steps: int, warmup: int):
    """The fused step on the other named workloads, in the same process after the main
    measurement, each timed like it (warm-up launches, CUDA events around every launch,
    a 256 MB L2 flush before each launch of a step that moves less than 4x the L2, plus
    its graph-replay time), so that one run of the default command records every
    configuration.  Returns one dict per workload."""
    import torch

    import kv_norm_rope_gb300 as k
    peak, _ = measured_peaks()
    out = []
    for name in names:
        batch = DeviceBatch(configs.WORKLOADS[name], dev)
        wl = batch.wl
        stream = torch.cuda.current_stream(dev)
        fn, call_args = batch.call(lib, stream.cuda_stream)
        for _ in range(warmup):
            st = fn(*call_args)
            if st != 0:
                raise RuntimeError(f"launch failed: {k.status_string(st)}")
        torch.cuda.synchronize(dev)
        if int(batch.err.item()) != 0:
            raise RuntimeError(f"device error bits {int(batch.err.item())} on {name}")
        flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) \
            if batch.bytes < 4 * (129 << 20) else None
        events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * steps)]
        torch.cuda.synchronize(dev)
        for i in range(steps):
            if flush is not None:
                flush.fill_(i & 0xFF)
            events[2 * i].record(stream)
            fn(*call_args)
            events[2 * i + 1].record(stream)
        torch.cuda.synchronize(dev)
        per_launch = [events[2 * i].elapsed_time(events[2 * i + 1]) / 1e3 for i in range(steps)]
        step_s = (statistics.mean(per_launch) if flush is not None
                  else events[0].elapsed_time(events[-1]) / 1e3 / steps)
        plan = k.launch_plan(wl.T, wl.H,
                             torch.cuda.get_device_properties(dev).multi_processor_count, 3)
        row = {"workload": name, "T": wl.T, "H": wl.H, "store": wl.store,
               "variant": {k.VARIANT_STREAM: "stream", k.VARIANT_SMALL: "small",
                           k.VARIANT_HALF: "half"}[plan.variant],
               "bytes_per_step": batch.bytes, "steps": steps,
               "ms_per_step": round(step_s * 1e3, 4),
               "GB/s": round(batch.bytes / step_s / 1e9, 1),
               "frac_of_measured_peak": round(batch.bytes / step_s / 1e9 / peak, 4),
               "tokens_per_s": round(wl.T / step_s, 1),
               "l2": "flushed before every launch (256 MB write)" if flush is not None
               else "inputs larger than L2"}
        if flush is not None:
            g_us = graph_device_us(batch, lib, dev, flush)
            row["graph_us_per_launch"] = round(g_us, 3)
            row["graph_GB/s"] = round(batch.bytes / g_us / 1e3, 1)
        if int(batch.err.item()) != 0:
            raise RuntimeError(f"device error bits {int(batch.err.item())} on {name}")
        out.append(row)
        del batch, flush, events
        torch.cuda.empty_cache()
    return out


def run_ours(args):
    import torch

    import kv_norm_rope_gb300 as k

    rank, world, local_rank = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    lib = k.lib()
    wl = rank_workload(configs.WORKLOADS[args.workload], rank)
    if args.tokens:
        if not 0 < args.tokens <= wl.T:
            raise SystemExit(f"--tokens must be in [1, {wl.T}]")
        # the first N tokens of the workload (its position and slot rules unchanged)
        wl = dataclasses.replace(wl, T=args.tokens)

    kac_before = known_answer_check() if rank == 0 else "skipped"
    copy_1g = copy_ceiling_gbs(dev, 1 << 30)
    copy_512m = copy_ceiling_gbs(dev, 1 << 29)
    batch = DeviceBatch(wl, dev, args.op, VARIANTS[args.variant], args.hidden)
    wl = batch.wl
    stream = torch.cuda.current_stream(dev)
    fn, call_args = batch.call(lib, stream.cuda_stream)
    for _ in range(args.warmup):
        st = fn(*call_args)
        if st != 0:
            raise RuntimeError(f"launch failed: {k.status_string(st)}")
    torch.cuda.synchronize(dev)
    if int(batch.err.item()) != 0:
        raise RuntimeError(f"device error bits {int(batch.err.item())}")

    sampler = ClockSampler(bus_id_of(local_rank)) if rank == 0 else None
    if sampler:
        sampler.start()
    # a step that moves less than 4x the L2 gets the L2 flushed (a 256 MB write)
    # before its launch, outside the launch's event pair
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if batch.bytes < 4 * (129 << 20) \
        else None
    events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * args.steps)]
    barrier(world)
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for i in range(args.steps):
        if flush is not None:
            flush.fill_(i & 0xFF)
        events[2 * i].record(stream)
        fn(*call_args)
        events[2 * i + 1].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    wall = time.perf_counter() - wall0
    clocks = sampler.stop() if sampler else None
    per_launch = [events[2 * i].elapsed_time(events[2 * i + 1]) / 1e3 for i in range(args.steps)]
    region = events[0].elapsed_time(events[-1]) / 1e3
    step_s = statistics.mean(per_launch) if flush is not None else region / args.steps
    t_step = max_over_ranks(step_s, world, dev)
    total_bytes = sum_over_ranks(float(batch.bytes), world, dev)
    total_tokens = sum_over_ranks(float(wl.T), world, dev)
    mean_launch = statistics.mean(per_launch)

    e2e = None
    if not args.no_e2e and args.op == "fused":
        e2e_gbs, h2d, d2h, e2e_dt, ceil, placement = e2e_run(batch, lib, args.e2e_steps)
        e2e_dt = max_over_ranks(e2e_dt, world, dev)
        hr_gbs, hr_h2d, hr_d2h, hr_dt = e2e_host_resident(batch, lib, args.e2e_steps)
        hr_dt = max_over_ranks(hr_dt, world, dev)
        copies = {"value": round(total_bytes / e2e_dt / 1e9, 2), "unit": "GB/s",
                  "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                  "ms_per_step": round(e2e_dt * 1e3, 3), "chunks": 16,
                  "link_gbs": round((h2d + d2h) / e2e_dt / 1e9, 1),
                  "how": "pinned host memory (separate input and output buffers) copied to and "
                         "from device buffers double-buffered by step; H2D and D2H copies overlap "
                         "across chunks and steps"}
        host = {"value": round(total_bytes / hr_dt / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": int(hr_h2d), "d2h_bytes_per_step": int(hr_d2h),
                "ms_per_step": round(hr_dt * 1e3, 3),
                "link_gbs": round((hr_h2d + hr_d2h) / hr_dt / 1e9, 1),
                "how": "every per-token buffer (q in place, kv, positions, slots, cache) in "
                       "pinned host memory, read and written by the kernel over NVLink-C2C"}
        # the user's choice: the faster of the two ways through the C ABI
        best = host if hr_dt <= e2e_dt else copies
        e2e = {"value": best["value"], "unit": "GB/s",
               "h2d_bytes_per_step": best["h2d_bytes_per_step"],
               "d2h_bytes_per_step": best["d2h_bytes_per_step"],
               "tokens_per_s": round(total_tokens / min(e2e_dt, hr_dt), 1),
               "ms_per_step": best["ms_per_step"],
               "mode": "host_resident" if best is host else "copies",
               "host_resident": host, "copies": copies,
               "link_ceilings": ceil,
               "frac_of_both_ways_ceiling": round(best["link_gbs"] / ceil["both_gbs"], 4)
               if ceil["both_gbs"] else None,
               "placement": placement}
    graph_us = graph_device_us(batch, lib, dev, flush) if flush is not None else None
    warm_us = graph_warm_us(batch, lib, dev) if flush is not None else None
    copy_us = graph_copy_us(batch.bytes, dev, flush) if flush is not None else None
    kac_after = known_answer_check() if rank == 0 else "skipped"
    if rank != 0:
        return 0

    peak, peak_kind = measured_peaks()
    achieved = batch.bytes / mean_launch / 1e9
    value = total_bytes / t_step / 1e9
    plan = k.launch_plan(wl.T, wl.H, torch.cuda.get_device_properties(dev).multi_processor_count,
                         3)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_step * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": wl.name.split("@")[0], "op": args.op, "T": wl.T, "H": wl.H,
                   "store": wl.store,
                   "num_blocks": wl.num_blocks, "block_size": wl.block_size,
                   "bytes_per_step": batch.bytes,
                   "l2": "flushed before every launch (256 MB write)" if flush is not None
                   else f"inputs larger than L2 ({batch.bytes / 1e9:.2f} GB per step)",
                   "io": IO_OF_OP[args.op],
                   **({"hidden": args.hidden} if args.op == "mxfp8" else {}),
                   "variant": (args.variant if args.variant != "auto" else
                               {k.VARIANT_STREAM: "stream", k.VARIANT_SMALL: "small",
                                k.VARIANT_HALF: "half"}[plan.variant])
                   if args.op in ("fused", "prenorm", "kv_only") else "n/a",
                   "parallelism": f"dp{world}" if world > 1 else "single"},
        "tokens_per_s": round(total_tokens / t_step, 1),
        "frac_of_copy_ceiling": round(value / world / copy_1g, 4),
        "self_check": self_check(value / world, achieved, copy_1g, copy_512m),
        "frac_of_8tbs": round(value / world / NOMINAL_HBM_GBS, 4),
        "copy_ceiling_gbs": {"1GiB": round(copy_1g, 1), "512MiB": round(copy_512m, 1)},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": profiled_traffic(wl.name.split("@")[0])
                     if args.op == "fused" and not args.tokens else None,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "launch_ms_mean": round(mean_launch * 1e3, 4),
                     "launch_ms_median": round(statistics.median(per_launch) * 1e3, 4)},
        "graph": None if graph_us is None else {
            "us_per_launch": round(graph_us, 3),
            "GB/s": round(batch.bytes / graph_us / 1e3, 1),
            "how": "CUDA graph of 50 (L2 flush, launch) pairs minus a graph of the 50 flushes: "
                   "the kernel's device time without the host launch latency that a single "
                   "event-timed launch after a flush includes",
            "warm_us_per_launch": round(warm_us, 3),
            "warm_how": "CUDA graph of 50 launches back to back, no flush: inputs that fit stay "
                        "in L2 and no flush's dirty lines are written back during the launch",
            "same_size_copy_us": {k_: round(v_, 3) for k_, v_ in copy_us.items()},
            "frac_of_same_size_copy": round(min(copy_us.values()) / graph_us, 4),
            "copy_how": "half the step's bytes moved between two device buffers (the same bytes "
                        "read plus written) by a memcpy and by an elementwise kernel, timed the "
                        "same way: what moving them costs at this size; the fraction is against "
                        "the faster"},
        "gpu_launches": args.steps,
        "ms_per_step_note": "mean launch time (L2 flushed between launches)" if flush is not None
        else "timed region / steps",
        "clocks": clocks,
        "wall_s_timed": round(wall, 3),
        "known_answer": {"before": kac_before, "after": kac_after},
    }
    if e2e is not None:
        line["e2e"] = e2e
    if not args.no_cpu_baseline and args.op == "fused":
        line["cpu_baseline"] = cpu_baseline(configs.WORKLOADS[args.workload], args.cpu_seconds)
    # the other configurations of the operator, when this is the default stress run; last,
    # and kept out of the headline if anything in them fails
    if (world == 1 and args.op == "fused" and args.workload == "stress" and not args.tokens
            and args.variant == "auto" and not args.no_other_configs):
        try:
            line["other_configs"] = other_configs(
                lib, dev, ("prefill", "bf16_store", "decode", "tiny"), min(args.steps, 30),
                args.warmup)
        except Exception as e:  # noqa: BLE001 - reported in the line, not fatal to it
            line["other_configs"] = {"error": f"{type(e).__name__}: {e}"[:300]}
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(configs.WORKLOADS), default="stress")
    ap.add_argument("--variant", choices=sorted(VARIANTS), default="auto",
                    help="launch variant of the fused op (default: the library's choice)")
    ap.add_argument("--op", choices=OPS, default="fused",
                    help="fused (default); prenorm: KV arrives normalised; kv_only: no q; "
                         "gather: read the FP8 cache back out; mxfp8: residual add + Gemma "
                         "RMSNorm + MXFP8 of [T, 7168] activation rows; indexer: indexer-K "
                         "quant-insert of [T, 128] rows; indexer_gather: read them back out")
    ap.add_argument("--hidden", type=int, default=MXFP8_HIDDEN,
                    help="row width of --op mxfp8 (a multiple of 128 up to 16384)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="run only the first N tokens of the workload (smaller profiling cases)")
    ap.add_argument("--e2e-steps", type=int, default=6)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="skip the other workloads that the default stress run also times")
    ap.add_argument("--cpu-seconds", type=float, default=2.0,
                    help="wall seconds of oracle work on all host cores for cpu_baseline")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
