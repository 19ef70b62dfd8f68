"""Run one workload through the CUDA library and through the oracle, and compare.

Test infrastructure shared by the GPU tests, the smoke check and the benchmark's
known-answer check.  Inputs come from ``synth`` (seeded, counter-based); the
GPU side goes through the C ABI binding ``kv_norm_rope_gb300``; the reference
side is ``oracle``.  Nothing here computes any part of the operator.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

import oracle
import synth
from oracle import compare
from synth import configs
from synth.configs import Workload


@dataclass
class Inputs:
    wl: Workload
    q: np.ndarray          # uint16 [T, H, 512]
    kv: np.ndarray         # uint16 [T, 512]
    w: np.ndarray          # uint16 [512]
    positions: np.ndarray  # int64 [T]
    slots: np.ndarray      # int64 [T]
    cos_sin: np.ndarray    # float32 [max_position, 64]
    poison: np.ndarray     # uint8 pre-image of the cache


def make_inputs(wl: Workload, positions=None, slots=None) -> Inputs:
    q = np.empty(wl.T * wl.H * 512, dtype=np.uint16)
    if q.size:
        configs.q_bits(wl, out_ptr=q.ctypes.data)
    kv = configs.kv_bits(wl)
    return Inputs(wl, q.reshape(wl.T, wl.H, 512), kv.reshape(wl.T, 512), configs.weight_bits(wl),
                  wl.positions() if positions is None else np.asarray(positions, np.int64),
                  wl.slot_mapping() if slots is None else np.asarray(slots, np.int64),
                  configs.cos_sin(wl), synth.poison_bytes(configs.cache_bytes(wl), seed=wl.seed + 77))


@dataclass
class GpuResult:
    q_tokens: np.ndarray   # token indices whose q rows were copied back
    q: np.ndarray          # uint16 [len(q_tokens), H, 512] (None when q_dev is kept instead)
    cache: np.ndarray      # uint8 cache image
    err: int
    q_dev: object = None   # the whole q tensor still on the device (run_gpu(keep_q=True))


def _q_host(q_dev, t0: int, t1: int) -> np.ndarray:
    import torch
    return q_dev[t0:t1].cpu().view(torch.int16).numpy().view(np.uint16)


def run_gpu(inp: Inputs, variant: int = 0, q_tokens: np.ndarray | None = None,
            store: str | None = None, device: str = "cuda:0", kv_norm: bool = True,
            keep_q: bool = False) -> GpuResult:
    """One call of the general entry point on fresh device copies of the inputs.
    keep_q leaves q on the device (GpuResult.q_dev) for a chunked comparison."""
    import torch

    import kv_norm_rope_gb300 as k

    wl = inp.wl
    store = store or wl.store
    dev = torch.device(device)
    q = torch.from_numpy(inp.q.view(np.int16)).view(torch.bfloat16).to(dev)
    kv = torch.from_numpy(inp.kv.view(np.int16)).view(torch.bfloat16).to(dev)
    w = torch.from_numpy(inp.w.view(np.int16)).view(torch.bfloat16).to(dev)
    pos = torch.from_numpy(inp.positions).to(dev)
    sl = torch.from_numpy(inp.slots).to(dev)
    cs = torch.from_numpy(inp.cos_sin).to(dev)
    cache = torch.from_numpy(inp.poison).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    k.insert(k.STORE_FP8 if store == "fp8" else k.STORE_BF16, q if wl.H > 0 else None, kv, w,
             pos, cs, sl, cache, wl.num_blocks, wl.block_size, wl.eps, device_error=err,
             variant=variant, num_heads=wl.H, kv_norm=kv_norm)
    torch.cuda.synchronize(dev)
    if keep_q:
        out = GpuResult(np.arange(wl.T, dtype=np.int64), None, cache.cpu().numpy(),
                        int(err.item()), q_dev=q)
        del kv, cache
        return out
    if q_tokens is None:
        q_tokens = np.arange(wl.T, dtype=np.int64)
        q_host = _q_host(q, 0, wl.T)
    else:
        idx = torch.from_numpy(q_tokens).to(dev)
        q_host = q.index_select(0, idx).cpu().view(torch.int16).numpy().view(np.uint16)
    out = GpuResult(q_tokens, q_host, cache.cpu().numpy(), int(err.item()))
    del q, kv, cache
    return out


def run_oracle_cache(inp: Inputs, store: str | None = None, n_threads: int = 0,
                     kv_norm: bool = True):
    """(cache image, error bits) of every token's KV row, from the oracle."""
    wl = inp.wl
    cache = inp.poison.copy()
    err = oracle.qnorm_rope_kv_insert(store or wl.store, None, inp.kv, inp.w, inp.positions,
                                      inp.cos_sin, inp.slots, cache, wl.num_blocks,
                                      wl.block_size, wl.eps, n_threads=n_threads,
                                      kv_norm=kv_norm)
    return cache, err


def run_oracle_q(inp: Inputs, q_tokens: np.ndarray, n_threads: int = 0):
    """(q rows of q_tokens after the step, error bits of their positions), from the oracle."""
    wl = inp.wl
    q = np.ascontiguousarray(inp.q[q_tokens])
    if wl.H == 0:
        return q, 0
    no_slots = np.full(q_tokens.size, -1, dtype=np.int64)
    err = oracle.qnorm_rope_kv_insert(wl.store, q, None, inp.w, inp.positions[q_tokens],
                                      inp.cos_sin, no_slots, None, wl.num_blocks, wl.block_size,
                                      wl.eps, n_threads=n_threads)
    return q, err


def run_oracle(inp: Inputs, q_tokens: np.ndarray | None = None, store: str | None = None,
               n_threads: int = 0, kv_norm: bool = True):
    """(q rows of q_tokens after the step, cache image, error bits) from the oracle."""
    cache, err = run_oracle_cache(inp, store, n_threads, kv_norm)
    if q_tokens is None:
        q_tokens = np.arange(inp.wl.T, dtype=np.int64)
    q, qerr = run_oracle_q(inp, q_tokens, n_threads)
    return q, cache, err | qerr


def compare_q(inp: Inputs, q_tokens: np.ndarray, gpu_q: np.ndarray, ref_q: np.ndarray,
              rep: compare.Report) -> compare.Report:
    """q rows of q_tokens: within one bf16 ulp of the oracle; rows of tokens whose
    position is outside the table must be the untouched inputs."""
    wl = inp.wl
    pos = inp.positions[q_tokens]
    valid_pos = (pos >= 0) & (pos < wl.max_position)
    if (~valid_pos).any():
        if not np.array_equal(gpu_q[~valid_pos], inp.q[q_tokens][~valid_pos]):
            rep.fail("q rows of tokens with out-of-range positions changed")
    compare.compare_bf16(gpu_q[valid_pos], ref_q[valid_pos], "q", rep)
    rep.q_rows += int(gpu_q.shape[0]) * int(gpu_q.shape[1])
    return rep


def compare_cache(inp: Inputs, gpu_cache: np.ndarray, ref_cache: np.ndarray,
                  store: str | None = None, rep: compare.Report | None = None) -> compare.Report:
    wl = inp.wl
    rep = compare.Report() if rep is None else rep
    if (store or wl.store) == "fp8":
        compare.compare_fp8_cache(gpu_cache, ref_cache, inp.poison, inp.slots, inp.positions,
                                  wl.max_position, wl.num_blocks, wl.block_size, rep)
    else:
        compare.compare_bf16_cache(gpu_cache, ref_cache, inp.poison, inp.slots, inp.positions,
                                   wl.max_position, wl.num_slots, rep)
    return rep


def compare_results(inp: Inputs, gpu: GpuResult, ref_q: np.ndarray, ref_cache: np.ndarray,
                    store: str | None = None) -> compare.Report:
    rep = compare.Report()
    compare_q(inp, gpu.q_tokens, gpu.q, ref_q, rep)
    return compare_cache(inp, gpu.cache, ref_cache, store, rep)


# q elements downloaded and checked against the oracle at a time (512 MiB of bf16)
Q_CHUNK_ELEMS = 1 << 28


def check(wl: Workload, variant: int = 0, inp: Inputs | None = None, store: str | None = None,
          kv_norm: bool = True) -> compare.Report:
    """Full round trip for one workload: every cache byte and every token's q rows
    compared with the oracle.  The GPU runs the whole batch in one call; its q is
    then copied back and checked in token chunks (tokens are independent, so the
    oracle's chunks are exact)."""
    inp = make_inputs(wl) if inp is None else inp
    gpu = run_gpu(inp, variant, store=store, kv_norm=kv_norm, keep_q=True)
    ref_cache, ref_err = run_oracle_cache(inp, store, kv_norm=kv_norm)
    rep = compare_cache(inp, gpu.cache, ref_cache, store)
    if wl.H > 0:
        step = max(1, Q_CHUNK_ELEMS // (wl.H * 512))
        for t0 in range(0, wl.T, step):
            t1 = min(wl.T, t0 + step)
            toks = np.arange(t0, t1, dtype=np.int64)
            ref_q, qerr = run_oracle_q(inp, toks)
            ref_err |= qerr
            compare_q(inp, toks, _q_host(gpu.q_dev, t0, t1), ref_q, rep)
    gpu.q_dev = None
    if gpu.err != ref_err:
        rep.fail(f"device error bits {gpu.err} != oracle {ref_err}")
    return rep
