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
    q: np.ndarray          # uint16 [len(q_tokens), H, 512]
    cache: np.ndarray      # uint8 cache image
    err: int


def run_gpu(inp: Inputs, variant: int = 0, q_tokens: np.ndarray | None = None,
            store: str | None = None, device: str = "cuda:0", kv_norm: bool = True) -> GpuResult:
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
    if q_tokens is None:
        q_tokens = np.arange(wl.T, dtype=np.int64)
        q_host = q.cpu().view(torch.int16).numpy().view(np.uint16).reshape(wl.T, wl.H, 512)
    else:
        idx = torch.from_numpy(q_tokens).to(dev)
        q_host = q.index_select(0, idx).cpu().view(torch.int16).numpy().view(np.uint16)
    out = GpuResult(q_tokens, q_host, cache.cpu().numpy(), int(err.item()))
    del q, kv, cache
    return out


def sample_tokens(T: int, n: int, seed: int) -> np.ndarray:
    """First and last 8 tokens plus a seeded random sample, sorted and distinct."""
    if T <= n:
        return np.arange(T, dtype=np.int64)
    ends = np.concatenate([np.arange(8), np.arange(T - 8, T)])
    rnd = synth.permutation(T, seed, 11)[: n - 16]
    return np.unique(np.concatenate([ends, rnd])).astype(np.int64)


def run_oracle(inp: Inputs, q_tokens: np.ndarray | None = None, store: str | None = None,
               n_threads: int = 0, kv_norm: bool = True):
    """(q rows of q_tokens after the step, cache image, error bits) from the oracle."""
    wl = inp.wl
    store = store or wl.store
    cache = inp.poison.copy()
    # KV rows of every token: the whole cache image
    err = oracle.qnorm_rope_kv_insert(store, None, inp.kv, inp.w, inp.positions, inp.cos_sin,
                                      inp.slots, cache, wl.num_blocks, wl.block_size, wl.eps,
                                      n_threads=n_threads, kv_norm=kv_norm)
    if q_tokens is None:
        q_tokens = np.arange(wl.T, dtype=np.int64)
    q = np.ascontiguousarray(inp.q[q_tokens])
    if wl.H == 0:
        return q, cache, err
    no_slots = np.full(q_tokens.size, -1, dtype=np.int64)
    err |= oracle.qnorm_rope_kv_insert(store, q, None, inp.w, inp.positions[q_tokens], inp.cos_sin,
                                       no_slots, None, wl.num_blocks, wl.block_size, wl.eps,
                                       n_threads=n_threads)
    return q, cache, err


def compare_results(inp: Inputs, gpu: GpuResult, ref_q: np.ndarray, ref_cache: np.ndarray,
                    store: str | None = None) -> compare.Report:
    wl = inp.wl
    store = store or wl.store
    rep = compare.Report()
    valid_pos = (inp.positions[gpu.q_tokens] >= 0) & (inp.positions[gpu.q_tokens] < wl.max_position)
    # q of tokens with an out-of-range position must be untouched
    if (~valid_pos).any():
        if not np.array_equal(gpu.q[~valid_pos], inp.q[gpu.q_tokens][~valid_pos]):
            rep.fail("q rows of tokens with out-of-range positions changed")
    compare.compare_bf16(gpu.q[valid_pos], ref_q[valid_pos], "q", rep)
    if store == "fp8":
        compare.compare_fp8_cache(gpu.cache, ref_cache, inp.poison, inp.slots[
            (inp.positions >= 0) & (inp.positions < wl.max_position)], wl.num_blocks,
            wl.block_size, rep)
    else:
        compare.compare_bf16_cache(gpu.cache, ref_cache, inp.poison, inp.slots[
            (inp.positions >= 0) & (inp.positions < wl.max_position)], wl.num_slots, rep)
    return rep


def check(wl: Workload, variant: int = 0, n_sample: int | None = None, inp: Inputs | None = None,
          store: str | None = None, kv_norm: bool = True) -> compare.Report:
    """Full round trip for one workload; q compared on all tokens or on a sample."""
    inp = make_inputs(wl) if inp is None else inp
    q_tokens = None if n_sample is None else sample_tokens(wl.T, n_sample, wl.seed + 5)
    gpu = run_gpu(inp, variant, q_tokens, store, kv_norm=kv_norm)
    ref_q, ref_cache, ref_err = run_oracle(inp, gpu.q_tokens, store, kv_norm=kv_norm)
    rep = compare_results(inp, gpu, ref_q, ref_cache, store)
    if gpu.err != ref_err:
        rep.fail(f"device error bits {gpu.err} != oracle {ref_err}")
    return rep
