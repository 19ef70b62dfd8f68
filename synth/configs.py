"""The five synthetic workloads and a generic small-case recipe.

Sizes follow the operator's statement of the problem: head_dim 512 (rope on the
trailing 64 dims, GPT-J interleaved pairs, theta 10000), q [T, H, 512] bf16,
one 512-wide latent KV row per token, a paged cache of num_blocks x 64 slots.
Each workload fixes how positions and slot_mapping are drawn; values are drawn
by ``synth.normal_bf16`` from the workload's seed.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

import synth

HEAD_DIM = 512
EPS = 1e-6
THETA = 10000.0


@dataclass(frozen=True)
class Workload:
    name: str
    T: int                  # tokens
    H: int                  # q heads
    store: str              # "fp8" (448 E4M3 + 7 UE8M0 + 64 bf16) or "bf16" (512 bf16)
    max_position: int       # rows of the cos/sin table
    num_blocks: int
    block_size: int
    seed: int
    tail_frac: float = 0.0  # share of q/kv elements multiplied by tail_mult
    tail_mult: float = 1.0
    eps: float = EPS

    @property
    def num_slots(self) -> int:
        return self.num_blocks * self.block_size

    def positions(self) -> np.ndarray:
        return _POSITIONS[self.name](self)

    def slot_mapping(self) -> np.ndarray:
        return _SLOTS[self.name](self)


TINY = Workload("tiny", 16, 8, "fp8", 4096, 4, 64, seed=0)
DECODE = Workload("decode", 256, 64, "fp8", 131072, 1024, 64, seed=1)
PREFILL = Workload("prefill", 32768, 64, "fp8", 4096, 1024, 64, seed=2)
BF16_STORE = Workload("bf16_store", 32768, 128, "bf16", 65536, 1024, 64, seed=3)
STRESS = Workload("stress", 131072, 128, "fp8", 4096, 2048, 64, seed=4,
                  tail_frac=1e-3, tail_mult=100.0)

WORKLOADS = {w.name: w for w in (TINY, DECODE, PREFILL, BF16_STORE, STRESS)}


def generic(T: int, H: int, store: str = "fp8", seed: int = 100, max_position: int = 4096,
            skip_frac: float = 0.1, tail_frac: float = 0.0, tail_mult: float = 1.0) -> Workload:
    """A small case: uniform positions, distinct random slots, skip_frac of tokens at -1."""
    blocks = max(1, -(-(2 * max(T, 1)) // 64))
    name = f"generic_T{T}_H{H}_{store}_s{seed}_k{skip_frac}"
    w = Workload(name, T, H, store, max_position, blocks, 64, seed, tail_frac, tail_mult)
    _POSITIONS[name] = lambda w: synth.uniform_int(w.T, w.max_position, w.seed, synth.TID_POS)
    _SLOTS[name] = lambda w: _random_slots(w, int(round(skip_frac * w.T)))
    return w


def _random_slots(w: Workload, n_skip: int) -> np.ndarray:
    slots = synth.permutation(w.num_slots, w.seed, synth.TID_SLOT)[: w.T].copy()
    if n_skip:
        skip = synth.permutation(w.T, w.seed, synth.TID_SKIP)[:n_skip]
        slots[skip] = -1
    return slots


def _request_positions(w: Workload, req_len: int = 4096) -> np.ndarray:
    return (np.arange(w.T, dtype=np.int64) % req_len)


def _request_slots(w: Workload, req_len: int = 4096) -> np.ndarray:
    n_chunks = w.num_slots // req_len
    chunks = synth.permutation(n_chunks, w.seed, synth.TID_SLOT)
    t = np.arange(w.T, dtype=np.int64)
    return chunks[t // req_len] * req_len + t % req_len


_POSITIONS = {
    "tiny": lambda w: synth.uniform_int(w.T, 4096, w.seed, synth.TID_POS),
    "decode": lambda w: synth.uniform_int(w.T, 131072, w.seed, synth.TID_POS),
    "prefill": _request_positions,
    "bf16_store": lambda w: synth.uniform_int(w.T, 65536, w.seed, synth.TID_POS),
    "stress": _request_positions,
}

_SLOTS = {
    "tiny": lambda w: _random_slots(w, 2),
    "decode": lambda w: _random_slots(w, int(round(0.1 * w.T))),
    "prefill": _request_slots,
    "bf16_store": lambda w: _random_slots(w, 0),
    "stress": _request_slots,
}


def q_bits(w: Workload, t0: int = 0, t1: int | None = None, out_ptr: int | None = None,
           n_threads: int = 0):
    """bf16 bits of q[t0:t1] (flattened [t1-t0, H, 512])."""
    t1 = w.T if t1 is None else t1
    per = w.H * HEAD_DIM
    return synth.normal_bf16((t1 - t0) * per, w.seed, synth.TID_Q, start=t0 * per,
                             tail_frac=w.tail_frac, tail_mult=w.tail_mult,
                             tail_id=synth.TID_Q_TAIL, out_ptr=out_ptr, n_threads=n_threads)


def kv_bits(w: Workload, t0: int = 0, t1: int | None = None, out_ptr: int | None = None):
    t1 = w.T if t1 is None else t1
    return synth.normal_bf16((t1 - t0) * HEAD_DIM, w.seed, synth.TID_KV, start=t0 * HEAD_DIM,
                             tail_frac=w.tail_frac, tail_mult=w.tail_mult,
                             tail_id=synth.TID_KV_TAIL, out_ptr=out_ptr)


INDEXER_DIM = 128


def indexer_k_bits(w: Workload, t0: int = 0, t1: int | None = None) -> np.ndarray:
    """bf16 bits of the indexer K rows k[t0:t1] (flattened [t1-t0, 128]), with the
    workload's tail share and multiplier."""
    t1 = w.T if t1 is None else t1
    return synth.normal_bf16((t1 - t0) * INDEXER_DIM, w.seed, synth.TID_IDX_K, start=t0 * INDEXER_DIM,
                             tail_frac=w.tail_frac, tail_mult=w.tail_mult,
                             tail_id=synth.TID_IDX_K_TAIL)


def indexer_cache_bytes(w: Workload) -> int:
    return w.num_slots * (INDEXER_DIM + 4)


def weight_bits(w: Workload) -> np.ndarray:
    return synth.normal_bf16(HEAD_DIM, w.seed, synth.TID_W, mean=1.0, std=0.1)


def cos_sin(w: Workload) -> np.ndarray:
    return synth.cos_sin_table(w.max_position, 64, THETA)


def cache_bytes(w: Workload) -> int:
    row = 584 if w.store == "fp8" else 1024
    return w.num_slots * row


def algorithmic_bytes(w: Workload, positions: np.ndarray | None = None,
                      slots: np.ndarray | None = None) -> int:
    """Bytes the operator must move once: q read+write, kv read, metadata,
    valid cache rows, the distinct cos/sin rows touched, the weight."""
    positions = w.positions() if positions is None else positions
    slots = w.slot_mapping() if slots is None else slots
    valid = int((slots >= 0).sum())
    row = 584 if w.store == "fp8" else 1024
    uniq = int(np.unique(positions).size)
    return (w.T * (2 * w.H * HEAD_DIM * 2 + HEAD_DIM * 2 + 16) + valid * row
            + uniq * 256 + HEAD_DIM * 2)
