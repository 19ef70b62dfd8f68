"""Seeded synthetic inputs for the fused q-norm / RoPE / KV-quant / paged-insert step.

This module draws numbers and nothing else: it holds none of the operator's
arithmetic, and neither the CPU oracle nor the CUDA library imports it.  The
tests, the benchmark and the smoke check call it to build the inputs that both
sides then receive.  Every tensor is a pure function of (seed, tensor id,
element index) -- see ``synth.c`` -- so a token range can be regenerated on
its own (the full-size parity tests regenerate only sampled tokens on the host).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "libsynth.so")

# tensor ids of the counter-based streams
TID_Q, TID_KV, TID_W, TID_POS, TID_SLOT, TID_POISON, TID_SKIP = 1, 2, 3, 4, 5, 7, 8
TID_Q_TAIL, TID_KV_TAIL = 9, 10
TID_IDX_K, TID_IDX_K_TAIL = 11, 12

_lib = None


def build(force: bool = False) -> str:
    """Compile ``synth.c`` into ``libsynth.so`` next to it (gcc, no CUDA)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, i32, dbl, vp = ctypes.c_uint64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        lib.synth_normal_bf16.argtypes = [vp, u64, u64, u64, u64, dbl, dbl, dbl, dbl, u64, i32]
        lib.synth_normal_bf16.restype = None
        lib.synth_u64.argtypes = [vp, u64, u64, u64, u64]
        lib.synth_u64.restype = None
        lib.synth_bytes.argtypes = [vp, u64, u64, u64, i32]
        lib.synth_bytes.restype = None
        _lib = lib
    return _lib


def normal_bf16(count: int, seed: int, tensor_id: int, start: int = 0, mean: float = 0.0,
                std: float = 1.0, tail_frac: float = 0.0, tail_mult: float = 1.0,
                tail_id: int = 0, out_ptr: int | None = None, n_threads: int = 0):
    """bf16 bit patterns of elements ``start .. start+count`` of an N(mean, std) tensor.

    Returns a uint16 numpy array, or fills ``out_ptr`` (a host address with room
    for ``count`` uint16) and returns None.
    """
    lib = _load()
    arr = None
    if out_ptr is None:
        arr = np.empty(count, dtype=np.uint16)
        out_ptr = arr.ctypes.data
    if count:
        lib.synth_normal_bf16(out_ptr, seed, tensor_id, start, count, mean, std,
                              tail_frac, tail_mult, tail_id, n_threads)
    return arr


def u64(seed: int, tensor_id: int, start: int, count: int) -> np.ndarray:
    out = np.empty(count, dtype=np.uint64)
    if count:
        _load().synth_u64(out.ctypes.data, seed, tensor_id, start, count)
    return out


def poison_bytes(count: int, seed: int, out_ptr: int | None = None, n_threads: int = 0):
    """Pseudo-random bytes used as the pre-image of output buffers."""
    arr = None
    if out_ptr is None:
        arr = np.empty(count, dtype=np.uint8)
        out_ptr = arr.ctypes.data
    if count:
        _load().synth_bytes(out_ptr, seed, TID_POISON, count, n_threads)
    return arr


def permutation(n: int, seed: int, tensor_id: int) -> np.ndarray:
    """A seeded permutation of range(n): indices sorted by their 64-bit keys."""
    keys = u64(seed, tensor_id, 0, n)
    return np.argsort(keys, kind="stable").astype(np.int64)


def uniform_int(n: int, high: int, seed: int, tensor_id: int) -> np.ndarray:
    """n integers in [0, high): key mod high (high <= 2^20 keeps the bias below 2^-44)."""
    return (u64(seed, tensor_id, 0, n) % np.uint64(high)).astype(np.int64)


def cos_sin_table(max_position: int, rope_dim: int = 64, theta: float = 10000.0) -> np.ndarray:
    """fp32 [max_position, rope_dim]: cos of the rope_dim/2 angles, then their sin.

    Angle of pair i at position p is p * theta^(-2i/rope_dim); computed in
    double, each entry rounded once to fp32.  Both sides read these same bits.
    """
    half = rope_dim // 2
    inv_freq = theta ** (-(2.0 * np.arange(half, dtype=np.float64)) / rope_dim)
    ang = np.arange(max_position, dtype=np.float64)[:, None] * inv_freq[None, :]
    out = np.empty((max_position, rope_dim), dtype=np.float32)
    out[:, :half] = np.cos(ang)
    out[:, half:] = np.sin(ang)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (for plotting / statistics)."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
