"""CPU oracle (fp64, plain C) of the fused q-norm / RoPE / KV-quant / paged-insert step.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline / reference arm are the only callers.  It shares no code with the CUDA
library and imports nothing from it.  See ``dsv4_oracle.c`` for the definition
it follows and the passages it cites.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsv4_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libdsv4oracle.so")

ERR_SLOT_RANGE = 1
ERR_POS_RANGE = 2
FP8_SLOT_BYTES = 584
FP8_DATA_BYTES = 576
INDEXER_DIM = 128
INDEXER_SLOT_BYTES = 132

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, no fast-math, no fp contraction)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
        lib.oracle_qnorm_rope_kv_insert.argtypes = [ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, vp,
                                                    i64, vp, vp,
                                                    i64, i32, i64, i32, f32, ctypes.c_int]
        lib.oracle_qnorm_rope_kv_insert.restype = i32
        lib.oracle_q_values.argtypes = [vp, vp, f32, vp]
        lib.oracle_kv_values.argtypes = [vp, vp, vp, f32, vp]
        lib.oracle_kv_rope_values.argtypes = [vp, vp, vp]
        lib.oracle_fp8_slot.argtypes = [vp, vp, vp]
        for name in ("oracle_bf16_rne_array", "oracle_e4m3_rne_array",
                     "oracle_bf16_value_array", "oracle_ue8m0_exponent_array"):
            getattr(lib, name).argtypes = [vp, vp, i64]
        lib.oracle_e4m3_value_array.argtypes = [vp, vp, i64]
        lib.oracle_dequant_gather.argtypes = [vp, i64, i32, vp, i64, vp]
        lib.oracle_dequant_gather.restype = i32
        lib.oracle_indexer_k_quant_insert.argtypes = [vp, vp, vp, i64, i32, i64]
        lib.oracle_indexer_k_quant_insert.restype = i32
        lib.oracle_indexer_k_gather.argtypes = [vp, i64, i32, vp, i64, vp, vp]
        lib.oracle_indexer_k_gather.restype = i32
        lib.oracle_gemma_rmsnorm_mxfp8.argtypes = [vp, vp, vp, i64, i64, f32, vp, vp, vp]
        lib.oracle_ue8m0_of_f32.argtypes = [f32]
        lib.oracle_ue8m0_of_f32.restype = ctypes.c_int
        lib.oracle_ue8m0_inverse.argtypes = [ctypes.c_int]
        lib.oracle_ue8m0_inverse.restype = ctypes.c_double
        lib.oracle_swizzled_scale_offset.argtypes = [i64, i64, i64]
        lib.oracle_swizzled_scale_offset.restype = i64
        lib.oracle_mxfp8_scale_bytes.argtypes = [i64, i64]
        lib.oracle_mxfp8_scale_bytes.restype = i64
        lib.oracle_ue8m0_exponent.argtypes = [ctypes.c_double]
        lib.oracle_ue8m0_exponent.restype = ctypes.c_int
        _lib = lib
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def qnorm_rope_kv_insert(store: str, q: np.ndarray | None, kv: np.ndarray | None, w: np.ndarray,
                         positions: np.ndarray, cos_sin: np.ndarray, slot_mapping: np.ndarray,
                         cache: np.ndarray, num_blocks: int, block_size: int, eps: float,
                         H: int | None = None, n_threads: int = 0, kv_norm: bool = True) -> int:
    """Run the oracle.  ``q`` (uint16 bf16 bits [T,H,512], or None) and ``cache``
    (uint8, poisoned pre-image) are modified in place.  ``kv_norm`` False takes the
    KV rows as already normalised (rotation only; ``w`` and ``eps`` unused for
    them).  Returns the error bits."""
    lib = _load()
    T = int(positions.shape[0])
    if q is not None:
        assert q.dtype == np.uint16 and q.flags.c_contiguous and q.size == T * q.shape[-2] * 512
        H = q.shape[-2] if H is None else H
    else:
        H = 0
    row = FP8_SLOT_BYTES if store == "fp8" else 1024
    if cache is not None:
        assert cache.dtype == np.uint8 and cache.flags.c_contiguous
        assert cache.size == num_blocks * block_size * row
    else:
        assert kv is None, "a cache image is needed when kv rows are given"

    w = _c(np.zeros(512, np.uint16) if w is None else w, np.uint16)
    pos = _c(positions, np.int64)
    cs = _c(cos_sin, np.float32)
    sl = _c(slot_mapping, np.int64)
    kvp = None
    if kv is not None:
        kv = _c(kv, np.uint16)
        kvp = kv.ctypes.data
    return int(lib.oracle_qnorm_rope_kv_insert(
        1 if store == "bf16" else 0, 1 if kv_norm else 0,
        q.ctypes.data if q is not None else None, kvp, w.ctypes.data,
        pos.ctypes.data, cs.ctypes.data, cs.shape[0], sl.ctypes.data,
        cache.ctypes.data if cache is not None else None,
        num_blocks, block_size, T, H, eps, n_threads))


def q_values(x: np.ndarray, cs_row: np.ndarray, eps: float) -> np.ndarray:
    """fp64 normalised + rotated q head (before bf16 rounding)."""
    x = _c(x, np.uint16)
    cs = _c(cs_row, np.float32)
    out = np.empty(512, dtype=np.float64)
    _load().oracle_q_values(x.ctypes.data, cs.ctypes.data, eps, out.ctypes.data)
    return out


def kv_values(x: np.ndarray, w: np.ndarray, cs_row: np.ndarray, eps: float) -> np.ndarray:
    """fp64 normalised, weighted, rotated KV row (before rounding/quantisation)."""
    x = _c(x, np.uint16)
    w = _c(np.zeros(512, np.uint16) if w is None else w, np.uint16)
    cs = _c(cs_row, np.float32)
    out = np.empty(512, dtype=np.float64)
    _load().oracle_kv_values(x.ctypes.data, w.ctypes.data, cs.ctypes.data, eps, out.ctypes.data)
    return out


def kv_rope_values(x: np.ndarray, cs_row: np.ndarray) -> np.ndarray:
    """fp64 rotated KV row that arrives normalised (no norm, no weight)."""
    x = _c(x, np.uint16)
    cs = _c(cs_row, np.float32)
    out = np.empty(512, dtype=np.float64)
    _load().oracle_kv_rope_values(x.ctypes.data, cs.ctypes.data, out.ctypes.data)
    return out


def fp8_slot(v: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """(576 data bytes, 8 scale bytes) of one slot from fp64 values."""
    v = _c(v, np.float64)
    data = np.empty(576, dtype=np.uint8)
    scale = np.empty(8, dtype=np.uint8)
    _load().oracle_fp8_slot(v.ctypes.data, data.ctypes.data, scale.ctypes.data)
    return data, scale


def bf16_rne(x: np.ndarray) -> np.ndarray:
    x = _c(x, np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_bf16_rne_array(x.ctypes.data, out.ctypes.data, x.size)
    return out


def e4m3_rne(x: np.ndarray) -> np.ndarray:
    x = _c(x, np.float64)
    out = np.empty(x.shape, dtype=np.uint8)
    _load().oracle_e4m3_rne_array(x.ctypes.data, out.ctypes.data, x.size)
    return out


def bf16_value(b: np.ndarray) -> np.ndarray:
    b = _c(b, np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_bf16_value_array(b.ctypes.data, out.ctypes.data, b.size)
    return out


def ue8m0_exponent(amax: np.ndarray) -> np.ndarray:
    a = _c(amax, np.float64)
    out = np.empty(a.shape, dtype=np.int32)
    _load().oracle_ue8m0_exponent_array(a.ctypes.data, out.ctypes.data, a.size)
    return out


def e4m3_value(codes: np.ndarray) -> np.ndarray:
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    _load().oracle_e4m3_value_array(c.ctypes.data, out.ctypes.data, c.size)
    return out


def dequant_gather(cache: np.ndarray, num_blocks: int, block_size: int, slots: np.ndarray):
    """(bf16 bits [n, 512], error bits): rows of an FP8 cache read back out."""
    cache = _c(cache, np.uint8)
    assert cache.size == num_blocks * block_size * FP8_SLOT_BYTES
    sl = _c(slots, np.int64)
    out = np.empty((sl.size, 512), dtype=np.uint16)
    err = _load().oracle_dequant_gather(cache.ctypes.data, num_blocks, block_size, sl.ctypes.data,
                                        sl.size, out.ctypes.data)
    return out, int(err)


def indexer_k_quant_insert(k: np.ndarray, slots: np.ndarray, cache: np.ndarray, num_blocks: int,
                           block_size: int) -> int:
    """Quantise indexer K rows (bf16 bits [T, 128]) into the indexer cache
    (uint8, num_blocks * block_size * 132 bytes) in place; returns the error bits."""
    k = _c(k, np.uint16)
    sl = _c(slots, np.int64)
    assert k.size == sl.size * INDEXER_DIM
    assert cache.dtype == np.uint8 and cache.flags.c_contiguous
    assert cache.size == num_blocks * block_size * INDEXER_SLOT_BYTES
    return int(_load().oracle_indexer_k_quant_insert(k.ctypes.data, sl.ctypes.data, cache.ctypes.data,
                                                     num_blocks, block_size, sl.size))


def indexer_k_gather(cache: np.ndarray, num_blocks: int, block_size: int, slots: np.ndarray):
    """(codes uint8 [n, 128], scales float32 [n], error bits) read from the indexer cache."""
    cache = _c(cache, np.uint8)
    assert cache.size == num_blocks * block_size * INDEXER_SLOT_BYTES
    sl = _c(slots, np.int64)
    k_out = np.empty((sl.size, INDEXER_DIM), dtype=np.uint8)
    scale = np.empty(sl.size, dtype=np.float32)
    err = _load().oracle_indexer_k_gather(cache.ctypes.data, num_blocks, block_size, sl.ctypes.data,
                                          sl.size, k_out.ctypes.data, scale.ctypes.data)
    return k_out, scale, int(err)


def mxfp8_scale_bytes(m: int, n: int) -> int:
    return int(_load().oracle_mxfp8_scale_bytes(m, n))


def swizzled_scale_offset(row: int, col: int, padded_cols: int) -> int:
    return int(_load().oracle_swizzled_scale_offset(row, col, padded_cols))


def ue8m0_of_f32(x: float) -> int:
    return int(_load().oracle_ue8m0_of_f32(x))


def ue8m0_inverse(e: int) -> float:
    return float(_load().oracle_ue8m0_inverse(e))


def gemma_rmsnorm_mxfp8(x: np.ndarray, residual: np.ndarray, gamma: np.ndarray, eps: float):
    """(residual_out bf16 bits [m, n], E4M3 codes [m, n], swizzled UE8M0 scales)."""
    x = _c(x, np.uint16)
    residual = _c(residual, np.uint16)
    gamma = _c(gamma, np.uint16)
    m, n = x.shape
    assert n % 128 == 0 and residual.shape == (m, n) and gamma.shape == (n,)
    res_out = np.empty((m, n), np.uint16)
    codes = np.empty((m, n), np.uint8)
    scales = np.empty(mxfp8_scale_bytes(m, n), np.uint8)
    _load().oracle_gemma_rmsnorm_mxfp8(x.ctypes.data, residual.ctypes.data, gamma.ctypes.data, m, n,
                                        eps, res_out.ctypes.data, codes.ctypes.data,
                                        scales.ctypes.data)
    return res_out, codes, scales
