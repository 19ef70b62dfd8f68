"""kv_norm_rope_gb300: Python binding of libdsv4kv, the GB300 (sm_103a) library for the
fused DeepSeek-V4 attention-input step (q RMSNorm + RoPE in place; KV RMSNorm with a
weight + RoPE + UE8M0/E4M3 quantisation + paged-cache insert).

Argument marshalling only: every step runs in the CUDA kernels of ``csrc/``, reached
through the C ABI declared in ``include/dsv4kv.h``.  There is no CPU fallback: if the
shared library is missing and cannot be built, importing the entry points raises.
PyTorch supplies device memory and the current stream.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import tempfile
from concurrent.futures import ThreadPoolExecutor

_HERE = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_HERE)
_CSRC = os.path.join(_HERE, "csrc")
_INCLUDE = os.path.join(_ROOT, "include")
LIB_PATH = os.path.join(_HERE, "libdsv4kv.so")
# the same sources with every global access tested against its buffer (DSV4_CHECK_BOUNDS)
CHECKED_LIB_PATH = os.path.join(_HERE, "libdsv4kv_checked.so")
_SOURCES = ["qnorm_rope_kv_insert.cu", "dequant_gather.cu",
            "gemma_rmsnorm_mxfp8.cu", "indexer_k.cu", "kv_rows.cu", "qnorm_rope_kv_insert_half.cu",
            "wait_check.cu",
            "api.cpp"]
_HEADERS = [os.path.join(_INCLUDE, "dsv4kv.h")] + [
    os.path.join(_CSRC, h)
    for h in ("launch.h", "ops.h", "fastdiv.h", "convert.cuh", "launch_status.h", "rowmath.cuh",
              "halfrow.cuh", "bulkcopy.cuh", "bounds.cuh", "bounds_range.h")]
NVCC_ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]

# status codes and constants (mirrors include/dsv4kv.h)
OK, ERR_NULL, ERR_SHAPE, ERR_ALIGN, ERR_VALUE, ERR_CUDA = range(6)
DEVERR_SLOT_RANGE, DEVERR_POS_RANGE, DEVERR_TIMEOUT, DEVERR_BOUNDS = 1, 2, 4, 8
STORE_FP8, STORE_BF16 = 0, 1
VARIANT_AUTO, VARIANT_SMALL, VARIANT_STREAM, VARIANT_HALF = 0, 1, 2, 4
FP8_SLOT_BYTES, BF16_SLOT_BYTES = 584, 1024

EXPORTS = ("dsv4_qnorm_rope_kv_quant_insert", "dsv4_qnorm_rope_kv_bf16_insert",
           "dsv4_qnorm_rope_kv_insert_variant", "dsv4_qnorm_rope_kv_rope_quant_insert",
           "dsv4_kv_norm_rope_insert", "dsv4_insert_ex", "dsv4_dequant_gather",
           "dsv4_add_gemma_rmsnorm_mxfp8", "dsv4_mxfp8_scale_bytes", "dsv4_launch_plan",
           "dsv4_fp8_cache_bytes", "dsv4_bf16_cache_bytes", "dsv4_indexer_k_quant_insert",
           "dsv4_indexer_k_gather", "dsv4_indexer_cache_bytes", "dsv4_check_bounded_wait",
           "dsv4_debug_bounds_flags", "dsv4_status_string")


class Dsv4Error(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {status_string(status)} (status {status})")
        self.status = status


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale(path: str) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    deps = [os.path.join(_CSRC, s) for s in _SOURCES] + _HEADERS
    return any(os.path.getmtime(d) > t for d in deps)


def _build_one(path: str, extra: list, verbose: bool) -> str:
    bdir = tempfile.mkdtemp(prefix="dsv4kv_build_", dir=_HERE)
    flags = NVCC_ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                         "-I", _INCLUDE, "-I", _CSRC] + extra
    if verbose:
        flags += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src) + ".o")
        subprocess.run([_nvcc()] + flags + ["-c", os.path.join(_CSRC, src), "-o", obj], check=True)
        return obj

    with ThreadPoolExecutor(len(_SOURCES)) as ex:
        objs = list(ex.map(compile_one, _SOURCES))
    tmp = os.path.join(bdir, os.path.basename(path))
    subprocess.run([_nvcc()] + NVCC_ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs,
                   check=True)
    os.replace(tmp, path)
    for f in objs:
        os.remove(f)
    os.rmdir(bdir)
    return path


def build(force: bool = False, verbose: bool = False, checked: bool | None = None) -> str:
    """Compile csrc/ for sm_103a with nvcc into libdsv4kv.so and its checked twin
    libdsv4kv_checked.so (DSV4_CHECK_BOUNDS: every global access tested against its
    buffer), both in-tree.  checked=False builds the release library only, True the
    checked one only.  Translation units compile in parallel and link the static CUDA
    runtime, so the libraries need only the driver at run time.  Returns the path of
    the release library (of the checked one for checked=True)."""
    jobs = []
    if checked is not True and (force or _stale(LIB_PATH)):
        jobs.append((LIB_PATH, []))
    if checked is not False and (force or _stale(CHECKED_LIB_PATH)):
        jobs.append((CHECKED_LIB_PATH, ["-DDSV4_CHECK_BOUNDS"]))
    with ThreadPoolExecutor(max(1, len(jobs))) as ex:
        list(ex.map(lambda j: _build_one(j[0], j[1], verbose), jobs))
    return CHECKED_LIB_PATH if checked else LIB_PATH


_lib = None


def lib():
    """The loaded libdsv4kv (built first if missing or older than its sources).  With
    DSV4KV_CHECKED=1 in the environment this is the checked build instead."""
    global _lib
    if _lib is None:
        checked = os.environ.get("DSV4KV_CHECKED", "") == "1"
        _lib = _load(build(checked=checked))
    return _lib


@contextlib.contextmanager
def checked_build():
    """Route every call made in the block through libdsv4kv_checked.so, whose kernels
    test each global access against its buffer (see dsv4_debug_bounds_flags)."""
    global _lib
    saved = lib()
    _lib = _load(build(checked=True))
    try:
        yield _lib
    finally:
        _lib = saved


def debug_bounds_flags(reset: bool = True) -> int:
    """dsv4_debug_bounds_flags of the loaded library: 0 or DEVERR_BOUNDS (checked
    build), -1 (release build)."""
    return int(lib().dsv4_debug_bounds_flags(1 if reset else 0))


def _load(path: str):
    """Open a built library and declare its entry points' argument types."""
    L = ctypes.CDLL(path)
    vp, i64, i32, f32, c_int = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                ctypes.c_float, ctypes.c_int)
    common = [vp, vp, vp, vp, vp, i64, vp, vp, i64, i32, i64, i32, f32, vp, vp]
    L.dsv4_qnorm_rope_kv_quant_insert.argtypes = common
    L.dsv4_qnorm_rope_kv_quant_insert.restype = c_int
    L.dsv4_qnorm_rope_kv_bf16_insert.argtypes = common
    L.dsv4_qnorm_rope_kv_bf16_insert.restype = c_int
    L.dsv4_qnorm_rope_kv_insert_variant.argtypes = [c_int, c_int] + common
    L.dsv4_qnorm_rope_kv_insert_variant.restype = c_int
    L.dsv4_insert_ex.argtypes = [c_int, c_int, c_int] + common
    L.dsv4_insert_ex.restype = c_int
    L.dsv4_qnorm_rope_kv_rope_quant_insert.argtypes = [vp, vp, vp, vp, i64, vp, vp, i64, i32,
                                                       i64, i32, f32, vp, vp]
    L.dsv4_qnorm_rope_kv_rope_quant_insert.restype = c_int
    L.dsv4_kv_norm_rope_insert.argtypes = [c_int, vp, vp, vp, vp, i64, vp, vp, i64, i32, i64,
                                           f32, vp, vp]
    L.dsv4_kv_norm_rope_insert.restype = c_int
    L.dsv4_dequant_gather.argtypes = [vp, i64, i32, vp, i64, vp, vp, vp]
    L.dsv4_dequant_gather.restype = c_int
    L.dsv4_add_gemma_rmsnorm_mxfp8.argtypes = [vp, vp, vp, i64, i32, f32, vp, vp, vp, vp]
    L.dsv4_add_gemma_rmsnorm_mxfp8.restype = c_int
    L.dsv4_mxfp8_scale_bytes.argtypes = [i64, i32]
    L.dsv4_mxfp8_scale_bytes.restype = ctypes.c_size_t
    L.dsv4_launch_plan.argtypes = [i64, i32, i32, i32, i32, ctypes.POINTER(Plan)]
    L.dsv4_launch_plan.restype = c_int
    L.dsv4_fp8_cache_bytes.argtypes = [i64, i32]
    L.dsv4_fp8_cache_bytes.restype = ctypes.c_size_t
    L.dsv4_bf16_cache_bytes.argtypes = [i64, i32]
    L.dsv4_bf16_cache_bytes.restype = ctypes.c_size_t
    L.dsv4_indexer_k_quant_insert.argtypes = [vp, vp, vp, i64, i32, i64, vp, vp]
    L.dsv4_indexer_k_quant_insert.restype = c_int
    L.dsv4_indexer_k_gather.argtypes = [vp, i64, i32, vp, i64, vp, vp, vp, vp]
    L.dsv4_indexer_k_gather.restype = c_int
    L.dsv4_indexer_cache_bytes.argtypes = [i64, i32]
    L.dsv4_indexer_cache_bytes.restype = ctypes.c_size_t
    L.dsv4_check_bounded_wait.argtypes = [i64, vp, vp]
    L.dsv4_check_bounded_wait.restype = c_int
    L.dsv4_debug_bounds_flags.argtypes = [c_int]
    L.dsv4_debug_bounds_flags.restype = c_int
    L.dsv4_status_string.argtypes = [c_int]
    L.dsv4_status_string.restype = ctypes.c_char_p
    return L


class Plan(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int32), ("threads", ctypes.c_int32), ("ctas", ctypes.c_int64),
                ("rows_per_warp", ctypes.c_int32), ("rows", ctypes.c_int64)]


def status_string(status: int) -> str:
    return lib().dsv4_status_string(status).decode()


def launch_plan(num_tokens: int, num_heads: int, sm_count: int, ctas_per_sm: int,
                variant: int = VARIANT_AUTO) -> Plan:
    plan = Plan()
    st = lib().dsv4_launch_plan(num_tokens, num_heads, sm_count, ctas_per_sm, variant,
                                ctypes.byref(plan))
    if st != OK:
        raise Dsv4Error(st, "dsv4_launch_plan")
    return plan


def fp8_cache_bytes(num_blocks: int, block_size: int) -> int:
    return int(lib().dsv4_fp8_cache_bytes(num_blocks, block_size))


def bf16_cache_bytes(num_blocks: int, block_size: int) -> int:
    return int(lib().dsv4_bf16_cache_bytes(num_blocks, block_size))


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream_handle(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _kinds():
    import torch
    two_byte = (torch.bfloat16, torch.int16) + ((torch.uint16,) if hasattr(torch, "uint16") else ())
    return {"bf16": two_byte, "i64": (torch.int64,), "f32": (torch.float32,),
            "u8": (torch.uint8, torch.int8), "i32": (torch.int32,), "bytes": None}


def _check(name: str, t, kind: str, numel: int | None = None, min_bytes: int | None = None):
    """Reject a tensor argument the C ABI cannot check: wrong element type (bf16 data
    may come as any 2-byte dtype), not contiguous, or the wrong number of elements /
    too few bytes.  Raw integer pointers pass unchecked; _on_cuda checks devices."""
    if t is None or isinstance(t, int):
        return
    allowed = _kinds()[kind]
    if allowed is not None and t.dtype not in allowed:
        raise TypeError(f"{name}: expected {kind} data, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name}: expected {numel} elements, got {t.numel()}")
    if min_bytes is not None and t.numel() * t.element_size() < min_bytes:
        raise ValueError(f"{name}: needs at least {min_bytes} bytes, has "
                         f"{t.numel() * t.element_size()}")


def _on_cuda(**tensors):
    """Every tensor argument lives on one CUDA device: there is no CPU path."""
    devices = set()
    for name, t in tensors.items():
        if t is None or isinstance(t, int):
            continue
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
        devices.add(t.device)
    if len(devices) > 1:
        raise ValueError(f"tensor arguments on several devices: {sorted(map(str, devices))}")


def _check_step(store_mode, q, kv, w, positions, cos_sin_cache, slot_mapping, kv_cache,
                num_blocks, block_size, device_error, T, H):
    _check("positions", positions, "i64", T)
    _check("slot_mapping", slot_mapping, "i64", T)
    _check("q", q, "bf16", T * H * 512)
    _check("kv", kv, "bf16", T * 512)
    _check("kv_norm_weight", w, "bf16", 512)
    _check("cos_sin_cache", cos_sin_cache, "f32")
    if not isinstance(cos_sin_cache, int) and cos_sin_cache.numel() % 64:
        raise ValueError("cos_sin_cache must hold rows of 64 fp32 (32 cos, 32 sin)")
    need = (fp8_cache_bytes if store_mode == STORE_FP8 else bf16_cache_bytes)(num_blocks, block_size)
    _check("kv_cache", kv_cache, "bytes", min_bytes=need)
    _check("device_error", device_error, "i32")
    _on_cuda(q=q, kv=kv, kv_norm_weight=w, positions=positions, cos_sin_cache=cos_sin_cache,
             slot_mapping=slot_mapping, kv_cache=kv_cache, device_error=device_error)


def _shape_args(q, kv, positions, cos_sin_cache):
    T = int(positions.shape[0])
    if q is None:
        H = 0
    else:
        H = int(q.shape[-2]) if q.dim() == 3 else int(q.numel() // max(T, 1) // 512)
    return T, H, int(cos_sin_cache.shape[0])


def insert(store_mode: int, q, kv, kv_norm_weight, positions, cos_sin_cache, slot_mapping,
           kv_cache, num_blocks: int, block_size: int, eps: float, device_error=None,
           stream=None, variant: int = VARIANT_AUTO, num_heads: int | None = None,
           kv_norm: bool = True) -> None:
    """Enqueue the fused step on ``stream`` (default: torch's current stream).

    q: bf16 [T, H, 512] (rewritten in place; None for KV rows only); kv: bf16 [T, 512];
    kv_norm_weight: bf16 [512] (unused, may be None, when ``kv_norm`` is False: the KV
    rows then arrive normalised); positions, slot_mapping: int64 [T]; cos_sin_cache:
    fp32 [max_position, 64]; kv_cache: uint8 (FP8, num_blocks*block_size*584 bytes) or
    bf16 [num_blocks, block_size, 512]; device_error: optional int32 [1].  Raises
    Dsv4Error on a rejected call.  Goes through dsv4_insert_ex.
    """
    T, H, max_pos = _shape_args(q, kv, positions, cos_sin_cache)
    if num_heads is not None:
        H = num_heads
    _check_step(store_mode, q, kv, kv_norm_weight if kv_norm else None, positions, cos_sin_cache,
                slot_mapping, kv_cache, num_blocks, block_size, device_error, T, H)
    st = lib().dsv4_insert_ex(
        store_mode, variant, 1 if kv_norm else 0, _ptr(q), _ptr(kv), _ptr(kv_norm_weight),
        _ptr(positions), _ptr(cos_sin_cache), max_pos, _ptr(slot_mapping), _ptr(kv_cache),
        num_blocks, block_size, T, H, eps, _ptr(device_error), _stream_handle(stream))
    if st != OK:
        raise Dsv4Error(st, "dsv4_insert_ex")


def qnorm_rope_kv_rope_quant_insert(q, kv, positions, cos_sin_cache, slot_mapping, kv_cache,
                                    num_blocks, block_size, eps, device_error=None,
                                    stream=None) -> None:
    """dsv4_qnorm_rope_kv_rope_quant_insert: KV rows arrive normalised (rope + FP8 only)."""
    T, H, max_pos = _shape_args(q, kv, positions, cos_sin_cache)
    _check_step(STORE_FP8, q, kv, None, positions, cos_sin_cache, slot_mapping, kv_cache,
                num_blocks, block_size, device_error, T, H)
    st = lib().dsv4_qnorm_rope_kv_rope_quant_insert(
        _ptr(q), _ptr(kv), _ptr(positions), _ptr(cos_sin_cache), max_pos, _ptr(slot_mapping),
        _ptr(kv_cache), num_blocks, block_size, T, H, eps, _ptr(device_error),
        _stream_handle(stream))
    if st != OK:
        raise Dsv4Error(st, "dsv4_qnorm_rope_kv_rope_quant_insert")


def kv_norm_rope_insert(store_mode: int, kv, kv_norm_weight, positions, cos_sin_cache,
                        slot_mapping, kv_cache, num_blocks, block_size, eps, device_error=None,
                        stream=None) -> None:
    """dsv4_kv_norm_rope_insert: KV rows only (norm with weight, rope, FP8 or bf16 store)."""
    T, _, max_pos = _shape_args(None, kv, positions, cos_sin_cache)
    _check_step(store_mode, None, kv, kv_norm_weight, positions, cos_sin_cache, slot_mapping,
                kv_cache, num_blocks, block_size, device_error, T, 0)
    st = lib().dsv4_kv_norm_rope_insert(
        store_mode, _ptr(kv), _ptr(kv_norm_weight), _ptr(positions), _ptr(cos_sin_cache),
        max_pos, _ptr(slot_mapping), _ptr(kv_cache), num_blocks, block_size, T, eps,
        _ptr(device_error), _stream_handle(stream))
    if st != OK:
        raise Dsv4Error(st, "dsv4_kv_norm_rope_insert")


def qnorm_rope_kv_quant_insert(q, kv, kv_norm_weight, positions, cos_sin_cache, slot_mapping,
                               kv_cache, num_blocks, block_size, eps, device_error=None,
                               stream=None) -> None:
    """dsv4_qnorm_rope_kv_quant_insert: FP8 (448 E4M3 + 7 UE8M0 + 64 bf16) cache rows."""
    T, H, max_pos = _shape_args(q, kv, positions, cos_sin_cache)
    _check_step(STORE_FP8, q, kv, kv_norm_weight, positions, cos_sin_cache, slot_mapping, kv_cache,
                num_blocks, block_size, device_error, T, H)
    st = lib().dsv4_qnorm_rope_kv_quant_insert(
        _ptr(q), _ptr(kv), _ptr(kv_norm_weight), _ptr(positions), _ptr(cos_sin_cache), max_pos,
        _ptr(slot_mapping), _ptr(kv_cache), num_blocks, block_size, T, H, eps,
        _ptr(device_error), _stream_handle(stream))
    if st != OK:
        raise Dsv4Error(st, "dsv4_qnorm_rope_kv_quant_insert")


def qnorm_rope_kv_bf16_insert(q, kv, kv_norm_weight, positions, cos_sin_cache, slot_mapping,
                              kv_cache, num_blocks, block_size, eps, device_error=None,
                              stream=None) -> None:
    """dsv4_qnorm_rope_kv_bf16_insert: 512 bf16 cache rows."""
    T, H, max_pos = _shape_args(q, kv, positions, cos_sin_cache)
    _check_step(STORE_BF16, q, kv, kv_norm_weight, positions, cos_sin_cache, slot_mapping,
                kv_cache, num_blocks, block_size, device_error, T, H)
    st = lib().dsv4_qnorm_rope_kv_bf16_insert(
        _ptr(q), _ptr(kv), _ptr(kv_norm_weight), _ptr(positions), _ptr(cos_sin_cache), max_pos,
        _ptr(slot_mapping), _ptr(kv_cache), num_blocks, block_size, T, H, eps,
        _ptr(device_error), _stream_handle(stream))
    if st != OK:
        raise Dsv4Error(st, "dsv4_qnorm_rope_kv_bf16_insert")


def dequant_gather(kv_cache, num_blocks: int, block_size: int, slots, out, device_error=None,
                   stream=None) -> None:
    """dsv4_dequant_gather: out (bf16 [n, 512]) = FP8 cache rows at ``slots`` read back."""
    n = int(slots.shape[0])
    _check("slots", slots, "i64", n)
    _check("kv_cache", kv_cache, "bytes", min_bytes=fp8_cache_bytes(num_blocks, block_size))
    _check("out", out, "bf16", n * 512)
    _check("device_error", device_error, "i32")
    _on_cuda(kv_cache=kv_cache, slots=slots, out=out, device_error=device_error)
    st = lib().dsv4_dequant_gather(_ptr(kv_cache), num_blocks, block_size, _ptr(slots),
                                   int(slots.shape[0]), _ptr(out), _ptr(device_error),
                                   _stream_handle(stream))
    if st != OK:
        raise Dsv4Error(st, "dsv4_dequant_gather")


def check_bounded_wait(max_cycles: int = 0, device_error=None, stream=None) -> None:
    """dsv4_check_bounded_wait: one warp waits, through the bulk-copy kernels' bounded
    wait, on an mbarrier nothing completes; after max_cycles SM cycles (0: the kernels'
    own limit, about a second) it ORs DEVERR_TIMEOUT into device_error (int32 [1])."""
    if max_cycles < 0:
        raise ValueError("max_cycles must be >= 0")
    _check("device_error", device_error, "i32")
    _on_cuda(device_error=device_error)
    st = lib().dsv4_check_bounded_wait(int(max_cycles), _ptr(device_error), _stream_handle(stream))
    if st != OK:
        raise Dsv4Error(st, "dsv4_check_bounded_wait")


def indexer_cache_bytes(num_blocks: int, block_size: int) -> int:
    return int(lib().dsv4_indexer_cache_bytes(num_blocks, block_size))


def indexer_k_quant_insert(k, slot_mapping, indexer_cache, num_blocks: int, block_size: int,
                           device_error=None, stream=None) -> None:
    """dsv4_indexer_k_quant_insert: k (bf16 [T, 128]) quantised into the indexer cache
    (uint8, indexer_cache_bytes(num_blocks, block_size)) at slot_mapping (int64 [T])."""
    T = int(slot_mapping.shape[0])
    _check("slot_mapping", slot_mapping, "i64", T)
    _check("k", k, "bf16", T * 128)
    _check("indexer_cache", indexer_cache, "bytes",
           min_bytes=indexer_cache_bytes(num_blocks, block_size))
    _check("device_error", device_error, "i32")
    _on_cuda(k=k, slot_mapping=slot_mapping, indexer_cache=indexer_cache, device_error=device_error)
    st = lib().dsv4_indexer_k_quant_insert(_ptr(k), _ptr(slot_mapping), _ptr(indexer_cache),
                                           num_blocks, block_size, int(slot_mapping.shape[0]),
                                           _ptr(device_error), _stream_handle(stream))
    if st != OK:
        raise Dsv4Error(st, "dsv4_indexer_k_quant_insert")


def indexer_k_gather(indexer_cache, num_blocks: int, block_size: int, slots, k_out, scale_out,
                     device_error=None, stream=None) -> None:
    """dsv4_indexer_k_gather: k_out (uint8 [n, 128]) and scale_out (fp32 [n]) read from
    the indexer cache at ``slots`` (int64 [n])."""
    n = int(slots.shape[0])
    _check("slots", slots, "i64", n)
    _check("indexer_cache", indexer_cache, "bytes",
           min_bytes=indexer_cache_bytes(num_blocks, block_size))
    _check("k_out", k_out, "u8", n * 128)
    _check("scale_out", scale_out, "f32", n)
    _check("device_error", device_error, "i32")
    _on_cuda(indexer_cache=indexer_cache, slots=slots, k_out=k_out, scale_out=scale_out,
             device_error=device_error)
    st = lib().dsv4_indexer_k_gather(_ptr(indexer_cache), num_blocks, block_size, _ptr(slots),
                                     int(slots.shape[0]), _ptr(k_out), _ptr(scale_out),
                                     _ptr(device_error), _stream_handle(stream))
    if st != OK:
        raise Dsv4Error(st, "dsv4_indexer_k_gather")


def mxfp8_scale_bytes(num_rows: int, hidden: int) -> int:
    return int(lib().dsv4_mxfp8_scale_bytes(num_rows, hidden))


def add_gemma_rmsnorm_mxfp8(x, residual, gamma, eps: float, residual_out, codes, scales,
                            stream=None) -> None:
    """dsv4_add_gemma_rmsnorm_mxfp8: residual add + Gemma RMSNorm + MXFP8 rows.

    x, residual, residual_out: bf16 [m, n]; gamma: bf16 [n]; codes: uint8 [m, n];
    scales: uint8, mxfp8_scale_bytes(m, n) bytes."""
    m, n = int(x.shape[0]), int(x.shape[1])
    for name, t in (("x", x), ("residual", residual), ("residual_out", residual_out)):
        _check(name, t, "bf16", m * n)
    _check("gamma", gamma, "bf16", n)
    _check("codes", codes, "u8", m * n)
    _check("scales", scales, "u8", min_bytes=mxfp8_scale_bytes(m, n))
    _on_cuda(x=x, residual=residual, gamma=gamma, residual_out=residual_out, codes=codes,
             scales=scales)
    st = lib().dsv4_add_gemma_rmsnorm_mxfp8(_ptr(x), _ptr(residual), _ptr(gamma), m, n, eps,
                                            _ptr(residual_out), _ptr(codes), _ptr(scales),
                                            _stream_handle(stream))
    if st != OK:
        raise Dsv4Error(st, "dsv4_add_gemma_rmsnorm_mxfp8")
