"""The library from a plain C program: no Python, no torch on the calling side.

tests/c/abi_demo.c is compiled with gcc against include/dsv4kv.h and linked with
libdsv4kv.so and the CUDA runtime; it reads the inputs of one fused step from
files, calls dsv4_qnorm_rope_kv_quant_insert and writes q and the cache back.
Its outputs must meet the oracle's parity bar like the Python path's.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

from synth import configs
from tests import harness

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import kv_norm_rope_gb300 as k  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_home():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def test_plain_c_caller(tmp_path):
    lib = k.build()
    cuda = _cuda_home()
    exe = tmp_path / "abi_demo"
    subprocess.run(["gcc", "-O2", "-std=c11", os.path.join(ROOT, "tests", "c", "abi_demo.c"),
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
                    "-o", str(exe), lib, "-L", os.path.join(cuda, "lib64"), "-lcudart",
                    f"-Wl,-rpath,{os.path.dirname(lib)}", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}"],
                   check=True)
    wl = configs.generic(300, 16, seed=61)
    inp = harness.make_inputs(wl)
    for name, arr in (("q", inp.q), ("kv", inp.kv), ("w", inp.w), ("pos", inp.positions),
                      ("slot", inp.slots), ("cs", inp.cos_sin), ("cache", inp.poison)):
        np.ascontiguousarray(arr).tofile(tmp_path / f"{name}.bin")
    out = subprocess.run([str(exe), str(tmp_path), str(wl.T), str(wl.H), str(wl.num_blocks),
                          str(wl.block_size), str(wl.max_position)], capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    q = np.fromfile(tmp_path / "q_out.bin", dtype=np.uint16).reshape(wl.T, wl.H, 512)
    cache = np.fromfile(tmp_path / "cache_out.bin", dtype=np.uint8)
    err = int((tmp_path / "err.txt").read_text())
    ref_q, ref_cache, ref_err = harness.run_oracle(inp)
    assert err == ref_err
    gpu = harness.GpuResult(np.arange(wl.T, dtype=np.int64), q, cache, err)
    rep = harness.compare_results(inp, gpu, ref_q, ref_cache)
    assert rep.ok, str(rep)
