"""Seeded random configurations of the fused step against the oracle.

Each case draws the token count, the head count (0 included: KV rows only), the
store mode, the block size, whether KV is normalised, the launch variant, a
heavy tail, skipped slots and a few out-of-range positions and slots, then
holds the GPU result to the parity bar (and the error word to the oracle's).
"""
import dataclasses

import numpy as np
import pytest

from synth import configs
from tests import harness

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import kv_norm_rope_gb300 as k  # noqa: E402

VARIANTS = [k.VARIANT_AUTO, k.VARIANT_SMALL, k.VARIANT_STREAM, k.VARIANT_HALF]


def _case(i):
    rng = np.random.default_rng(1000 + i)
    T = int(rng.choice([1, 2, 3, 5, 31, 64, 127, 500, 1023, 2500]))
    H = int(rng.choice([0, 1, 2, 3, 8, 17, 64, 128]))
    if T * H > 200_000:
        T = max(1, 200_000 // H)
    store = str(rng.choice(["fp8", "bf16"]))
    tail = float(rng.choice([0.0, 0.0, 0.01, 0.2]))
    base = configs.generic(T, H, store=store, seed=2000 + i, skip_frac=float(rng.choice([0.0, 0.1, 0.5])),
                           tail_frac=tail, tail_mult=float(rng.choice([10.0, 100.0, 1e4])))
    bs = int(rng.choice([1, 2, 3, 5, 16, 64, 100, 1024]))
    wl = dataclasses.replace(base, num_blocks=max(1, -(-2 * T // bs)), block_size=bs)
    nslots = wl.num_slots
    slots = np.full(T, -1, np.int64)
    perm = rng.permutation(nslots)[:T]
    keep = rng.random(T) >= float(rng.choice([0.0, 0.1, 0.5]))
    slots[keep] = perm[keep]
    positions = rng.integers(0, wl.max_position, T).astype(np.int64)
    if T > 4 and rng.random() < 0.5:
        positions[rng.integers(0, T)] = wl.max_position + int(rng.integers(0, 5))
        slots[rng.integers(0, T)] = nslots + int(rng.integers(0, 5))
    variant = int(rng.choice(VARIANTS))
    kv_norm = bool(rng.random() < 0.75)
    return wl, positions, slots, variant, kv_norm


@pytest.mark.parametrize("i", range(40))
def test_random_configuration(i):
    wl, positions, slots, variant, kv_norm = _case(i)
    inp = harness.make_inputs(wl, positions=positions, slots=slots)
    gpu = harness.run_gpu(inp, variant, kv_norm=kv_norm)
    ref_q, ref_cache, ref_err = harness.run_oracle(inp, kv_norm=kv_norm)
    assert gpu.err == ref_err, (wl, variant, kv_norm)
    rep = harness.compare_results(inp, gpu, ref_q, ref_cache)
    assert rep.ok, f"{wl} variant {variant} kv_norm {kv_norm}: {rep}"
