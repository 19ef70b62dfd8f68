"""The exact scale decision for blocks whose fp32 amax is too close to a UE8M0 boundary.

The kernels settle such blocks in fp32 float-float arithmetic and use fp64 only where
that cannot decide: a value within 2^-38 of the boundary, or an element whose square or
product leaves the range where the fp32 steps are exact.  These tests drive each path
(ties that only fp64 settles, near misses the fp32 path settles, out-of-range elements)
and check the cache rows against the oracle and across every kernel.
"""
import dataclasses

import numpy as np
import pytest

import synth
from synth import configs
from tests import harness
from tests.test_parity_gpu import VARIANTS, _near_boundary_rows

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import kv_norm_rope_gb300 as k  # noqa: E402

# one cos/sin row: cos 1, sin 0 (the rope leaves its dims unrotated)
IDENT = np.array([[1.0] * 32 + [0.0] * 32], np.float32)


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    """float64 values that are exact in bf16 -> their bf16 bit patterns."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    bits = f.view(np.uint32)
    assert not np.any(bits & 0xFFFF), "value not exact in bf16"
    return (bits >> 16).astype(np.uint16)


def _check_everywhere(inp: harness.Inputs):
    """Every fused variant and the KV-only kernel against the oracle; all caches equal."""
    ref_q, ref_cache, _ = harness.run_oracle(inp)
    caches = []
    for v in VARIANTS:
        gpu = harness.run_gpu(inp, v)
        rep = harness.compare_results(inp, gpu, ref_q, ref_cache)
        assert rep.ok, f"variant {v}: {rep}"
        caches.append(gpu.cache)
    wl0 = dataclasses.replace(inp.wl, H=0, name=inp.wl.name + "_h0")
    alone = harness.run_gpu(dataclasses.replace(inp, wl=wl0, q=np.empty((wl0.T, 0, 512), np.uint16)),
                            k.VARIANT_STREAM)
    caches.append(alone.cache)
    for c in caches[1:]:
        assert np.array_equal(c, caches[0])


def _tie_inputs(T: int, eps: float, seed: int) -> harness.Inputs:
    """Rows of +-2^k (random signs, k per row) and a weight whose 64-dim blocks are 2^j_b
    with one element 1.75 * 2^j_b: x * r is exactly +-1 when eps = 0, so every block's
    amax is exactly the boundary 1.75 * 2^j_b (not above it: scale exponent j_b - 8)."""
    rng = np.random.default_rng(seed)
    kexp = rng.integers(-4, 5, size=T)
    x = rng.choice([-1.0, 1.0], size=(T, 512)) * np.exp2(kexp)[:, None]
    jb = np.array([-2, 0, 3, 1, -1, 2, 0])
    w = np.ones(512)
    for b in range(7):
        w[64 * b:64 * b + 64] = 2.0 ** jb[b]
        w[64 * b + int(rng.integers(64))] = 1.75 * 2.0 ** jb[b]
    kv = _bf16_bits(x)
    wl = configs.Workload(f"ties_eps{eps:g}", T, 1, "fp8", 1, -(-T // 64), 64, seed, eps=eps)
    return harness.Inputs(wl, kv[:, None, :].copy(), kv, _bf16_bits(w), np.zeros(T, np.int64),
                          np.arange(T, dtype=np.int64), IDENT,
                          synth.poison_bytes(wl.num_slots * 584, seed=seed))


@pytest.mark.parametrize("eps", [0.0, 1e-6])
def test_block_amax_on_a_boundary(eps):
    """eps = 0: exact ties, left to the fp64 decision; eps = 1e-6: a hair below every
    boundary (within the fp32 band), settled by the fp32 float-float decision."""
    inp = _tie_inputs(300, eps, seed=41)
    _check_everywhere(inp)
    # the tie rows: every nope byte decodes to 256 or 448 at scale 2^(j_b - 8)
    if eps == 0.0:
        gpu = harness.run_gpu(inp, k.VARIANT_STREAM)
        T, bs = inp.wl.T, inp.wl.block_size
        for t in (0, 1, T - 1):
            blk, off = divmod(t, bs)
            base = blk * bs * 584
            scales = gpu.cache[base + bs * 576 + off * 8: base + bs * 576 + off * 8 + 7]
            assert scales.tolist() == [127 + j - 8 for j in (-2, 0, 3, 1, -1, 2, 0)]


def test_element_out_of_fp32_range_takes_the_fp64_path():
    """Near-boundary rows with one element of 2^-100 (its square underflows fp32): the
    fp32 decision declines and the fp64 one decides, in every kernel."""
    rows, kv_all, w = _near_boundary_rows(n_scan=60_000)
    rows = rows[:120]
    kv = np.ascontiguousarray(kv_all[rows])
    kv[:, 300] = 0x0D80  # bf16 2^-100
    T = int(rows.size)
    wl = configs.Workload("near_boundary_tiny", T, 1, "fp8", 1, -(-T // 64), 64, 43)
    inp = harness.Inputs(wl, kv[:, None, :].copy(), kv, w, np.zeros(T, np.int64),
                         np.arange(T, dtype=np.int64)[::-1].copy(), IDENT,
                         synth.poison_bytes(wl.num_slots * 584, seed=4))
    _check_everywhere(inp)


def test_near_boundary_rows_agree_across_kernels():
    """The near-boundary rows of the parity suite, settled by the fp32 decision: every
    kernel writes the same bytes as the oracle."""
    rows, kv_all, w = _near_boundary_rows(n_scan=100_000)
    kv = np.ascontiguousarray(kv_all[rows])
    T = int(rows.size)
    assert T >= 40
    wl = configs.Workload("near_boundary_all", T, 1, "fp8", 1, -(-T // 64), 64, 44)
    inp = harness.Inputs(wl, kv[:, None, :].copy(), kv, w, np.zeros(T, np.int64),
                         np.arange(T, dtype=np.int64), IDENT,
                         synth.poison_bytes(wl.num_slots * 584, seed=5))
    _check_everywhere(inp)


# row scales of the tiny-row test: normal rows, rows whose squares are still normal in
# fp32, rows whose squares are subnormal (below 2^-63) and rows of bf16 subnormals
TINY_SCALES = [1.0, 2.0**-50, 2.0**-64, 2.0**-70, 2.0**-100, 2.0**-115, 2.0**-124, 2.0**-128]


def _scaled_bits(bits: np.ndarray, scale: np.ndarray) -> np.ndarray:
    """bf16 bit patterns times a per-row power of two, rounded to bf16 (nearest even)."""
    f = synth.bf16_bits_to_f32(bits).reshape(scale.shape[0], -1) * scale[:, None].astype(np.float32)
    t = torch.from_numpy(np.ascontiguousarray(f, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).reshape(bits.shape)


@pytest.mark.parametrize("kv_norm", [True, False])
@pytest.mark.parametrize("store", ["fp8", "bf16"])
def test_tiny_rows_with_eps_zero(store, kv_norm):
    """With eps = 0, rows scaled down by 2^-50 .. 2^-128 normalise like their unscaled
    selves: squares below the fp32 normal range must not decide r.  Every variant and the
    KV-only kernel against the oracle, and all caches equal."""
    wl = dataclasses.replace(configs.generic(64, 3, store=store, seed=151), eps=0.0)
    base = harness.make_inputs(wl)
    tok_scale = np.array([TINY_SCALES[t % len(TINY_SCALES)] for t in range(wl.T)])
    q = _scaled_bits(base.q.reshape(wl.T, -1), tok_scale).reshape(base.q.shape)
    # the KV rows run through the scales in another order than the q rows of their token
    kv = _scaled_bits(base.kv, tok_scale[::-1].copy())
    inp = dataclasses.replace(base, q=q, kv=kv)
    assert np.all((kv & 0x7FFF).reshape(wl.T, -1).max(axis=1) > 0)  # no all-zero row
    ref_q, ref_cache, ref_err = harness.run_oracle(inp, kv_norm=kv_norm)
    caches = []
    for v in VARIANTS:
        gpu = harness.run_gpu(inp, v, kv_norm=kv_norm)
        rep = harness.compare_results(inp, gpu, ref_q, ref_cache)
        assert rep.ok, f"variant {v}: {rep}"
        assert gpu.err == ref_err == 0
        caches.append(gpu.cache)
    wl0 = dataclasses.replace(wl, H=0, name=wl.name + "_h0")
    alone = harness.run_gpu(dataclasses.replace(inp, wl=wl0, q=np.empty((wl0.T, 0, 512), np.uint16)),
                            k.VARIANT_STREAM, kv_norm=kv_norm)
    caches.append(alone.cache)
    for c in caches[1:]:
        assert np.array_equal(c, caches[0])
