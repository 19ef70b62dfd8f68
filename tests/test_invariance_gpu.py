"""Every launch variant gives bit-identical outputs: a token's rows depend only on that
token's inputs, not on which warp, CTA or variant processed them (the property the
SGLang K-tokens-per-block change relies on, section "Modifications")."""
import numpy as np
import pytest

from synth import configs
from tests import harness

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import kv_norm_rope_gb300 as k  # noqa: E402


@pytest.mark.parametrize("wl", [configs.DECODE, configs.generic(2049, 64, seed=12),
                                configs.generic(1500, 128, store="bf16", seed=13),
                                configs.generic(777, 3, seed=14, tail_frac=0.02, tail_mult=100.0)],
                         ids=lambda w: w.name)
def test_variants_bit_identical(wl):
    inp = harness.make_inputs(wl)
    outs = [harness.run_gpu(inp, v) for v in (k.VARIANT_SMALL, k.VARIANT_STREAM, k.VARIANT_HALF,
                                              k.VARIANT_AUTO)]
    for o in outs[1:]:
        assert np.array_equal(o.q, outs[0].q)
        assert np.array_equal(o.cache, outs[0].cache)
        assert o.err == outs[0].err


@pytest.mark.parametrize("T,H", [(405, 8), (406, 8), (3647, 0), (3649, 0)])
def test_auto_at_its_small_switch(T, H):
    """Rows just below and just above the warp slots of a 152-SM GB300 (3648), where AUTO
    switches from one row per warp to the half-warp or KV-row kernel: the same bytes as
    the streaming kernel on either side."""
    inp = harness.make_inputs(configs.generic(T, H, seed=16 + T))
    a = harness.run_gpu(inp, k.VARIANT_AUTO)
    b = harness.run_gpu(inp, k.VARIANT_STREAM)
    assert np.array_equal(a.q, b.q) and np.array_equal(a.cache, b.cache) and a.err == b.err


def test_repeat_is_deterministic():
    wl = configs.generic(3000, 32, seed=15)
    inp = harness.make_inputs(wl)
    a = harness.run_gpu(inp)
    b = harness.run_gpu(inp)
    assert np.array_equal(a.q, b.q) and np.array_equal(a.cache, b.cache)
