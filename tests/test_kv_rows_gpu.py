"""The KV-row kernel (calls with no q heads, one row per quarter-warp) on the GPU.

Its cache rows must be bit-identical to those the fused kernel writes for the
same KV inputs (same sums, same butterfly, same elementwise operations, same
exact decision near a scale boundary), and must meet the oracle's parity bar
on their own, including warps in which some quarter-warps' rows are skipped.
"""
import dataclasses

import numpy as np
import pytest

import synth
from synth import configs
from tests import harness
from tests.test_parity_gpu import _near_boundary_rows

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import kv_norm_rope_gb300 as k  # noqa: E402


def _kv_only(inp: harness.Inputs) -> harness.Inputs:
    """The same KV rows, positions and slots with no q heads."""
    wl = dataclasses.replace(inp.wl, H=0, name=inp.wl.name + "_h0")
    return dataclasses.replace(inp, wl=wl, q=np.empty((wl.T, 0, 512), np.uint16))


@pytest.mark.parametrize("kv_norm", [True, False])
@pytest.mark.parametrize("wl", [configs.generic(4099, 4, seed=70),
                                configs.generic(3001, 4, store="bf16", seed=71),
                                configs.generic(2222, 4, seed=72, tail_frac=0.02, tail_mult=100.0)],
                         ids=lambda w: w.name)
def test_cache_rows_bit_identical_to_fused_kernel(wl, kv_norm):
    inp = harness.make_inputs(wl)
    fused = harness.run_gpu(inp, k.VARIANT_STREAM, q_tokens=np.arange(2), kv_norm=kv_norm)
    alone = harness.run_gpu(_kv_only(inp), k.VARIANT_STREAM, kv_norm=kv_norm)
    assert alone.err == fused.err
    assert np.array_equal(alone.cache, fused.cache)
    # and the other KV-only variants agree with it
    for v in (k.VARIANT_SMALL,):
        other = harness.run_gpu(_kv_only(inp), v, kv_norm=kv_norm)
        assert np.array_equal(other.cache, alone.cache)


def test_scale_decisions_near_boundaries_kv_only():
    """Rows whose block amax sits within 2^-13 of a UE8M0 boundary go through the
    kernel's fp64 decision; against the oracle and against the fused kernel."""
    rows, kv_all, w = _near_boundary_rows()
    T = int(rows.size)
    assert T >= 100
    wl = configs.Workload("near_boundary_kv", T, 0, "fp8", 1, -(-T // 64), 64, 31)
    ident = np.array([[1.0] * 32 + [0.0] * 32], np.float32)
    inp = harness.Inputs(wl, np.empty((T, 0, 512), np.uint16), np.ascontiguousarray(kv_all[rows]),
                         w, np.zeros(T, np.int64), np.arange(T, dtype=np.int64)[::-1].copy(), ident,
                         synth.poison_bytes(wl.num_slots * 584, seed=3))
    gpu = harness.run_gpu(inp, k.VARIANT_STREAM)
    ref_q, ref_cache, ref_err = harness.run_oracle(inp)
    rep = harness.compare_results(inp, gpu, ref_q, ref_cache)
    assert rep.ok, str(rep)
    fused_inp = dataclasses.replace(inp, wl=dataclasses.replace(wl, H=1, name="near_boundary_kv1"),
                                    q=np.ascontiguousarray(kv_all[rows][:, None, :]))
    fused = harness.run_gpu(fused_inp, k.VARIANT_STREAM)
    assert np.array_equal(fused.cache, gpu.cache)


@pytest.mark.parametrize("store", ["fp8", "bf16"])
def test_quads_with_rows_skipped(store):
    """Tokens alternate between written and skipped rows (negative slot, slot past the
    cache, position outside the table), so many warps' groups of four rows have one to
    three idle quarters, and a few groups are skipped whole."""
    T = 3003
    wl = configs.generic(T, 0, store=store, seed=80, skip_frac=0.0)
    base = harness.make_inputs(wl)
    slots = base.slots.copy()
    pos = base.positions.copy()
    slots[1::4] = -1
    slots[2::8] = wl.num_slots + 7
    pos[3::8] = wl.max_position + 1
    pos[7::16] = -5
    slots[20:24] = -1
    slots[1000:1004] = -1
    inp = dataclasses.replace(base, slots=slots, positions=pos)
    gpu = harness.run_gpu(inp, k.VARIANT_STREAM)
    ref_q, ref_cache, ref_err = harness.run_oracle(inp)
    assert gpu.err == ref_err == (k.DEVERR_SLOT_RANGE | k.DEVERR_POS_RANGE)
    rep = harness.compare_results(inp, gpu, ref_q, ref_cache)
    assert rep.ok, str(rep)


@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 7, 8, 9, 63, 65, 4095, 12345])
def test_ragged_token_counts(T):
    rep = harness.check(configs.generic(T, 0, seed=90 + T), k.VARIANT_STREAM)
    assert rep.ok, str(rep)



def test_offsets_past_2_gib():
    """2^21 + 5 KV rows through the bulk-copy kernel: kv offsets reach 2.15 GB and cache
    offsets 2.45 GB, past 2^31 bytes; every cache row against the oracle."""
    wl = configs.generic(2 ** 21 + 5, 0, seed=95, skip_frac=0.01)
    rep = harness.check(wl, k.VARIANT_STREAM)
    assert rep.ok, str(rep)
