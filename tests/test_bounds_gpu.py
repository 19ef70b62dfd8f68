"""The bounds-checked build (libdsv4kv_checked.so) on the GPU.

Every kernel of that build tests each global load and store against the buffer it
belongs to before making it, skips an access that would leave the buffer and
records DSV4_DEVERR_BOUNDS.  Here each operation runs once on the release library
and once on the checked one, over the edges of its indexing (ragged tails, odd block
sizes, skipped, out-of-range and past-the-cache slots, offsets past 2^31 bytes): the
checked run must record no skipped access and give the same bytes as the release
run.  (The whole GPU suite can also run on the checked build: DSV4KV_CHECKED=1.)
"""
import numpy as np
import pytest

import synth
from synth import configs
from tests import harness

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import kv_norm_rope_gb300 as k  # noqa: E402

DEV = torch.device("cuda:0")
VARIANTS = [k.VARIANT_AUTO, k.VARIANT_SMALL, k.VARIANT_STREAM, k.VARIANT_HALF]


def _release_and_checked(fn):
    """fn() on the release library, then on the checked one; (release, checked)
    results, asserting that the checked run skipped nothing."""
    released = fn()
    with k.checked_build():
        assert k.debug_bounds_flags(reset=True) == 0
        checked = fn()
        flags = k.debug_bounds_flags(reset=True)
    assert flags == 0, f"the checked build skipped an access (flags {flags})"
    return released, checked


def _same_step(a: harness.GpuResult, b: harness.GpuResult):
    assert a.err == b.err and not a.err & k.DEVERR_BOUNDS
    assert np.array_equal(a.cache, b.cache)
    assert np.array_equal(a.q, b.q)


def test_library_kinds():
    """The release build records nothing (-1); the checked one starts clean (0).  Under
    DSV4KV_CHECKED=1 the default library is the checked one."""
    import os
    default = 0 if os.environ.get("DSV4KV_CHECKED") == "1" else -1
    assert k.debug_bounds_flags() == default
    with k.checked_build():
        assert k.debug_bounds_flags() == 0


@pytest.mark.parametrize("store", ["fp8", "bf16"])
@pytest.mark.parametrize("bs", [1, 3, 64])
def test_fused_step_every_variant(store, bs):
    wl = configs.generic(777, 5, store=store, seed=300 + bs)
    wl = configs.Workload(wl.name + f"_bs{bs}", wl.T, wl.H, store, wl.max_position,
                          -(-2 * wl.T // bs), bs, wl.seed)
    configs._POSITIONS[wl.name] = lambda w: synth.uniform_int(w.T, w.max_position, w.seed, 4)
    configs._SLOTS[wl.name] = lambda w: configs._random_slots(w, 70)
    inp = harness.make_inputs(wl)
    pos, slots = inp.positions.copy(), inp.slots.copy()
    pos[3], pos[700] = -1, wl.max_position           # positions outside the table
    slots[11], slots[776] = wl.num_slots, wl.num_slots + 5  # slots past the cache
    inp = harness.make_inputs(wl, positions=pos, slots=slots)
    for v in VARIANTS:
        for kv_norm in (True, False):
            a, b = _release_and_checked(lambda: harness.run_gpu(inp, v, kv_norm=kv_norm))
            _same_step(a, b)
            assert a.err == k.DEVERR_POS_RANGE | k.DEVERR_SLOT_RANGE


@pytest.mark.parametrize("store", ["fp8", "bf16"])
@pytest.mark.parametrize("T", [1, 5, 2047, 5003])
def test_kv_rows_only(store, T):
    inp = harness.make_inputs(configs.generic(T, 0, store=store, seed=310 + T))
    for v in VARIANTS[:3]:
        a, b = _release_and_checked(lambda: harness.run_gpu(inp, v))
        _same_step(a, b)


def test_full_prefill_workload():
    """32768 tokens x 64 heads (2.1 GB of q) in the launch configuration the benchmark
    times."""
    inp = harness.make_inputs(configs.PREFILL)
    a, b = _release_and_checked(lambda: harness.run_gpu(inp, q_tokens=np.arange(0, 32768, 97)))
    _same_step(a, b)


def test_kv_rows_past_2_gib():
    """2^21 + 5 KV rows: kv offsets reach 2.15 GB and cache offsets 2.45 GB."""
    inp = harness.make_inputs(configs.generic(2 ** 21 + 5, 0, seed=95, skip_frac=0.01))
    a, b = _release_and_checked(lambda: harness.run_gpu(inp, k.VARIANT_STREAM))
    _same_step(a, b)


def test_reader():
    wl = configs.generic(3001, 2, seed=320)
    inp = harness.make_inputs(wl)
    cache = torch.from_numpy(harness.run_gpu(inp).cache).to(DEV)
    slots = np.concatenate([inp.slots, [-1, wl.num_slots, wl.num_slots + 7, 0]]).astype(np.int64)
    s = torch.from_numpy(slots).to(DEV)

    def read():
        out = torch.full((slots.size, 512), 0x5A5A, dtype=torch.int16, device=DEV)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        k.dequant_gather(cache, wl.num_blocks, wl.block_size, s, out, device_error=err)
        torch.cuda.synchronize()
        return out.cpu().numpy(), int(err.item())

    (a, ea), (b, eb) = _release_and_checked(read)
    assert np.array_equal(a, b) and ea == eb == k.DEVERR_SLOT_RANGE


@pytest.mark.parametrize("bs,offset", [(64, 0), (3, 4)])
def test_indexer_insert_and_gather(bs, offset):
    n = 2500
    nb = -(-2 * n // bs)
    kb = synth.normal_bf16(n * 128, 21, synth.TID_IDX_K).reshape(n, 128)
    sl = synth.permutation(nb * bs, 21, synth.TID_SLOT)[:n].astype(np.int64)
    sl[5], sl[6], sl[7] = -1, nb * bs, nb * bs + 3
    poison = synth.poison_bytes(nb * bs * 132, 21)
    kt = torch.from_numpy(kb.view(np.int16)).to(DEV)
    st = torch.from_numpy(sl).to(DEV)

    def run():
        buf = torch.zeros(nb * bs * 132 + 16, dtype=torch.uint8, device=DEV)
        cache = buf[offset:offset + nb * bs * 132]
        cache.copy_(torch.from_numpy(poison))
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        k.indexer_k_quant_insert(kt, st, cache, nb, bs, device_error=err)
        k_out = torch.full((n, 128), 0xA5, dtype=torch.uint8, device=DEV)
        s_out = torch.full((n,), 7.0, dtype=torch.float32, device=DEV)
        k.indexer_k_gather(cache, nb, bs, st, k_out, s_out, device_error=err)
        torch.cuda.synchronize()
        return cache.cpu().numpy(), k_out.cpu().numpy(), s_out.cpu().numpy(), int(err.item())

    a, b = _release_and_checked(run)
    for x, y in zip(a[:3], b[:3]):
        assert np.array_equal(x, y)
    assert a[3] == b[3] == k.DEVERR_SLOT_RANGE


@pytest.mark.parametrize("m,n", [(1, 128), (129, 7168), (300, 16384)])
def test_mxfp8(m, n):
    x = synth.normal_bf16(m * n, 31, 1).reshape(m, n)
    r = synth.normal_bf16(m * n, 31, 2).reshape(m, n)
    g = synth.normal_bf16(n, 31, 3, std=0.2)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV)

    def run():
        out = torch.empty((m, n), dtype=torch.int16, device=DEV)
        codes = torch.empty((m, n), dtype=torch.uint8, device=DEV)
        scales = torch.full((k.mxfp8_scale_bytes(m, n),), 0xCD, dtype=torch.uint8, device=DEV)
        k.add_gemma_rmsnorm_mxfp8(t(x), t(r), t(g), 1e-6, out, codes, scales)
        torch.cuda.synchronize()
        return out.cpu().numpy(), codes.cpu().numpy(), scales.cpu().numpy()

    a, b = _release_and_checked(run)
    for x_, y_ in zip(a, b):
        assert np.array_equal(x_, y_)
