"""Out-of-range device data is reported through the error word and its writes are
skipped; nothing traps or waits.  Compared with the oracle, which skips the same
writes and reports the same bits."""
import numpy as np
import pytest

from synth import configs
from tests import harness

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import kv_norm_rope_gb300 as k  # noqa: E402


def _faulty_inputs(store):
    wl = configs.generic(40, 6, store=store, seed=404)
    inp = harness.make_inputs(wl)
    pos = inp.positions.copy()
    slots = inp.slots.copy()
    pos[3] = -1                    # before the table
    pos[7] = wl.max_position       # one past the table
    slots[11] = wl.num_slots       # one past the cache
    slots[12] = wl.num_slots + 999
    slots[13] = -7                 # any negative slot: skip, no error
    return harness.make_inputs(wl, positions=pos, slots=slots)


@pytest.mark.parametrize("variant", [k.VARIANT_AUTO, k.VARIANT_SMALL, k.VARIANT_STREAM,
                                     k.VARIANT_HALF])
@pytest.mark.parametrize("store", ["fp8", "bf16"])
def test_out_of_range_flagged_and_skipped(store, variant):
    inp = _faulty_inputs(store)
    gpu = harness.run_gpu(inp, variant)
    ref_q, ref_cache, ref_err = harness.run_oracle(inp)
    assert gpu.err == ref_err == (k.DEVERR_POS_RANGE | k.DEVERR_SLOT_RANGE)
    rep = harness.compare_results(inp, gpu, ref_q, ref_cache)
    assert rep.ok, str(rep)
    # tokens with a bad position keep their q rows unchanged
    assert np.array_equal(gpu.q[3], inp.q[3]) and np.array_equal(gpu.q[7], inp.q[7])


def test_error_word_is_optional():
    inp = _faulty_inputs("fp8")
    wl = inp.wl
    dev = torch.device("cuda:0")
    t = lambda a: torch.from_numpy(a).to(dev)
    q = t(inp.q.view(np.int16)).view(torch.bfloat16)
    kv = t(inp.kv.view(np.int16)).view(torch.bfloat16)
    w = t(inp.w.view(np.int16)).view(torch.bfloat16)
    cache = t(inp.poison)
    k.qnorm_rope_kv_quant_insert(q, kv, w, t(inp.positions), t(inp.cos_sin), t(inp.slots), cache,
                                 wl.num_blocks, wl.block_size, wl.eps, device_error=None)
    torch.cuda.synchronize()
    _, ref_cache, _ = harness.run_oracle(inp)
    rep = harness.compare_results(inp, harness.GpuResult(
        np.arange(wl.T), q.cpu().view(torch.int16).numpy().view(np.uint16).reshape(wl.T, wl.H, 512),
        cache.cpu().numpy(), 0), harness.run_oracle(inp)[0], ref_cache)
    assert rep.ok, str(rep)


def test_rejected_call_launches_nothing():
    cache = torch.full((584 * 64,), 0x5A, dtype=torch.uint8, device="cuda")
    q = torch.ones(4, 2, 512, dtype=torch.bfloat16, device="cuda")
    kv = torch.ones(4, 512, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(512, dtype=torch.bfloat16, device="cuda")
    i = torch.zeros(4, dtype=torch.int64, device="cuda")
    cs = torch.zeros(16, 64, device="cuda")
    with pytest.raises(k.Dsv4Error) as ex:
        k.qnorm_rope_kv_quant_insert(q, kv, w, i, cs, i, cache, 1, 64, -1.0)  # negative eps
    assert ex.value.status == k.ERR_VALUE
    torch.cuda.synchronize()
    assert bool((cache == 0x5A).all()) and bool((q == 1).all())


def test_bounded_wait_runs_out_and_reports():
    """A wait that nothing completes gives up after its cycle budget, ORs the timeout bit
    into the error word and returns; the context stays usable for the next launch."""
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    k.check_bounded_wait(1 << 24, err)  # ~8 ms at 2 GHz
    t1.record()
    torch.cuda.synchronize()
    assert int(err.item()) == k.DEVERR_TIMEOUT
    ms = t0.elapsed_time(t1)
    assert 1e3 * (1 << 24) / 2.2e9 <= ms < 1000.0, ms
    # the kernels' own limit (about a second), with no error word
    k.check_bounded_wait(0, None)
    torch.cuda.synchronize()
    rep = harness.check(configs.TINY)
    assert rep.ok, str(rep)
