"""The FP8 cache reader on the GPU against the oracle's reader, bit for bit (the
values are exact, so the one rounding, to bf16, is the same on both sides)."""
import json
import os

import numpy as np
import pytest

import oracle
import synth
from synth import configs
from tests import harness

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import kv_norm_rope_gb300 as k  # noqa: E402

DEV = torch.device("cuda:0")


def _gather_gpu(cache: np.ndarray, num_blocks: int, block_size: int, slots: np.ndarray):
    c = torch.from_numpy(cache).to(DEV)
    s = torch.from_numpy(np.ascontiguousarray(slots, np.int64)).to(DEV)
    out = torch.full((slots.size, 512), 0x5A5A, dtype=torch.int16, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    k.dequant_gather(c, num_blocks, block_size, s, out, device_error=err)
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.uint16), int(err.item())


def _same(a: np.ndarray, b: np.ndarray) -> bool:
    """bit-equal, except that any NaN equals any NaN"""
    nan_a = ((a & 0x7F80) == 0x7F80) & ((a & 0x7F) != 0)
    nan_b = ((b & 0x7F80) == 0x7F80) & ((b & 0x7F) != 0)
    return bool(np.array_equal(nan_a, nan_b) and np.array_equal(a[~nan_a], b[~nan_b]))


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "stress"])
def test_gather_of_inserted_rows(name):
    wl = configs.WORKLOADS[name]
    inp = harness.make_inputs(wl) if wl.T <= 32768 else None
    if inp is None:  # stress: KV rows only (no q) to keep the host copy small
        kv_wl = configs.Workload(wl.name + "_kvonly", wl.T, 0, wl.store, wl.max_position,
                                 wl.num_blocks, wl.block_size, wl.seed, wl.tail_frac, wl.tail_mult)
        configs._POSITIONS[kv_wl.name] = configs._POSITIONS[wl.name]
        configs._SLOTS[kv_wl.name] = configs._SLOTS[wl.name]
        inp = harness.make_inputs(kv_wl)
        wl = kv_wl
    gpu = harness.run_gpu(inp, q_tokens=np.arange(min(wl.T, 4)))
    # the rows in token order, plus skipped and out-of-range slots
    slots = np.concatenate([inp.slots, [-1, wl.num_slots, wl.num_slots + 5, -9]])
    got, err = _gather_gpu(gpu.cache, wl.num_blocks, wl.block_size, slots)
    ref, ref_err = oracle.dequant_gather(gpu.cache, wl.num_blocks, wl.block_size, slots)
    assert err == ref_err == k.DEVERR_SLOT_RANGE
    assert np.array_equal(got, ref)
    assert np.all(got[:wl.T][inp.slots < 0] == 0) and np.all(got[-4:] == 0)


@pytest.mark.parametrize("bs", [1, 3, 64])
def test_gather_of_poisoned_cache(bs):
    """Arbitrary bytes: every E4M3 code (NaN included) and every scale byte 0..255."""
    nb = 4096 // bs + 1
    cache = synth.poison_bytes(nb * bs * 584, seed=bs)
    slots = synth.permutation(nb * bs, 7, 5).astype(np.int64)
    got, err = _gather_gpu(cache, nb, bs, slots)
    ref, ref_err = oracle.dequant_gather(cache, nb, bs, slots)
    assert err == ref_err == 0
    assert _same(got, ref)


GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")))


def test_golden_gather_rows_on_gpu():
    for case in GOLDEN["gather_cases"]:
        src = next(c for c in GOLDEN["kv_cases"] if c["name"] == case["of"])
        cache = np.zeros(584, np.uint8)
        data = []
        for count, val in src["fp8_data"]:
            if isinstance(val, str):
                a = int(val.split(":")[1], 16)
                data += [a & 0xFF, a >> 8] * (2 * count)
            else:
                data += [val] * count
        cache[:576] = data
        sc = []
        for count, val in src["fp8_scale"]:
            sc += [val] * count
        cache[576:] = sc
        got, err = _gather_gpu(cache, 1, 1, np.array([0, -1], np.int64))
        want = []
        for count, val in case["row"]:
            want += [int(val, 16)] * count
        assert err == 0
        assert np.array_equal(got[0], np.array(want, np.uint16)) and np.all(got[1] == 0)


def test_gather_empty_and_rejected():
    out = torch.zeros((0, 512), dtype=torch.int16, device=DEV)
    c = torch.zeros(584, dtype=torch.uint8, device=DEV)
    k.dequant_gather(c, 1, 1, torch.zeros(0, dtype=torch.int64, device=DEV), out)
    with pytest.raises(k.Dsv4Error):
        k.dequant_gather(c, 0, 1, torch.zeros(3, dtype=torch.int64, device=DEV),
                         torch.zeros((3, 512), dtype=torch.int16, device=DEV))


def test_gather_past_2_gib_offsets():
    """A 2.45 GB cache written by the KV-row kernel (2^21 + 5 rows, random slots over
    4.2 M), 262144 of its rows read back in a random order: about 12% of them lie past
    2^31 bytes (slot >= 3.68 M); every row against the oracle's reader."""
    wl = configs.generic(2 ** 21 + 5, 0, seed=96, skip_frac=0.01)
    inp = harness.make_inputs(wl)
    gpu = harness.run_gpu(inp)
    slots = inp.slots[synth.permutation(wl.T, 96, 13)[:262144]]
    assert int((slots >= (2 ** 31) // 584).sum()) > 10000
    got, err = _gather_gpu(gpu.cache, wl.num_blocks, wl.block_size, slots)
    ref, ref_err = oracle.dequant_gather(gpu.cache, wl.num_blocks, wl.block_size, slots)
    assert err == ref_err == 0
    assert np.array_equal(got, ref)
