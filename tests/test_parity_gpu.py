"""GPU parity: the CUDA path (through the C ABI) against the oracle, element by element.

Bar (from the operator's accuracy requirement): cache bytes that are written, UE8M0
scale bytes and untouched bytes bit-exact; E4M3 payload bit-exact except at <= 1e-4
of elements, each at most one E4M3 step away; bf16 outputs within one bf16 ulp.
"""
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
if not torch.cuda.is_available():  # pragma: no cover - CPU runs deselect the gpu mark
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import kv_norm_rope_gb300 as k  # noqa: E402

VARIANTS = [k.VARIANT_AUTO, k.VARIANT_SMALL, k.VARIANT_STREAM, k.VARIANT_HALF]


def _check(wl, variant=k.VARIANT_AUTO, inp=None, store=None):
    """Every q row of every token and every cache byte against the oracle."""
    rep = harness.check(wl, variant, inp, store)
    assert rep.ok, str(rep)
    return rep


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("name", ["tiny", "decode"])
def test_small_workloads(name, variant):
    _check(configs.WORKLOADS[name], variant)


@pytest.mark.parametrize("store", ["fp8", "bf16"])
@pytest.mark.parametrize("H", [8, 64, 128])
@pytest.mark.parametrize("T", [1, 4, 17, 511, 512, 777, 1000, 4096])
def test_shape_sweep(T, H, store):
    _check(configs.generic(T, H, store=store, seed=1000 + T + H))


@pytest.mark.parametrize("name", ["prefill", "bf16_store", "stress"])
def test_full_size_workloads(name):
    """Full sizes in the launch configuration the benchmark times (AUTO): every
    cache byte and every token's q rows compared (q checked in token chunks after
    the one whole-batch launch)."""
    rep = _check(configs.WORKLOADS[name], k.VARIANT_AUTO)
    wl = configs.WORKLOADS[name]
    assert rep.q_rows == wl.T * wl.H, rep.q_rows


def test_heavy_tails_all_variants():
    wl = configs.generic(3000, 16, seed=77, tail_frac=0.01, tail_mult=100.0)
    inp = harness.make_inputs(wl)
    for v in VARIANTS:
        _check(wl, v, inp=inp)


@pytest.mark.parametrize("store", ["fp8", "bf16"])
@pytest.mark.parametrize("bs", [1, 3, 7, 64, 256, 1024])
def test_block_sizes(bs, store):
    """Odd block sizes put FP8 data rows on 8-byte (not 16-byte) boundaries; large
    ones put a whole batch in one or two blocks."""
    wl = configs.generic(200, 4, seed=bs)
    wl = configs.Workload(wl.name + f"_bs{bs}_{store}", wl.T, wl.H, store, wl.max_position,
                          -(-2 * wl.T // bs), bs, wl.seed)
    configs._POSITIONS[wl.name] = lambda w: synth.uniform_int(w.T, w.max_position, w.seed, 4)
    configs._SLOTS[wl.name] = lambda w: configs._random_slots(w, 17)
    for v in VARIANTS:
        _check(wl, v)


def test_single_head_alternating_rows():
    for store in ("fp8", "bf16"):
        wl = configs.generic(999, 1, store=store, seed=5)
        for v in VARIANTS:
            _check(wl, v)


# ---------------------------------------------------------------- hand cases on the GPU

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")))


def _bf16(v):
    return int(np.array([v], np.float32).view(np.uint32)[0]) >> 16


def _row(runs):
    out = []
    for count, val in runs:
        if isinstance(val, str) and val.startswith("pair:"):
            a, b = (float(t) for t in val[5:].split(","))
            out += [_bf16(a), _bf16(b)] * count
        else:
            out += [_bf16(float(val))] * count
    return np.array(out, np.uint16)


def _bytes(runs, n):
    out = []
    for count, val in runs:
        if isinstance(val, str) and val.startswith("bf16le_pair:"):
            a, b = (int(t, 16) for t in val[12:].split(","))
            out += [a & 0xFF, a >> 8, b & 0xFF, b >> 8] * count
        elif isinstance(val, str) and val.startswith("bf16le:"):
            a = int(val[7:], 16)
            out += [a & 0xFF, a >> 8] * (2 * count)
        else:
            out += [int(val)] * count
    assert len(out) == n
    return np.array(out, np.uint8)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("case", GOLDEN["kv_cases"], ids=lambda c: c["name"])
def test_golden_kv_rows_on_gpu(case, variant):
    """Hand-derived cache bytes, including amax exactly on 448*2^-4 and just above."""
    ident = np.array([1.0] * 32 + [0.0] * 32, np.float32)
    quarter = np.array([0.0] * 32 + [1.0] * 32, np.float32)
    table = np.stack([ident, quarter])
    x = _row(case["kv"])
    w = _row(case["w"])
    pos = 0 if case["cos_sin"] == "identity" else 1
    T = 3
    wl = configs.Workload("golden_" + case["name"], T, 2, "fp8", 2, 1, 4, 0, eps=case["eps"])
    q = np.stack([np.stack([_row([[512, -4.0]]), x])] * T)
    inp = harness.Inputs(wl, np.ascontiguousarray(q), np.stack([x] * T), w,
                         np.full(T, pos, np.int64), np.array([2, -1, 0], np.int64), table,
                         synth.poison_bytes(4 * 584, seed=1))
    gpu = harness.run_gpu(inp, variant)
    assert gpu.err == 0
    expect = inp.poison.copy()
    for slot in (2, 0):
        expect[576 * slot:576 * slot + 576] = _bytes(case["fp8_data"], 576)
        expect[2304 + 8 * slot:2304 + 8 * slot + 8] = _bytes(case["fp8_scale"], 8)
    assert np.array_equal(gpu.cache, expect)
    ref_q, ref_cache, _ = harness.run_oracle(inp)
    assert np.array_equal(ref_cache, expect)
    rep = harness.compare_results(inp, gpu, ref_q, ref_cache)
    assert rep.ok, str(rep)


@pytest.mark.parametrize("case", GOLDEN["q_cases"], ids=lambda c: c["name"])
def test_golden_q_rows_on_gpu(case):
    ident = np.array([1.0] * 32 + [0.0] * 32, np.float32)
    quarter = np.array([0.0] * 32 + [1.0] * 32, np.float32)
    x = _row(case["x"])
    wl = configs.Workload("golden_q_" + case["name"], 2, 3, "fp8", 2, 1, 4, 0, eps=case["eps"])
    pos = 0 if case["cos_sin"] == "identity" else 1
    inp = harness.Inputs(wl, np.ascontiguousarray(np.stack([np.stack([x] * 3)] * 2)),
                         np.stack([x] * 2), _row([[512, 1.0]]), np.full(2, pos, np.int64),
                         np.array([-1, -1], np.int64), np.stack([ident, quarter]),
                         synth.poison_bytes(4 * 584, seed=2))
    gpu = harness.run_gpu(inp)
    want = []
    for count, val in case["out"]:
        if val.startswith("pair:"):
            a, b = (int(t, 16) for t in val[5:].split(","))
            want += [a, b] * count
        else:
            want += [int(val, 16)] * count
    want = np.array(want, np.uint16)
    for t in range(2):
        for h in range(3):
            assert np.array_equal(gpu.q[t, h], want)
    assert np.array_equal(gpu.cache, inp.poison)


def _near_boundary_rows(n_scan=200_000, seed=31, band=2.0**-13):
    """KV rows (with the weight) whose exact block amax lies within a relative
    `band` of some 448*2^k: screened in numpy fp64, then judged by the oracle."""
    wl = configs.generic(n_scan, 1, seed=seed)
    kv = configs.kv_bits(wl).reshape(n_scan, 512)
    w = configs.weight_bits(wl)
    wd = oracle.bf16_value(w)
    keep = []
    for c0 in range(0, n_scan, 20000):
        x = oracle.bf16_value(kv[c0:c0 + 20000])
        r = 1.0 / np.sqrt(np.sum(x * x, axis=1) / 512 + np.float64(np.float32(1e-6)))
        v = np.abs(x[:, :448] * r[:, None] * wd[None, :448]).reshape(-1, 7, 64).max(axis=2)
        l2 = np.log2(v / 448.0)
        dist = np.abs(l2 - np.round(l2))
        keep.append(c0 + np.nonzero((dist < band / np.log(2)).any(axis=1))[0])
    return np.concatenate(keep), kv, w


def test_scale_decisions_near_boundaries():
    """Rows whose block amax sits within 2^-13 of a UE8M0 boundary: the kernel's fp32
    guess is too close to call there, so its exact fallback path decides them."""
    rows, kv_all, w = _near_boundary_rows()
    assert rows.size >= 100
    T = int(rows.size)
    wl = configs.Workload("near_boundary", T, 1, "fp8", 1, -(-T // 64), 64, 31)
    ident = np.array([[1.0] * 32 + [0.0] * 32], np.float32)
    inp = harness.Inputs(wl, np.ascontiguousarray(kv_all[rows][:, None, :]),
                         np.ascontiguousarray(kv_all[rows]), w, np.zeros(T, np.int64),
                         np.arange(T, dtype=np.int64), ident,
                         synth.poison_bytes(wl.num_slots * 584, seed=3))
    for v in VARIANTS:
        gpu = harness.run_gpu(inp, v)
        ref_q, ref_cache, _ = harness.run_oracle(inp)
        rep = harness.compare_results(inp, gpu, ref_q, ref_cache)
        assert rep.ok, str(rep)


# ---------------------------------------------------------------- edges

def test_zero_tokens_touch_nothing():
    cache = torch.full((584 * 64,), 0xA5, dtype=torch.uint8, device="cuda")
    q = torch.empty(0, 8, 512, dtype=torch.bfloat16, device="cuda")
    e = torch.empty(0, 512, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(512, dtype=torch.bfloat16, device="cuda")
    i = torch.empty(0, dtype=torch.int64, device="cuda")
    cs = torch.zeros(16, 64, device="cuda")
    k.qnorm_rope_kv_quant_insert(q, e, w, i, cs, i, cache, 1, 64, 1e-6)
    torch.cuda.synchronize()
    assert bool((cache == 0xA5).all())


def test_runs_on_a_side_stream():
    wl = configs.TINY
    inp = harness.make_inputs(wl)
    dev = torch.device("cuda:0")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        q = torch.from_numpy(inp.q.view(np.int16)).view(torch.bfloat16).to(dev)
        kv = torch.from_numpy(inp.kv.view(np.int16)).view(torch.bfloat16).to(dev)
        w = torch.from_numpy(inp.w.view(np.int16)).view(torch.bfloat16).to(dev)
        pos = torch.from_numpy(inp.positions).to(dev)
        sl = torch.from_numpy(inp.slots).to(dev)
        cs = torch.from_numpy(inp.cos_sin).to(dev)
        cache = torch.from_numpy(inp.poison).to(dev)
        k.qnorm_rope_kv_quant_insert(q, kv, w, pos, cs, sl, cache, wl.num_blocks, wl.block_size,
                                     wl.eps, stream=s)
    s.synchronize()
    ref_q, ref_cache, _ = harness.run_oracle(inp)
    gpu = harness.GpuResult(np.arange(wl.T), q.cpu().view(torch.int16).numpy().view(np.uint16)
                            .reshape(wl.T, wl.H, 512), cache.cpu().numpy(), 0)
    rep = harness.compare_results(inp, gpu, ref_q, ref_cache)
    assert rep.ok, str(rep)


# ---------------------------------------------------------------- KV arriving normalised / KV only

@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("store", ["fp8", "bf16"])
def test_prenormalised_kv(store, variant):
    """The FlagGems operator form: q-norm + rope, KV rope + quant + insert (no KV norm)."""
    for T, H in [(17, 8), (1000, 64), (333, 1)]:
        rep = harness.check(configs.generic(T, H, store=store, seed=2000 + T), variant,
                            kv_norm=False)
        assert rep.ok, str(rep)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("store", ["fp8", "bf16"])
def test_kv_rows_only(store, variant):
    """The SGLang fused_norm_rope_flashmla form: KV rows only, no q."""
    for T in (1, 64, 2048, 5000):
        rep = harness.check(configs.generic(T, 0, store=store, seed=3000 + T), variant)
        assert rep.ok, str(rep)


@pytest.mark.parametrize("case", GOLDEN["prenormalised_kv_cases"], ids=lambda c: c["name"])
def test_golden_prenormalised_rows_on_gpu(case):
    ident = np.array([1.0] * 32 + [0.0] * 32, np.float32)
    quarter = np.array([0.0] * 32 + [1.0] * 32, np.float32)
    x = _row(case["kv"])
    pos = 0 if case["cos_sin"] == "identity" else 1
    wl = configs.Workload("golden_pn_" + case["name"], 2, 1, "fp8", 2, 1, 4, 0, eps=0.0)
    inp = harness.Inputs(wl, np.ascontiguousarray(np.stack([x[None]] * 2)), np.stack([x] * 2),
                         np.zeros(512, np.uint16), np.full(2, pos, np.int64),
                         np.array([3, 1], np.int64), np.stack([ident, quarter]),
                         synth.poison_bytes(4 * 584, seed=4))
    for v in VARIANTS:
        gpu = harness.run_gpu(inp, v, kv_norm=False)
        expect = inp.poison.copy()
        for slot in (3, 1):
            expect[576 * slot:576 * slot + 576] = _bytes(case["fp8_data"], 576)
            expect[2304 + 8 * slot:2304 + 8 * slot + 8] = _bytes(case["fp8_scale"], 8)
        assert np.array_equal(gpu.cache, expect)


@pytest.mark.parametrize("name", ["prefill", "stress"])
def test_full_size_kv_only_and_prenormalised(name):
    wl = configs.WORKLOADS[name]
    kv_wl = configs.Workload(wl.name + "_kvonly", wl.T, 0, wl.store, wl.max_position,
                             wl.num_blocks, wl.block_size, wl.seed, wl.tail_frac, wl.tail_mult)
    configs._POSITIONS[kv_wl.name] = configs._POSITIONS[wl.name]
    configs._SLOTS[kv_wl.name] = configs._SLOTS[wl.name]
    rep = harness.check(kv_wl, k.VARIANT_AUTO)
    assert rep.ok, str(rep)
    if name == "prefill":
        rep = harness.check(wl, k.VARIANT_AUTO, kv_norm=False)
        assert rep.ok, str(rep)


def test_public_entries_match_ex():
    """dsv4_qnorm_rope_kv_rope_quant_insert and dsv4_kv_norm_rope_insert give the same
    bytes as the general entry with the corresponding flags."""
    wl = configs.generic(700, 16, seed=41)
    inp = harness.make_inputs(wl)
    dev = torch.device("cuda:0")
    t = lambda a: torch.from_numpy(a).to(dev)
    q = t(inp.q.view(np.int16)).view(torch.bfloat16)
    kv = t(inp.kv.view(np.int16)).view(torch.bfloat16)
    w = t(inp.w.view(np.int16)).view(torch.bfloat16)
    cache = t(inp.poison)
    k.qnorm_rope_kv_rope_quant_insert(q, kv, t(inp.positions), t(inp.cos_sin), t(inp.slots), cache,
                                      wl.num_blocks, wl.block_size, wl.eps)
    torch.cuda.synchronize()
    ref = harness.run_gpu(inp, kv_norm=False)
    assert np.array_equal(cache.cpu().numpy(), ref.cache)
    assert np.array_equal(q.cpu().view(torch.int16).numpy().view(np.uint16), ref.q)
    cache2 = t(inp.poison)
    k.kv_norm_rope_insert(k.STORE_FP8, kv, w, t(inp.positions), t(inp.cos_sin), t(inp.slots),
                          cache2, wl.num_blocks, wl.block_size, wl.eps)
    torch.cuda.synchronize()
    ref2 = harness.run_gpu(inp)
    assert np.array_equal(cache2.cpu().numpy(), ref2.cache)


@pytest.mark.parametrize("variant", VARIANTS)
def test_positions_at_both_ends_of_the_table(variant):
    """Positions 0 and max_position - 1 (the last row of the cos/sin table) are in
    range; max_position is the first one out of range."""
    wl = configs.generic(64, 8, seed=140, max_position=1000, skip_frac=0.0)
    pos = np.where(np.arange(64) % 3 == 0, 0, 999).astype(np.int64)
    pos[5] = 1000
    inp = harness.make_inputs(wl, positions=pos)
    gpu = harness.run_gpu(inp, variant)
    ref_q, ref_cache, ref_err = harness.run_oracle(inp)
    assert gpu.err == ref_err == k.DEVERR_POS_RANGE
    rep = harness.compare_results(inp, gpu, ref_q, ref_cache)
    assert rep.ok, str(rep)


@pytest.mark.parametrize("store", ["fp8", "bf16"])
def test_host_resident_buffers(store):
    """Pinned host memory is addressable by the kernels at the same address (NVLink-C2C
    on GB300): the step run through the C ABI on host-resident q, kv, positions, slots and
    cache writes the bytes the device-resident run writes."""
    wl = configs.generic(3000, 16, store=store, seed=160)
    inp = harness.make_inputs(wl)
    ref = harness.run_gpu(inp)
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    q, kv = pin(inp.q.view(np.int16)), pin(inp.kv.view(np.int16))
    pos, sl, cache = pin(inp.positions), pin(inp.slots), pin(inp.poison)
    dev = torch.device("cuda:0")
    w = torch.from_numpy(inp.w.view(np.int16)).to(dev)
    cs = torch.from_numpy(inp.cos_sin).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    fn = (k.lib().dsv4_qnorm_rope_kv_quant_insert if store == "fp8"
          else k.lib().dsv4_qnorm_rope_kv_bf16_insert)
    st = fn(q.data_ptr(), kv.data_ptr(), w.data_ptr(), pos.data_ptr(), cs.data_ptr(),
            wl.max_position, sl.data_ptr(), cache.data_ptr(), wl.num_blocks, wl.block_size, wl.T,
            wl.H, wl.eps, err.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == k.OK
    torch.cuda.synchronize()
    assert int(err.item()) == ref.err
    assert np.array_equal(q.numpy().view(np.uint16), ref.q)
    assert np.array_equal(cache.numpy(), ref.cache)
