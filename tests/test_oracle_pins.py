"""Pins of the oracle's row algebra, quantiser and cache layout (CPU only).

Each check is tied to something other than the oracle itself: hand-derived
bytes (tests/golden/hand_cases.json, each case citing the passage it follows),
numpy complex multiplication for the rotation, closed forms for the RMS norm,
the E4M3 rounding bound for the payload, and a brute-force 4-token case whose
expected cache image is assembled from the hand-derived rows at hand-computed
offsets.  Together they fail on a dropped term (eps, weight, 1/512), a wrong
sign or index in the rotation, swapped cos/sin columns, a wrong scale rule,
or a misplaced cache byte.
"""
import json
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")
with open(GOLDEN) as f:
    CASES = json.load(f)

F32_IDENTITY = np.array([1.0] * 32 + [0.0] * 32, dtype=np.float32)
F32_QUARTER = np.array([0.0] * 32 + [1.0] * 32, dtype=np.float32)


def _bf16(v: float) -> int:
    """bits of a bf16-exact float (checked)"""
    b = int(np.array([v], dtype=np.float32).view(np.uint32)[0]) >> 16
    assert float(np.array([b << 16], dtype=np.uint32).view(np.float32)[0]) == v
    return b


def _expand_values(runs):
    out = []
    for count, val in runs:
        if isinstance(val, str) and val.startswith("pair:"):
            a, b = (float(t) for t in val[5:].split(","))
            out += [_bf16(a), _bf16(b)] * count
        else:
            out += [_bf16(float(val))] * count
    assert len(out) == 512
    return np.array(out, dtype=np.uint16)


def _expand_bytes(runs, n):
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
    assert len(out) == n, (len(out), n)
    return np.array(out, dtype=np.uint8)


def _expand_bf16_row(runs):
    out = []
    for count, val in runs:
        if val.startswith("pair:"):
            a, b = (int(t, 16) for t in val[5:].split(","))
            out += [a, b] * count
        else:
            out += [int(val, 16)] * count
    assert len(out) == 512
    return np.array(out, dtype=np.uint16)


def _table(kind):
    return {"identity": F32_IDENTITY, "quarter_turn": F32_QUARTER}[kind]


@pytest.mark.parametrize("case", CASES["kv_cases"], ids=lambda c: c["name"])
def test_golden_kv_fp8_slot(case):
    x = _expand_values(case["kv"])
    w = _expand_values(case["w"])
    v = oracle.kv_values(x, w, _table(case["cos_sin"]), case["eps"])
    data, scale = oracle.fp8_slot(v)
    assert np.array_equal(data, _expand_bytes(case["fp8_data"], 576))
    assert np.array_equal(scale, _expand_bytes(case["fp8_scale"], 8))


@pytest.mark.parametrize("case", [c for c in CASES["kv_cases"] if "bf16_row" in c],
                         ids=lambda c: c["name"])
def test_golden_kv_bf16_row(case):
    x = _expand_values(case["kv"])
    w = _expand_values(case["w"])
    v = oracle.kv_values(x, w, _table(case["cos_sin"]), case["eps"])
    assert np.array_equal(oracle.bf16_rne(v), _expand_bf16_row(case["bf16_row"]))


@pytest.mark.parametrize("case", CASES["q_cases"], ids=lambda c: c["name"])
def test_golden_q_row(case):
    x = _expand_values(case["x"])
    y = oracle.q_values(x, _table(case["cos_sin"]), case["eps"])
    assert np.array_equal(oracle.bf16_rne(y), _expand_bf16_row(case["out"]))


def _rand_row(seed, tid=1):
    return synth.normal_bf16(512, seed, tid)


def test_rotation_matches_complex_multiply():
    """Pairs (448+2i, 449+2i) turn by angle i of the row: cos in column i, sin in 32+i."""
    table = synth.cos_sin_table(4096)
    for seed, p in [(1, 1), (2, 1234), (3, 4095), (4, 77)]:
        x = _rand_row(seed)
        xd = oracle.bf16_value(x)
        r = 1.0 / np.sqrt(np.mean(xd * xd) + np.float64(np.float32(1e-6)))
        y = oracle.q_values(x, table[p], 1e-6)
        z = (xd[448::2] + 1j * xd[449::2]) * r
        rot = z * (table[p, :32].astype(np.float64) + 1j * table[p, 32:].astype(np.float64))
        assert np.allclose(y[448::2], rot.real, rtol=0, atol=1e-12)
        assert np.allclose(y[449::2], rot.imag, rtol=0, atol=1e-12)
        assert np.allclose(y[:448], xd[:448] * r, rtol=1e-15, atol=0)


def test_position_zero_is_identity():
    table = synth.cos_sin_table(8)
    assert np.array_equal(table[0], F32_IDENTITY)
    for seed in range(5):
        x = _rand_row(seed)
        y = oracle.q_values(x, table[0], 1e-6)
        xd = oracle.bf16_value(x)
        r = 1.0 / np.sqrt(np.sum(xd * xd) / 512 + np.float64(np.float32(1e-6)))
        assert np.array_equal(y, xd * r)


def test_rotation_preserves_pair_norms():
    table = synth.cos_sin_table(4096)
    w = synth.normal_bf16(512, 9, 3, mean=1.0, std=0.1)
    for seed, p in [(11, 3), (12, 999), (13, 4000)]:
        x = _rand_row(seed, 2)
        v0 = oracle.kv_values(x, w, table[0], 1e-6)
        v = oracle.kv_values(x, w, table[p], 1e-6)
        c = table[p, :32].astype(np.float64)
        s = table[p, 32:].astype(np.float64)
        n0 = v0[448::2] ** 2 + v0[449::2] ** 2
        n1 = v[448::2] ** 2 + v[449::2] ** 2
        assert np.allclose(n1, n0 * (c * c + s * s), rtol=1e-13, atol=0)
        assert np.array_equal(v[:448], v0[:448])


def test_rms_closed_forms():
    ones = np.full(512, _bf16(1.0), dtype=np.uint16)
    for seed in range(6):
        x = _rand_row(seed, 2)
        xd = oracle.bf16_value(x)
        ms = np.mean(xd * xd)
        v = oracle.kv_values(x, ones, F32_IDENTITY, 0.0)
        assert abs(np.mean(v * v) - 1.0) < 1e-14
        eps = float(np.float32(0.37))
        v = oracle.kv_values(x, ones, F32_IDENTITY, eps)
        assert abs(np.mean(v * v) - ms / (ms + eps)) < 1e-14
        y = oracle.q_values(x, F32_IDENTITY, 0.0)
        assert abs(np.mean(y * y) - 1.0) < 1e-14


def test_weight_scales_each_dim():
    x = _rand_row(21, 2)
    ones = np.full(512, _bf16(1.0), dtype=np.uint16)
    base = oracle.kv_values(x, ones, F32_IDENTITY, 1e-6)
    for j in (0, 63, 64, 300, 447, 448, 511):
        w = ones.copy()
        w[j] = _bf16(2.0)
        v = oracle.kv_values(x, w, F32_IDENTITY, 1e-6)
        expect = base.copy()
        expect[j] *= 2
        assert np.array_equal(v, expect)


def _e4m3_decode(codes):
    codes = codes.astype(np.int64)
    sign = np.where(codes & 0x80, -1.0, 1.0)
    e = (codes >> 3) & 0xF
    m = codes & 7
    mag = np.where(e == 0, m * 2.0**-9, (8 + m) * np.ldexp(1.0, e - 10))
    return sign * mag


def test_quantisation_bound_and_minimal_scale():
    """Dequantised payload lies within half an E4M3 step (times the block scale)
    of v, and s is the smallest exponent whose 448 * 2^s covers amax."""
    table = synth.cos_sin_table(4096)
    w = synth.normal_bf16(512, 5, 3, mean=1.0, std=0.1)
    for seed in range(40):
        x = synth.normal_bf16(512, 100 + seed, 2, tail_frac=0.05, tail_mult=100.0, tail_id=10)
        v = oracle.kv_values(x, w, table[seed * 97 % 4096], 1e-6)
        data, scale = oracle.fp8_slot(v)
        assert scale[7] == 0
        for b in range(7):
            blk = v[64 * b:64 * b + 64]
            s = int(scale[b]) - 127
            amax = np.max(np.abs(blk))
            assert amax <= 448.0 * 2.0**s
            assert s == -127 or amax > 448.0 * 2.0 ** (s - 1)
            deq = _e4m3_decode(data[64 * b:64 * b + 64]) * 2.0**s
            a = np.abs(blk) * 2.0**-s
            e = np.floor(np.log2(np.maximum(a, 2.0**-6)))
            half_step = 2.0 ** (e - 3) / 2 * 2.0**s
            assert np.all(np.abs(deq - blk) <= half_step * (1 + 1e-12))
        rope = data[448:].view(np.uint16)
        assert np.array_equal(rope, oracle.bf16_rne(v[448:]))


def _rows_for(name):
    c = next(c for c in CASES["kv_cases"] if c["name"] == name)
    return c, _expand_values(c["kv"]), _expand_values(c["w"])


def test_brute_force_four_tokens_layout_and_skips():
    """4 tokens, 2 blocks x 4 slots, w = 1, eps 0.  Table row 0 is the identity,
    row 1 the quarter turn.  Slot 5 = block 1 offset 1, slot -1 = skipped,
    slot 0 = block 0 offset 0, slot 7 = block 1 offset 3.  FP8 block b starts
    at b*4*584; slot o's data at +576*o, its scale at +4*576 + 8*o.  Every
    other byte keeps the poison.  q (one head, the Q1 row) comes back equal to
    its input at position 0 (r = 1) and as the Q1 image at position 1."""
    h1, x_h1, w1 = _rows_for("H1_constant_row")
    h2, x_h2, _ = _rows_for("H2_single_spike")
    h3, x_h3, _ = _rows_for("H3_quarter_turn_kv")
    q1 = next(c for c in CASES["q_cases"] if c["name"] == "Q1_quarter_turn")
    qx = _expand_values(q1["x"])
    kv = np.stack([x_h1, x_h2, x_h2, x_h3])
    q = np.ascontiguousarray(np.stack([qx] * 4).reshape(4, 1, 512))
    positions = np.array([0, 0, 0, 1], dtype=np.int64)
    slots = np.array([5, -1, 0, 7], dtype=np.int64)
    table = np.stack([F32_IDENTITY, F32_QUARTER])
    poison = synth.poison_bytes(2 * 4 * 584, seed=3)
    cache = poison.copy()
    err = oracle.qnorm_rope_kv_insert("fp8", q, kv, w1, positions, table, slots, cache, 2, 4, 0.0)
    assert err == 0
    expect = poison.copy()

    def put(case, slot):
        blk, off = divmod(slot, 4)
        base = blk * 4 * 584
        expect[base + 576 * off: base + 576 * off + 576] = _expand_bytes(case["fp8_data"], 576)
        expect[base + 2304 + 8 * off: base + 2304 + 8 * off + 8] = _expand_bytes(case["fp8_scale"], 8)

    put(h1, 5)
    put(h2, 0)
    put(h3, 7)
    assert np.array_equal(cache, expect)
    for t in range(3):
        assert np.array_equal(q[t, 0], qx)
    assert np.array_equal(q[3, 0], _expand_bf16_row(q1["out"]))


def test_bf16_store_layout_and_skips():
    c, x, w = _rows_for("H2_single_spike")
    poison = synth.poison_bytes(3 * 2 * 1024, seed=4)
    cache = poison.copy()
    kv = np.stack([x, x, x])
    slots = np.array([4, -1, 1], dtype=np.int64)
    err = oracle.qnorm_rope_kv_insert("bf16", None, kv, w, np.zeros(3, np.int64),
                                      synth.cos_sin_table(1), slots, cache, 3, 2, 0.0)
    assert err == 0
    expect = poison.copy()
    row = _expand_bf16_row(c["bf16_row"]).view(np.uint8)
    expect[4 * 1024:5 * 1024] = row
    expect[1 * 1024:2 * 1024] = row
    assert np.array_equal(cache, expect)


def test_out_of_range_slot_and_position_are_flagged_and_skipped():
    c, x, w = _rows_for("H1_constant_row")
    poison = synth.poison_bytes(584 * 4, seed=5)
    cache = poison.copy()
    q = np.ascontiguousarray(np.stack([_expand_values([[512, -4.0]])] * 3).reshape(3, 1, 512))
    q0 = q.copy()
    kv = np.stack([x, x, x])
    positions = np.array([0, 2, 0], dtype=np.int64)      # 2 is past a 2-row table
    slots = np.array([4, 0, 1], dtype=np.int64)          # 4 is past 1 block x 4 slots
    err = oracle.qnorm_rope_kv_insert("fp8", q, kv, w, positions, synth.cos_sin_table(2), slots,
                                      cache, 1, 4, 0.0)
    assert err == oracle.ERR_SLOT_RANGE | oracle.ERR_POS_RANGE
    assert np.all(q[0] == _bf16(-1.0)) and np.array_equal(q[1], q0[1]) and np.all(q[2] == _bf16(-1.0))
    expect = poison.copy()
    expect[576:1152] = _expand_bytes(c["fp8_data"], 576)
    expect[2304 + 8:2304 + 16] = _expand_bytes(c["fp8_scale"], 8)
    assert np.array_equal(cache, expect)


def test_thread_split_does_not_change_bits():
    from synth import configs
    wl = configs.generic(300, 4, seed=8)
    q = configs.q_bits(wl).reshape(wl.T, wl.H, 512)
    kv = configs.kv_bits(wl)
    outs = []
    for nt in (1, 3, 8):
        qq = q.copy()
        cache = synth.poison_bytes(configs.cache_bytes(wl), seed=1)
        oracle.qnorm_rope_kv_insert("fp8", qq, kv, configs.weight_bits(wl), wl.positions(),
                                    configs.cos_sin(wl), wl.slot_mapping(), cache, wl.num_blocks,
                                    wl.block_size, wl.eps, n_threads=nt)
        outs.append((qq, cache))
    for qq, cache in outs[1:]:
        assert np.array_equal(qq, outs[0][0]) and np.array_equal(cache, outs[0][1])


@pytest.mark.parametrize("case", CASES["prenormalised_kv_cases"], ids=lambda c: c["name"])
def test_golden_prenormalised_kv_rows(case):
    """KV rows that arrive normalised: rotation and quantisation only."""
    x = _expand_values(case["kv"])
    v = oracle.kv_rope_values(x, _table(case["cos_sin"]))
    data, scale = oracle.fp8_slot(v)
    assert np.array_equal(data, _expand_bytes(case["fp8_data"], 576))
    assert np.array_equal(scale, _expand_bytes(case["fp8_scale"], 8))
    if "bf16_row" in case:
        assert np.array_equal(oracle.bf16_rne(v), _expand_bf16_row(case["bf16_row"]))


def test_prenormalised_driver_ignores_weight_and_eps():
    """Through the batch driver (KV only, no q): the weight and eps do not enter the
    KV rows when they arrive normalised, and a row of exact RMS 1 with w = 1 and
    eps = 0 gives the same image with or without the norm."""
    h3, x_h3, w1 = _rows_for("H3_quarter_turn_kv")
    pn2 = next(c for c in CASES["prenormalised_kv_cases"] if c["name"] == "PN2_not_renormalised")
    x_pn2 = _expand_values(pn2["kv"])
    table = np.stack([F32_IDENTITY, F32_QUARTER])
    poison = synth.poison_bytes(4 * 584, seed=9)
    kv = np.stack([x_h3, x_pn2])
    pos = np.array([1, 0], np.int64)
    slots = np.array([3, 1], np.int64)
    w_odd = synth.normal_bf16(512, 3, 3, mean=1.0, std=0.5)
    for w, eps in [(w1, 0.0), (w_odd, 0.25)]:
        cache = poison.copy()
        err = oracle.qnorm_rope_kv_insert("fp8", None, kv, w, pos, table, slots, cache, 1, 4, eps,
                                          kv_norm=False)
        assert err == 0
        expect = poison.copy()
        expect[576 * 3:576 * 4] = _expand_bytes(h3["fp8_data"], 576)
        expect[2304 + 24:2304 + 32] = _expand_bytes(h3["fp8_scale"], 8)
        expect[576:1152] = _expand_bytes(pn2["fp8_data"], 576)
        expect[2304 + 8:2304 + 16] = _expand_bytes(pn2["fp8_scale"], 8)
        assert np.array_equal(cache, expect)
    # with the norm on, the RMS-1 row is unchanged and the 2.0 row becomes 1.0 (= H1)
    cache = poison.copy()
    oracle.qnorm_rope_kv_insert("fp8", None, kv, w1, pos, table, slots, cache, 1, 4, 0.0)
    h1 = next(c for c in CASES["kv_cases"] if c["name"] == "H1_constant_row")
    assert np.array_equal(cache[576 * 3:576 * 4], _expand_bytes(h3["fp8_data"], 576))
    assert np.array_equal(cache[576:1152], _expand_bytes(h1["fp8_data"], 576))


# ---------------------------------------------------------------- reading the cache back

def test_e4m3_decode_matches_torch_for_every_code():
    import torch
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_value(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


@pytest.mark.parametrize("case", CASES["gather_cases"], ids=lambda c: c["name"])
def test_golden_gather_rows(case):
    src = next(c for c in CASES["kv_cases"] if c["name"] == case["of"])
    cache = np.zeros(584, np.uint8)
    cache[:576] = _expand_bytes(src["fp8_data"], 576)
    cache[576:584] = _expand_bytes(src["fp8_scale"], 8)
    out, err = oracle.dequant_gather(cache, 1, 1, np.array([0, -1, 0], np.int64))
    assert err == 0
    assert np.array_equal(out[0], _expand_bf16_row(case["row"]))
    assert np.array_equal(out[2], out[0]) and np.all(out[1] == 0)


def test_gather_round_trip_bound():
    """gather(insert(x)) is within half an E4M3 step (times the block scale) of the
    exact v on the quantised dims, and equals bf16(v) on the rope dims."""
    from synth import configs
    wl = configs.generic(300, 1, seed=61, tail_frac=0.02, tail_mult=100.0)
    kv = configs.kv_bits(wl).reshape(wl.T, 512)
    w = configs.weight_bits(wl)
    cs = configs.cos_sin(wl)
    pos = wl.positions()
    slots = synth.permutation(wl.num_slots, 5, 5)[: wl.T]
    cache = np.zeros(wl.num_slots * 584, np.uint8)
    assert oracle.qnorm_rope_kv_insert("fp8", None, kv, w, pos, cs, slots, cache, wl.num_blocks,
                                       wl.block_size, wl.eps) == 0
    out, err = oracle.dequant_gather(cache, wl.num_blocks, wl.block_size, slots)
    assert err == 0
    got = oracle.bf16_value(out)
    for t in range(wl.T):
        v = oracle.kv_values(kv[t], w, cs[pos[t]], wl.eps)
        scale = cache.reshape(wl.num_blocks, -1)[slots[t] // 64, 64 * 576 + 8 * (slots[t] % 64):][:7]
        for b in range(7):
            s = 2.0 ** (int(scale[b]) - 127)
            a = np.abs(v[64 * b:64 * b + 64]) / s
            e = np.floor(np.log2(np.maximum(a, 2.0**-6)))
            half_step = 2.0 ** (e - 3) / 2 * s
            assert np.all(np.abs(got[t, 64 * b:64 * b + 64] - v[64 * b:64 * b + 64])
                          <= half_step * (1 + 1e-12))
        assert np.array_equal(out[t, 448:], oracle.bf16_rne(v[448:]))


def test_gather_skips_and_flags():
    cache = synth.poison_bytes(2 * 4 * 584, seed=8)
    out, err = oracle.dequant_gather(cache, 2, 4, np.array([-1, 8, 100, -7], np.int64))
    assert err == oracle.ERR_SLOT_RANGE and np.all(out == 0)
    out, err = oracle.dequant_gather(cache, 2, 4, np.array([-1, 3], np.int64))
    assert err == 0 and np.all(out[0] == 0)
