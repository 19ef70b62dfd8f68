"""Pins of the oracle's indexer-K quant-insert and gather (CPU only).

The indexer consumes K as contiguous [N, 128] E4M3 rows with one non-negative
fp32 scale per row (rocm-aiter PR #1, "Motivation"); the norm-rope-store kernel
keeps a separate indexer path (SGLang PR #33358, "Modifications").  The oracle
takes one power-of-two scale per 128-element row, 2^s with s the smallest
integer such that amax <= 448 * 2^s (clamped to [-127, 127]), and the paged
layout: per block, bs rows of 128 codes, then bs little-endian fp32 scales.

Pinned here by numpy's frexp (the scale), torch's float8_e4m3fn cast (the
codes), hand rows, the half-step error bound, and byte-level layout checks
against a poisoned cache.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from synth import configs

DIM = 128
SLOT = 132


def _bf16_bits(v):
    return (np.array(v, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _poisoned(nb, bs, seed=5):
    return synth.poison_bytes(nb * bs * SLOT, seed)


def _scale_at(cache, bs, slot):
    blk, off = divmod(slot, bs)
    base = blk * bs * SLOT + bs * DIM + off * 4
    return cache[base:base + 4].view(np.float32)[0]


def _codes_at(cache, bs, slot):
    blk, off = divmod(slot, bs)
    base = blk * bs * SLOT + off * DIM
    return cache[base:base + DIM]


def _want_scale_exponent(amax):
    """ceil(log2(amax / 448)) clamped to [-127, 127], -127 for amax = 0."""
    if amax == 0:
        return -127
    f, e = np.frexp(np.float64(amax) / 448.0)        # amax/448 = f * 2^e, f in [0.5, 1)
    ceil_log2 = e - 1 if f == 0.5 else e
    return int(min(127, max(-127, ceil_log2)))


def _insert_one(row_bits, bs=4, slot=1):
    cache = _poisoned(1, bs)
    err = oracle.indexer_k_quant_insert(row_bits[None], np.array([slot]), cache, 1, bs)
    assert err == 0
    return _codes_at(cache, bs, slot), _scale_at(cache, bs, slot)


def test_hand_rows():
    # all 1.0: 448 * 2^-9 = 0.875 < 1 <= 1.75 = 448 * 2^-8 -> scale 2^-8; code of 256 is 0x78
    codes, scale = _insert_one(np.full(DIM, _bf16_bits(1.0), np.uint16))
    assert scale == 2.0 ** -8 and np.all(codes == 0x78)
    # amax exactly 1.75 = 448 * 2^-8 keeps scale 2^-8 and codes 448 -> 0x7E
    row = np.full(DIM, _bf16_bits(1.0), np.uint16)
    row[17] = _bf16_bits(-1.75)
    codes, scale = _insert_one(row)
    assert scale == 2.0 ** -8 and codes[17] == 0xFE and codes[0] == 0x78
    # next bf16 above 1.75 (1.7578125) needs 2^-7; 1.0 * 2^7 = 128 -> 0x70
    row[17] = _bf16_bits(1.7578125)
    codes, scale = _insert_one(row)
    assert scale == 2.0 ** -7 and codes[0] == 0x70
    # 1.7578125 * 128 = 225 lies between E4M3 values 224 and 240 -> 224 = 0x76
    assert codes[17] == 0x76
    # all -0.0: amax 0 -> s = -127, scale 2^-127 (an fp32 subnormal), codes negative zero
    codes, scale = _insert_one(np.full(DIM, 0x8000, np.uint16))
    assert scale == np.float32(2.0 ** -127) and np.all(codes == 0x80)
    assert np.array(scale, np.float32).view(np.uint32) == 0x00400000   # 2^22 * 2^-149
    # amax 2^-130 (a bf16 subnormal): s would be -139, clamped to -127;
    # 2^-130 * 2^127 = 2^-3 -> code 0x20 (exponent field 4, mantissa 0)
    codes, scale = _insert_one(np.full(DIM, _bf16_bits(2.0 ** -130), np.uint16))
    assert scale == np.float32(2.0 ** -127) and np.all(codes == 0x20)
    # the largest bf16, (2 - 2^-7) * 2^127: 448 * 2^119 < it <= 448 * 2^120 -> s = 120
    big = (2.0 - 2.0 ** -7) * 2.0 ** 127
    codes, scale = _insert_one(np.full(DIM, _bf16_bits(big), np.uint16))
    assert scale == np.float32(2.0 ** 120)
    assert np.all(codes == oracle.e4m3_rne(np.array([big / 2.0 ** 120]))[0])


@pytest.mark.parametrize("seed,tail", [(1, 0.0), (2, 0.02), (3, 0.3)])
def test_scale_and_codes_against_numpy_and_torch(seed, tail):
    T, bs = 300, 16
    nb = -(-T // bs) + 1
    k = synth.normal_bf16(T * DIM, seed, synth.TID_IDX_K, tail_frac=tail, tail_mult=1e4,
                          tail_id=synth.TID_IDX_K_TAIL).reshape(T, DIM)
    slots = synth.permutation(nb * bs, seed, synth.TID_SLOT)[:T]
    cache = _poisoned(nb, bs)
    assert oracle.indexer_k_quant_insert(k, slots, cache, nb, bs) == 0
    kf = torch.from_numpy(k.view(np.int16)).view(torch.bfloat16).float()
    for t in range(T):
        s = _want_scale_exponent(float(kf[t].abs().max()))
        scale = _scale_at(cache, bs, int(slots[t]))
        assert scale == np.float32(2.0 ** s), (t, scale, s)
        # x * 2^-s is exact in float32 here (no bf16 row of these draws gets near
        # the fp32 subnormal range), so torch's RNE cast is an independent encoder
        scaled = kf[t] * float(2.0 ** -s)
        want = scaled.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(_codes_at(cache, bs, int(slots[t])), want), t


def _e4m3_decode(c):
    c = c.astype(np.int64)
    e = (c >> 3) & 0xF
    m = c & 7
    mag = np.where(e == 0, m * 2.0**-9, (8 + m) * np.ldexp(1.0, e - 10))
    return np.where(c & 0x80, -mag, mag)


def test_half_step_bound_on_heavy_tails():
    w = configs.STRESS
    T = 512
    k = configs.indexer_k_bits(w, 0, T).reshape(T, DIM)
    slots = np.arange(T, dtype=np.int64)
    nb, bs = T // 64, 64
    cache = _poisoned(nb, bs)
    assert oracle.indexer_k_quant_insert(k, slots, cache, nb, bs) == 0
    x = oracle.bf16_value(k)
    for t in range(T):
        scale = float(_scale_at(cache, bs, t))
        a = np.abs(x[t]) / scale
        assert a.max() <= 448.0 and (a.max() > 224.0 or a.max() == 0)
        step = 2.0 ** (np.floor(np.log2(np.maximum(a, 2.0**-6))) - 3) * scale
        deq = _e4m3_decode(_codes_at(cache, bs, t)) * scale
        assert np.all(np.abs(deq - x[t]) <= step / 2)


def test_layout_untouched_bytes_and_errors():
    nb, bs = 3, 5                                   # odd block size: rows straddle nothing
    T = 9
    k = synth.normal_bf16(T * DIM, 7, synth.TID_IDX_K).reshape(T, DIM)
    slots = np.array([0, 14, -1, 6, 15, 3, -7, 9, 100], np.int64)   # 15, 100 out of range
    cache = _poisoned(nb, bs)
    before = cache.copy()
    err = oracle.indexer_k_quant_insert(k, slots, cache, nb, bs)
    assert err == oracle.ERR_SLOT_RANGE
    written = np.zeros(cache.size, bool)
    for s in slots:
        if 0 <= s < nb * bs:
            blk, off = divmod(int(s), bs)
            b0 = blk * bs * SLOT
            written[b0 + off * DIM:b0 + off * DIM + DIM] = True
            written[b0 + bs * DIM + off * 4:b0 + bs * DIM + off * 4 + 4] = True
    assert written.sum() == 5 * SLOT                # slots 0, 14, 6, 3, 9
    assert np.array_equal(cache[~written], before[~written])
    # each valid row: its own codes and scale, independent of where it sits
    for t, s in enumerate(slots):
        if 0 <= s < nb * bs:
            codes, scale = _insert_one(k[t])
            assert np.array_equal(_codes_at(cache, bs, int(s)), codes)
            assert _scale_at(cache, bs, int(s)) == scale


def test_gather_round_trip():
    nb, bs = 4, 8
    T = 20
    k = synth.normal_bf16(T * DIM, 8, synth.TID_IDX_K, tail_frac=0.05, tail_mult=300.0,
                          tail_id=synth.TID_IDX_K_TAIL).reshape(T, DIM)
    slots = synth.permutation(nb * bs, 8, synth.TID_SLOT)[:T]
    cache = _poisoned(nb, bs)
    assert oracle.indexer_k_quant_insert(k, slots, cache, nb, bs) == 0
    order = np.array(list(slots[::-1]) + [-1, nb * bs, 0], np.int64)
    codes, scales, err = oracle.indexer_k_gather(cache, nb, bs, order)
    assert err == oracle.ERR_SLOT_RANGE
    for n, s in enumerate(order):
        if 0 <= s < nb * bs:
            assert np.array_equal(codes[n], _codes_at(cache, bs, int(s)))
            assert scales[n] == _scale_at(cache, bs, int(s))
        else:
            assert not codes[n].any() and scales[n] == 0.0
    # the gathered rows dequantise to within half a step of the inputs
    x = oracle.bf16_value(k[::-1])
    deq = _e4m3_decode(codes[:T]) * scales[:T, None].astype(np.float64)
    assert np.all(np.abs(deq - x) <= np.abs(x) * 2.0**-4 + scales[:T, None] * 2.0**-10)
