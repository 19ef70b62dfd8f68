"""Pins of the oracle's encoders against library casts and exact arithmetic (CPU only).

The bf16 and E4M3 encoders are compared bit for bit with torch's CPU casts
(float32 -> bfloat16 and float32 -> float8_e4m3fn, both round-to-nearest-even):
all 65536 bf16 patterns at 21 scalings, random float32 inputs with half of the
E4M3 cases in the subnormal range below 2^-6, and every midpoint.  The T-Head
section of FlagGems-vllm PR #684 names the two classic encoder faults this
catches: flushing subnormals, and treating exponent 15 / mantissa 0 (= 256) as
an overflow.  Doubles that float32 cannot hold are pinned by exact arithmetic:
a value just above (below) a midpoint must round up (down) whatever the parity.
"""
import math

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


def _all_bf16_values():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    return bits, vals


def test_bf16_value_exact_for_all_patterns():
    bits, ref = _all_bf16_values()
    got = oracle.bf16_value(bits)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


def test_bf16_rne_fixed_points():
    bits, vals = _all_bf16_values()
    ok = ~np.isnan(vals)
    assert np.array_equal(oracle.bf16_rne(vals[ok]), bits[ok])


def test_bf16_rne_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(1234)
    raw = rng.integers(0, 2**32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    x32 = raw.view(np.float32)
    x32 = x32[np.isfinite(x32)]
    # every bf16 midpoint (9 significant bits: exact in float32), both signs
    bits, vals = _all_bf16_values()
    fin = np.isfinite(vals) & (np.abs(vals) < 3.3e38)
    lo = vals[fin]
    up = torch.from_numpy((bits[fin].astype(np.int32) + 1).astype(np.uint16).view(np.int16)) \
        .view(torch.bfloat16).to(torch.float64).numpy()
    same_sign = np.isfinite(up) & (np.sign(up) == np.sign(lo))
    mids = ((lo + up) / 2)[same_sign].astype(np.float32)
    xs = np.concatenate([x32, mids])
    ref = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_rne(xs.astype(np.float64))
    assert np.array_equal(got, ref)


def test_bf16_rne_rounds_doubles_once():
    """1 + 2^-8 is the midpoint of 1.0 and 1 + 2^-7: a hair above must go up,
    a hair below down, exactly at it to the even neighbour (1.0)."""
    one = 1.0
    cases = [
        (one + 2**-8 + 2**-40, 0x3F81),
        (one + 2**-8 - 2**-40, 0x3F80),
        (one + 2**-8, 0x3F80),
        (one + 3 * 2**-8, 0x3F82),          # midpoint of 0x3F81 and 0x3F82: even is 0x3F82
        (-(one + 2**-8 + 2**-45), 0xBF81),
        (2.0**-133, 0x0001),                 # smallest subnormal
        (2.0**-134, 0x0000),                 # half of it: tie to even zero
        (2.0**-134 * (1 + 2**-30), 0x0001),
        ((2 - 2**-7) * 2.0**127, 0x7F7F),    # largest finite bf16
        ((2 - 2**-8) * 2.0**127, 0x7F80),    # the overflow midpoint rounds to inf
        ((2 - 2**-8 - 2**-30) * 2.0**127, 0x7F7F),
    ]
    xs = np.array([c[0] for c in cases])
    got = oracle.bf16_rne(xs)
    assert [int(g) for g in got] == [c[1] for c in cases]


def _e4m3_table():
    codes = np.arange(256, dtype=np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    return codes, vals


def test_e4m3_round_trip_every_code():
    codes, vals = _e4m3_table()
    ok = ~np.isnan(vals)
    assert ok.sum() == 254
    assert np.array_equal(oracle.e4m3_rne(vals[ok]), codes[ok])
    assert vals[0x78] == 256.0 and vals[0x7E] == 448.0 and vals[0x01] == 2.0**-9


def test_e4m3_matches_torch_scaled_bf16_grid():
    _, vals = _all_bf16_values()
    vals = vals[np.isfinite(vals)]
    xs = np.concatenate([vals * 2.0**k for k in range(-10, 11)])
    xs = xs[np.abs(xs) <= 464.0].astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_rne(xs.astype(np.float64))
    assert np.array_equal(got, ref)


def test_e4m3_matches_torch_random_half_subnormal():
    rng = np.random.default_rng(99)
    n = 2_000_000
    sub = rng.uniform(0, 2.0**-6, n // 2)
    norm = np.exp(rng.uniform(math.log(2.0**-6), math.log(448.0), n - n // 2))
    xs = np.concatenate([sub, norm]) * rng.choice([-1.0, 1.0], n)
    xs = xs.astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_rne(xs.astype(np.float64))
    assert np.array_equal(got, ref)
    assert (np.abs(xs) < 2.0**-6).mean() >= 0.5


def test_e4m3_midpoints_and_doubles():
    codes, vals = _e4m3_table()
    pos = np.sort(vals[(vals >= 0) & ~np.signbit(vals) & np.isfinite(vals)])
    mids = (pos[:-1] + pos[1:]) / 2
    # ties go to the even code of the two neighbours
    lo_codes = np.array([int(np.where(vals[:128] == v)[0][0]) for v in pos[:-1]])
    hi_codes = lo_codes + 1
    even = np.where(lo_codes % 2 == 0, lo_codes, hi_codes)
    assert np.array_equal(oracle.e4m3_rne(mids), even.astype(np.uint8))
    # a hair above / below a midpoint decides it regardless of parity
    eps = mids * 2.0**-40
    assert np.array_equal(oracle.e4m3_rne(mids + eps), hi_codes.astype(np.uint8))
    assert np.array_equal(oracle.e4m3_rne(mids - eps), lo_codes.astype(np.uint8))


def test_e4m3_saturation_and_specials():
    xs = np.array([448.0 * (1 + 2.0**-20), 1000.0, np.inf, -np.inf, -448.5, np.nan, -0.0, -(2.0**-11)])
    got = oracle.e4m3_rne(xs)
    assert [int(g) for g in got] == [0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F, 0x80, 0x80]


def test_ue8m0_exponent_boundaries():
    ks = np.arange(-120, 121)
    at = 448.0 * np.ldexp(1.0, ks)
    assert np.array_equal(oracle.ue8m0_exponent(at), ks)
    assert np.array_equal(oracle.ue8m0_exponent(np.nextafter(at, np.inf)), ks + 1)
    assert np.array_equal(oracle.ue8m0_exponent(np.nextafter(at, 0)), ks)
    special = oracle.ue8m0_exponent(np.array([0.0, 1e-300, 448.0 * 2.0**-127, 448.0 * 2.0**-128, 1e300]))
    assert list(special) == [-127, -127, -127, -127, 127]


def test_ue8m0_exponent_vs_high_precision_log():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.prec = 200
    rng = np.random.default_rng(7)
    amax = np.exp(rng.uniform(-60, 60, 20000))
    got = oracle.ue8m0_exponent(amax)
    for a, s in zip(amax, got):
        l2 = mpmath.log(mpmath.mpf(float(a)) / 448, 2)
        frac = l2 - mpmath.floor(l2)
        if frac < 1e-12 or frac > 1 - 1e-12:
            continue
        assert s == int(mpmath.ceil(l2))
