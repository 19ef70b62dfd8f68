"""Pins of the oracle's residual-add + Gemma RMSNorm + MXFP8 quantiser (CPU only).

The steps follow the vLLM minimax_m3 finalize_allreduce_norm page (the single-GPU
part of _LamportGemmaRMSNormMxfp8Kernel): prenorm = bf16(x + residual); Gemma
scale 1 + w; normed rounded to bf16; UE8M0 of fp32(amax * fp32(1/448)) rounded
up to a power of two; E4M3 of normed * 2^(127 - e); 128x4 swizzled scales with
zeroed padding rows.  Pinned by numpy float32 arithmetic, torch casts, hand
rows, the layout's bijection and the E4M3 rounding bound.
"""
import numpy as np
import pytest
import torch

import oracle
import synth


def _bf16_bits(v):
    return (np.array(v, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _row(n, v):
    return np.full(n, _bf16_bits(v), np.uint16)


def test_ue8m0_rounds_up_to_a_power_of_two():
    rng = np.random.default_rng(3)
    xs = np.concatenate([np.exp(rng.uniform(-100, 87, 20000)).astype(np.float32),
                         np.ldexp(np.float32(1), np.arange(-149, 127)).astype(np.float32),
                         np.array([0.0, -1.0, 3e38, 1e-45], np.float32)])
    for x in xs:
        got = oracle.ue8m0_of_f32(float(x))
        if not x > 0:
            want = 0
        else:
            f, e = np.frexp(np.float64(x))          # x = f * 2^e, f in [0.5, 1)
            ceil_log2 = e - 1 if f == 0.5 else e
            want = int(min(254, max(0, ceil_log2 + 127)))
        assert got == want, (x, got, want)


def test_inverse_scale():
    assert oracle.ue8m0_inverse(0) == 0.0 and oracle.ue8m0_inverse(254) == 0.0
    assert oracle.ue8m0_inverse(127) == 1.0 and oracle.ue8m0_inverse(119) == 256.0
    assert oracle.ue8m0_inverse(253) == 2.0 ** -126


def test_prenorm_add_matches_fp32_add_then_bf16():
    """bf16(x + r) from exact doubles equals torch's fp32 add then bf16 rounding."""
    a = synth.normal_bf16(1 << 20, 5, 1, std=3.0)
    b = synth.normal_bf16(1 << 20, 5, 2, std=0.01, tail_frac=0.3, tail_mult=1000.0, tail_id=9)
    ta = torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).float()
    tb = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).float()
    ref = (ta + tb).bfloat16().view(torch.int16).numpy().view(np.uint16)
    got, _, _ = oracle.gemma_rmsnorm_mxfp8(a.reshape(-1, 1024), b.reshape(-1, 1024),
                                           np.zeros(1024, np.uint16), 1e-6)
    assert np.array_equal(got.ravel(), ref)


def test_swizzled_layout_positions_and_bijection():
    # hand-derived: within a 512-byte tile, row r, block c sits at 16*(r%32) + 4*((r%128)//32) + c%4
    for (r, c, pc, off) in [(0, 0, 4, 0), (0, 1, 4, 1), (0, 3, 4, 3), (32, 0, 4, 4), (1, 0, 4, 16),
                            (127, 3, 4, 511), (0, 4, 8, 512), (128, 0, 8, 1024), (129, 5, 8, 1024 + 512 + 16 + 1)]:
        assert oracle.swizzled_scale_offset(r, c, pc) == off
    for m, n in [(1, 128), (129, 512), (300, 768)]:
        rows, cols = -(-m // 128) * 128, -(-(n // 32) // 4) * 4
        assert oracle.mxfp8_scale_bytes(m, n) == rows * cols
        offs = sorted(oracle.swizzled_scale_offset(r, c, cols) for r in range(rows) for c in range(cols))
        assert offs == list(range(rows * cols))


def test_hand_rows():
    n = 256
    zero = _row(n, 0.0)
    # x = 1, residual 0, gamma 0: prenorm 1, r = 1, normed 1; fp32(1 * fl(1/448)) has
    # ceil(log2) = -8 -> e = 119; code 1 * 2^8 = 256 = 0x78
    res, codes, scales = oracle.gemma_rmsnorm_mxfp8(_row(n, 1.0)[None], zero[None], zero, 0.0)
    assert np.all(res == 0x3F80) and np.all(codes == 0x78)
    assert np.all(scales[[oracle.swizzled_scale_offset(0, c, 8) for c in range(8)]] == 119)
    assert scales.size == 128 * 8 and np.count_nonzero(scales) == 8
    # x = 1, residual 1 (prenorm 2 = 0x4000), gamma 1 (scale 2): r = 0.5, normed = 2;
    # e = ceil(log2(2/448)) + 127 = 120; code 2 * 2^7 = 256 = 0x78
    res, codes, scales = oracle.gemma_rmsnorm_mxfp8(_row(n, 1.0)[None], _row(n, 1.0)[None],
                                                    _row(n, 1.0), 0.0)
    assert np.all(res == 0x4000) and np.all(codes == 0x78)
    assert scales[oracle.swizzled_scale_offset(0, 3, 8)] == 120
    # eps inside the root: x = 1 everywhere, eps = 3 -> r = 0.5, normed 0.5; e = 118 (2^-9 >= 0.5/448)
    _, codes, scales = oracle.gemma_rmsnorm_mxfp8(_row(n, 1.0)[None], zero[None], zero, 3.0)
    assert np.all(codes == 0x78) and scales[0] == 118
    # all-zero row: amax 0 -> e = 0 and inverse 0; codes keep the sign of zero
    _, codes, scales = oracle.gemma_rmsnorm_mxfp8(_row(n, -0.0)[None], _row(n, -0.0)[None], zero, 1e-6)
    assert np.all(codes == 0x80) and np.all(scales == 0)


def test_amax_on_448_times_power_of_two_follows_fp32():
    """normed amax = 1.75 = 448 * 2^-8: the page multiplies by fp32(1/448), so the
    exponent is whatever that fp32 product rounds to -- checked with numpy float32."""
    n = 128
    g = _row(n, 0.0)
    g[5] = _bf16_bits(0.75)                 # normed = prenorm * r * (1 + g) = 1 + g with x const
    _, codes, scales = oracle.gemma_rmsnorm_mxfp8(_row(n, 4.0)[None], _row(n, 0.0)[None], g, 0.0)
    prod = np.float32(1.75) * np.float32(1.0 / 448.0)
    f, e = np.frexp(np.float64(prod))
    want = (e - 1 if f == 0.5 else e) + 127
    assert scales[oracle.swizzled_scale_offset(0, 0, 4)] == want
    inv = 2.0 ** (127 - want)
    assert codes[0, 5] == oracle.e4m3_rne(np.array([1.75 * inv]))[0]


def _e4m3_decode(c):
    c = c.astype(np.int64)
    e = (c >> 3) & 0xF
    m = c & 7
    mag = np.where(e == 0, m * 2.0**-9, (8 + m) * np.ldexp(1.0, e - 10))
    return np.where(c & 0x80, -mag, mag)


@pytest.mark.parametrize("m,n", [(3, 128), (130, 512), (17, 3072)])
def test_quantisation_bound_and_padding(m, n):
    x = synth.normal_bf16(m * n, 9, 1, tail_frac=0.01, tail_mult=50.0, tail_id=9).reshape(m, n)
    r = synth.normal_bf16(m * n, 9, 2).reshape(m, n)
    g = synth.normal_bf16(n, 9, 3, std=0.3)
    res, codes, scales = oracle.gemma_rmsnorm_mxfp8(x, r, g, 1e-6)
    cols = n // 32
    pre = oracle.bf16_value(res)
    rr = 1.0 / np.sqrt(np.mean(pre * pre, axis=1) + np.float64(np.float32(1e-6)))
    normed = oracle.bf16_value(oracle.bf16_rne(pre * rr[:, None] * (1.0 + oracle.bf16_value(g))[None]))
    for row in range(m):
        for c in range(cols):
            e = int(scales[oracle.swizzled_scale_offset(row, c, cols)])
            blk = normed[row, 32 * c:32 * c + 32]
            s = 2.0 ** (e - 127)
            a = np.abs(blk) / s
            assert np.max(a) <= 448.0
            step = 2.0 ** (np.floor(np.log2(np.maximum(a, 2.0**-6))) - 3) * s
            deq = _e4m3_decode(codes[row, 32 * c:32 * c + 32]) * s
            assert np.all(np.abs(deq - blk) <= step / 2 * (1 + 1e-12))
    padded = np.ones(scales.size, bool)
    padded[[oracle.swizzled_scale_offset(row, c, cols) for row in range(m) for c in range(cols)]] = False
    assert np.all(scales[padded] == 0)


def test_normed_is_rounded_to_bf16_before_quantising():
    """x = 4 everywhere, eps 0: r = 1/4 and normed = 1 + g exactly.  With
    g = 2^-4 * (1 + 2^-7), 1 + g = 1.06298828125 rounds to bf16 1.0625, which the
    scale 2^8 (amax ~1.06 -> e = 119) takes to 272, an E4M3 midpoint: ties to even
    give 256 = 0x78.  Quantising the unrounded value would give 288 = 0x79."""
    n = 128
    g = _row(n, 0.0)
    g[7] = _bf16_bits(0.0625 * (1 + 2.0**-7))
    _, codes, scales = oracle.gemma_rmsnorm_mxfp8(_row(n, 4.0)[None], _row(n, 0.0)[None], g, 0.0)
    assert scales[0] == 119
    assert codes[0, 7] == 0x78 and codes[0, 6] == 0x78


def test_fp32_product_with_inverse_448_matches_exact_quotient_on_bf16():
    """For every positive finite bf16 amax, the exponent from the page's fp32
    product amax * fp32(1/448) equals the exponent of the exact quotient amax / 448:
    a bf16 value is never within fp32 error of 448 * 2^k unless it equals it."""
    bits = np.arange(1, 0x7F80, dtype=np.uint32).astype(np.uint16)
    a = oracle.bf16_value(bits)
    prod = (a.astype(np.float32) * np.float32(1.0 / 448.0)).astype(np.float32)
    exact = a / 448.0
    for p, q in zip(prod, exact):
        f, e = np.frexp(q)
        want = int(min(254, max(0, (e - 1 if f == 0.5 else e) + 127)))
        assert oracle.ue8m0_of_f32(float(p)) == want
