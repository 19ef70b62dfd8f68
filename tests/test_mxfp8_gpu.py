"""Residual add + Gemma RMSNorm + MXFP8 on the GPU against the oracle.

Bar: residual_out bit-exact; scale bytes (and the zeroed padding rows) bit-exact;
E4M3 codes bit-exact except at most 1e-4 of them, each one step away (the kernel
forms the bf16-rounded normed value in fp32, the oracle in fp64; they can land on
different sides of a bf16 midpoint)."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import kv_norm_rope_gb300 as k  # noqa: E402

DEV = torch.device("cuda:0")


def _inputs(m, n, seed, tail=0.0):
    x = synth.normal_bf16(m * n, seed, 1, tail_frac=tail, tail_mult=100.0, tail_id=9).reshape(m, n)
    r = synth.normal_bf16(m * n, seed, 2, std=2.0).reshape(m, n)
    g = synth.normal_bf16(n, seed, 3, std=0.2)
    return x, r, g


def _gpu(x, r, g, eps, in_place=False):
    m, n = x.shape
    t = lambda a: torch.from_numpy(a.view(np.int16)).to(DEV)
    tx, tr, tg = t(x), t(r), t(g)
    out = tr if in_place else torch.full((m, n), 0x3333, dtype=torch.int16, device=DEV)
    codes = torch.full((m, n), 0xAB, dtype=torch.uint8, device=DEV)
    scales = torch.full((k.mxfp8_scale_bytes(m, n),), 0xCD, dtype=torch.uint8, device=DEV)
    k.add_gemma_rmsnorm_mxfp8(tx, tr, tg, eps, out, codes, scales)
    torch.cuda.synchronize()
    return (out.cpu().numpy().view(np.uint16), codes.cpu().numpy(), scales.cpu().numpy())


def _ord(c):
    c = c.astype(np.int64)
    return np.where(c & 0x80, -(c & 0x7F), c & 0x7F)


def _check(x, r, g, eps=1e-6, in_place=False):
    res, codes, scales = _gpu(x, r, g, eps, in_place)
    ref_res, ref_codes, ref_scales = oracle.gemma_rmsnorm_mxfp8(x, r, g, eps)
    assert np.array_equal(res, ref_res)
    assert np.array_equal(scales, ref_scales)
    d = np.abs(_ord(codes) - _ord(ref_codes))
    assert d.max() <= 1
    assert (d != 0).sum() <= max(1, 1e-4 * d.size), (d != 0).sum()
    return (d != 0).sum()


@pytest.mark.parametrize("n", [128, 512, 1024, 3072, 7168, 8192, 16384])
@pytest.mark.parametrize("m", [1, 7, 129])
def test_shapes(m, n):
    _check(*_inputs(m, n, seed=m * 7 + n))


def test_many_rows_heavy_tails():
    _check(*_inputs(1000, 2048, seed=5, tail=0.01))


def test_in_place_residual():
    _check(*_inputs(300, 1024, seed=6), in_place=True)


def test_zero_rows_and_eps():
    x = np.zeros((3, 256), np.uint16)
    r = np.zeros((3, 256), np.uint16)
    g = synth.normal_bf16(256, 1, 3)
    _check(x, r, g, eps=1e-6)
    x, r, g = _inputs(5, 256, seed=9)
    _check(x, r, g, eps=0.5)


def test_empty_batch_is_a_no_op():
    z = torch.zeros((0, 256), dtype=torch.int16, device=DEV)
    g = torch.zeros(256, dtype=torch.int16, device=DEV)
    k.add_gemma_rmsnorm_mxfp8(z, z, g, 1e-6, z, torch.zeros(0, dtype=torch.uint8, device=DEV),
                              torch.zeros(0, dtype=torch.uint8, device=DEV))


def test_tiny_rows_with_eps_zero():
    """With eps = 0, rows whose prenorm lies near 2^-70 .. 2^-128 (squares subnormal in
    fp32) normalise like their unscaled selves: the kernel rescales them by 2^64 before
    taking r.  Residual, scales and codes against the oracle."""
    m, n = 8, 1024
    x, r, g = _inputs(m, n, seed=41)
    scales = np.array([1.0, 2.0**-50, 2.0**-64, 2.0**-70, 2.0**-100, 2.0**-115, 2.0**-124,
                       2.0**-128], np.float32)

    def scaled(bits):
        f = synth.bf16_bits_to_f32(bits).reshape(m, n) * scales[:, None]
        return torch.from_numpy(np.ascontiguousarray(f)).to(torch.bfloat16).view(torch.int16) \
            .numpy().view(np.uint16)

    xs, rs = scaled(x), scaled(r)
    assert np.all((xs & 0x7FFF).max(axis=1) > 0)
    _check(xs, rs, g, eps=0.0)
