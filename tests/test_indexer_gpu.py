"""Indexer-K quant-insert and gather on the GPU against the oracle, bit for bit.

The scale is decided on exact bf16 values and the codes are an exact
power-of-two scaling followed by one E4M3 rounding, so every cache byte (codes,
scales and the untouched poison), every gathered byte and the error word must
be identical on both sides.
"""
import numpy as np
import pytest

import oracle
import synth
from synth import configs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import kv_norm_rope_gb300 as k  # noqa: E402

DEV = torch.device("cuda:0")
SLOT = 132


def _insert_gpu(kbits, slots, nb, bs, poison_seed=11, cache_offset=0):
    """Run the GPU insert into a poisoned cache; cache_offset shifts the cache by
    that many bytes inside its allocation (4: the 4-byte store path)."""
    n = nb * bs * SLOT
    poison = synth.poison_bytes(n, poison_seed)
    buf = torch.zeros(n + 16, dtype=torch.uint8, device=DEV)
    cache = buf[cache_offset:cache_offset + n]
    cache.copy_(torch.from_numpy(poison))
    kt = torch.from_numpy(np.ascontiguousarray(kbits).view(np.int16)).to(DEV)
    st = torch.from_numpy(np.ascontiguousarray(slots, np.int64)).to(DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    k.indexer_k_quant_insert(kt, st, cache, nb, bs, device_error=err)
    torch.cuda.synchronize()
    return poison, cache.cpu().numpy(), int(err.item())


def _gather_gpu(cache, nb, bs, slots, cache_offset=0):
    n = cache.size
    buf = torch.zeros(n + 16, dtype=torch.uint8, device=DEV)
    c = buf[cache_offset:cache_offset + n]
    c.copy_(torch.from_numpy(cache))
    s = torch.from_numpy(np.ascontiguousarray(slots, np.int64)).to(DEV)
    k_out = torch.full((slots.size, 128), 0xA5, dtype=torch.uint8, device=DEV)
    scale = torch.full((slots.size,), 7.0, dtype=torch.float32, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    k.indexer_k_gather(c, nb, bs, s, k_out, scale, device_error=err)
    torch.cuda.synchronize()
    return k_out.cpu().numpy(), scale.cpu().numpy(), int(err.item())


def _check(kbits, slots, nb, bs, cache_offset=0):
    poison, got, err = _insert_gpu(kbits, slots, nb, bs, cache_offset=cache_offset)
    ref = poison.copy()
    ref_err = oracle.indexer_k_quant_insert(kbits, slots, ref, nb, bs)
    assert err == ref_err
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"{bad.size} cache bytes differ, first at {bad[:8]}"
    return got


def _case(T, bs, seed, skip=0.1, extra_blocks=1, tail=0.0, mult=1.0, oob=False):
    nb = -(-T // bs) + extra_blocks
    kbits = synth.normal_bf16(T * 128, seed, synth.TID_IDX_K, tail_frac=tail, tail_mult=mult,
                              tail_id=synth.TID_IDX_K_TAIL).reshape(T, 128)
    slots = synth.permutation(nb * bs, seed, synth.TID_SLOT)[:T].copy()
    n_skip = int(round(skip * T))
    if n_skip:
        slots[synth.permutation(T, seed, synth.TID_SKIP)[:n_skip]] = -1
    if oob and T > 2:
        slots[T // 2] = nb * bs + 3
    return kbits, slots, nb


@pytest.mark.parametrize("T", [1, 2, 7, 17, 511, 1000, 4097])
@pytest.mark.parametrize("bs", [64, 16, 3, 2, 1])
def test_insert_shapes(T, bs):
    kbits, slots, nb = _case(T, bs, seed=T * 7 + bs, oob=(T % 2 == 1))
    _check(kbits, slots, nb, bs)


@pytest.mark.parametrize("bs", [64, 2])
def test_insert_four_byte_store_path(bs):
    """A cache that is only 4-byte aligned takes the two-store path."""
    kbits, slots, nb = _case(999, bs, seed=bs + 40, oob=True)
    _check(kbits, slots, nb, bs, cache_offset=4)


@pytest.mark.parametrize("tail,mult", [(0.01, 100.0), (0.3, 1e4), (0.05, 1e-30)])
def test_insert_heavy_tails_and_tiny_rows(tail, mult):
    kbits, slots, nb = _case(3000, 64, seed=int(tail * 1000), skip=0.0, tail=tail, mult=mult)
    _check(kbits, slots, nb, 64)


def test_insert_special_rows():
    def bits(v):
        return (np.array(v, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    rows = [np.full(128, bits(1.0), np.uint16), np.full(128, 0x8000, np.uint16),
            np.zeros(128, np.uint16), np.full(128, bits(2.0 ** -130), np.uint16),
            np.full(128, 0x7F7F, np.uint16), np.full(128, 0xFF7F, np.uint16),
            np.full(128, 0x0001, np.uint16)]
    r = np.full(128, bits(1.0), np.uint16)
    r[5] = bits(1.75)
    rows.append(r)
    r = r.copy()
    r[5] = bits(-1.7578125)
    rows.append(r)
    r = np.full(128, bits(3.0), np.uint16)
    r[::3] = 0x8001                                  # mixed tiny negatives
    rows.append(r)
    kbits = np.stack(rows)
    slots = np.arange(kbits.shape[0], dtype=np.int64)[::-1].copy()
    _check(kbits, slots, 1, 64)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["prefill", "stress"])
def test_insert_full_size(name):
    wl = configs.WORKLOADS[name]
    kbits = configs.indexer_k_bits(wl).reshape(wl.T, 128)
    _check(kbits, wl.slot_mapping(), wl.num_blocks, wl.block_size)


@pytest.mark.parametrize("bs,offset", [(64, 0), (3, 0), (64, 4)])
def test_gather_round_trip(bs, offset):
    kbits, slots, nb = _case(2000, bs, seed=bs + 3, tail=0.01, mult=100.0)
    cache = _check(kbits, slots, nb, bs)
    order = np.concatenate([slots[::-1], [-1, nb * bs, nb * bs + 100, 0]]).astype(np.int64)
    got_k, got_s, err = _gather_gpu(cache, nb, bs, order, cache_offset=offset)
    ref_k, ref_s, ref_err = oracle.indexer_k_gather(cache, nb, bs, order)
    assert err == ref_err == k.DEVERR_SLOT_RANGE
    assert np.array_equal(got_k, ref_k)
    assert np.array_equal(got_s.view(np.uint32), ref_s.view(np.uint32))


def test_gather_of_poisoned_cache():
    nb, bs = 40, 64
    cache = synth.poison_bytes(nb * bs * SLOT, 99)
    slots = synth.permutation(nb * bs, 9, synth.TID_SLOT).astype(np.int64)
    got_k, got_s, err = _gather_gpu(cache, nb, bs, slots)
    ref_k, ref_s, ref_err = oracle.indexer_k_gather(cache, nb, bs, slots)
    assert err == ref_err == 0
    assert np.array_equal(got_k, ref_k)
    assert np.array_equal(got_s.view(np.uint32), ref_s.view(np.uint32))


def test_empty_calls_launch_nothing():
    cache = torch.zeros(SLOT * 64, dtype=torch.uint8, device=DEV)
    empty_k = torch.zeros((0, 128), dtype=torch.int16, device=DEV)
    empty_s = torch.zeros(0, dtype=torch.int64, device=DEV)
    k.indexer_k_quant_insert(empty_k, empty_s, cache, 1, 64)
    k.indexer_k_gather(cache, 1, 64, empty_s, torch.zeros((0, 128), dtype=torch.uint8, device=DEV),
                       torch.zeros(0, dtype=torch.float32, device=DEV))
    torch.cuda.synchronize()
    assert int(cache.sum().item()) == 0


@pytest.mark.parametrize("std", [1e-39, 1e-20, 1e30, 1e37])
def test_insert_extreme_scales(std):
    """Rows of bf16 subnormals (the exponent clamps at -127) up to rows near the
    top of the bf16 range."""
    T, bs = 600, 64
    nb = -(-T // bs)
    kbits = synth.normal_bf16(T * 128, 5, synth.TID_IDX_K, std=std).reshape(T, 128)
    _check(kbits, np.arange(T, dtype=np.int64), nb, bs)
