"""C-ABI tests that need no GPU: the library loads, exports every function the header
declares, rejects bad arguments on the host before touching CUDA, plans launches as
documented, and has no CPU fallback."""
import ctypes
import math
import os
import re

import pytest

import kv_norm_rope_gb300 as k

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "dsv4kv.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsv4_[a-z0-9_]+)\s*\(", text)))


def test_header_declarations_are_exported():
    names = _declared_functions()
    assert names == sorted(k.EXPORTS)
    lib = k.lib()
    for n in names:
        assert hasattr(lib, n)


def test_status_strings():
    assert k.status_string(k.OK) == "ok"
    assert "align" in k.status_string(k.ERR_ALIGN)
    assert k.status_string(99) == "unknown status"


def test_cache_bytes():
    assert k.fp8_cache_bytes(1024, 64) == 1024 * 64 * 584
    assert k.bf16_cache_bytes(2048, 64) == 2048 * 64 * 1024
    assert k.fp8_cache_bytes(0, 64) == 0


# fake device pointers: never dereferenced, because every call below is rejected
# (or returns early) on the host
A = 1 << 20


def _call(store=0, variant=0, q=A, kv=A, w=A, pos=A, cs=A, max_pos=4096, slot=A, cache=A,
          nb=4, bs=64, T=16, H=8, eps=1e-6, err=None):
    return k.lib().dsv4_qnorm_rope_kv_insert_variant(store, variant, q, kv, w, pos, cs, max_pos,
                                                     slot, cache, nb, bs, T, H, eps, err, None)


@pytest.mark.parametrize("kw,status", [
    (dict(T=-1), k.ERR_SHAPE), (dict(H=0), k.ERR_SHAPE), (dict(nb=0), k.ERR_SHAPE),
    (dict(bs=0), k.ERR_SHAPE), (dict(max_pos=0), k.ERR_SHAPE),
    (dict(T=2**62), k.ERR_SHAPE),
    (dict(eps=-1.0), k.ERR_VALUE), (dict(eps=math.inf), k.ERR_VALUE), (dict(eps=math.nan), k.ERR_VALUE),
    (dict(store=2), k.ERR_VALUE), (dict(variant=7), k.ERR_VALUE),
    (dict(q=None), k.ERR_NULL), (dict(kv=None), k.ERR_NULL), (dict(w=None), k.ERR_NULL),
    (dict(pos=None), k.ERR_NULL), (dict(cs=None), k.ERR_NULL), (dict(slot=None), k.ERR_NULL),
    (dict(cache=None), k.ERR_NULL),
    (dict(q=A + 8), k.ERR_ALIGN), (dict(kv=A + 2), k.ERR_ALIGN), (dict(w=A + 4), k.ERR_ALIGN),
    (dict(cs=A + 8), k.ERR_ALIGN), (dict(pos=A + 4), k.ERR_ALIGN), (dict(slot=A + 1), k.ERR_ALIGN),
    (dict(cache=A + 4), k.ERR_ALIGN), (dict(store=1, cache=A + 8), k.ERR_ALIGN),
    (dict(err=A + 2), k.ERR_ALIGN),
])
def test_host_validation(kw, status):
    assert _call(**kw) == status


def test_fp8_cache_needs_only_8_byte_alignment():
    # 8-byte aligned FP8 cache passes validation; with no T it returns before CUDA
    assert _call(cache=A + 8, T=0) == k.OK


def test_zero_tokens_is_a_no_op():
    assert _call(T=0, q=None, kv=None, w=None, pos=None, cs=None, slot=None, cache=None) == k.OK


def test_public_entries_validate_like_the_variant_entry():
    lib = k.lib()
    assert lib.dsv4_qnorm_rope_kv_quant_insert(A, A, A, A, A, 4096, A, A, 4, 64, -1, 8, 1e-6,
                                               None, None) == k.ERR_SHAPE
    assert lib.dsv4_qnorm_rope_kv_bf16_insert(A, A, A, A, A, 4096, A, A + 8, 4, 64, 5, 8, 1e-6,
                                              None, None) == k.ERR_ALIGN


def test_no_cpu_fallback_without_a_gpu():
    """A valid call on a machine without a GPU must fail loudly, not compute on the host."""
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; covered by the GPU tests")
    assert _call() == k.ERR_CUDA
    # the binding refuses host tensors before any call: there is no CPU path
    with pytest.raises(ValueError, match="CUDA tensor"):
        k.insert(k.STORE_FP8, torch.zeros(16, 8, 512, dtype=torch.bfloat16),
                 torch.zeros(16, 512, dtype=torch.bfloat16), torch.zeros(512, dtype=torch.bfloat16),
                 torch.zeros(16, dtype=torch.int64), torch.zeros(4096, 64),
                 torch.zeros(16, dtype=torch.int64), torch.zeros(4 * 64 * 584, dtype=torch.uint8),
                 4, 64, 1e-6, stream=0)


def test_launch_plan_small_and_stream():
    # 16 tokens x 9 rows = 144 rows: one row per warp, 2-warp CTAs
    p = k.launch_plan(16, 8, 152, 4)
    assert (p.variant, p.threads, p.rows_per_warp, p.rows, p.ctas) == (k.VARIANT_SMALL, 64, 1, 144, 72)
    # 131072 x 129 rows: persistent grid, 4 CTAs on each of 152 SMs
    p = k.launch_plan(131072, 128, 152, 4)
    assert (p.variant, p.threads, p.ctas, p.rows) == (k.VARIANT_STREAM, 256, 608, 131072 * 129)
    # the crossovers: with q heads, rows below the warp slots go SMALL, below 12
    # rounds of 3-row groups HALF; beyond, STREAM
    warp_slots = 152 * 4 * 8
    rnd = warp_slots * p.rows_per_warp
    assert k.launch_plan(warp_slots // 9 - 1, 8, 152, 4).variant == k.VARIANT_SMALL
    assert k.launch_plan(warp_slots // 9 + 1, 8, 152, 4).variant == k.VARIANT_HALF
    assert k.launch_plan(12 * rnd // 65 - 1, 64, 152, 4).variant == k.VARIANT_HALF
    assert k.launch_plan(12 * rnd // 65 + 1, 64, 152, 4).variant == k.VARIANT_STREAM
    # KV rows only: never HALF (they have their own kernel behind STREAM); the same
    # switch at the warp slots
    assert k.launch_plan(warp_slots - 1, 0, 152, 4).variant == k.VARIANT_SMALL
    assert k.launch_plan(warp_slots + 1, 0, 152, 4).variant == k.VARIANT_STREAM
    # forced variants
    assert k.launch_plan(131072, 128, 152, 4, k.VARIANT_SMALL).ctas == 131072 * 129 // 2
    p = k.launch_plan(3, 1, 152, 4, k.VARIANT_STREAM)
    assert p.ctas == 1 and p.rows == 6
    p = k.launch_plan(0, 1, 152, 4)
    assert p.ctas >= 1 and p.rows == 0


def test_launch_plan_rejects():
    for args in [(-1, 8, 152, 4), (16, -1, 152, 4), (16, 8, 0, 4), (16, 8, 152, 0)]:
        with pytest.raises(k.Dsv4Error):
            k.launch_plan(*args)
    with pytest.raises(k.Dsv4Error):
        k.launch_plan(16, 8, 152, 4, 9)
    plan = k.Plan()
    assert k.lib().dsv4_launch_plan(16, 8, 152, 4, 0, None) == k.ERR_NULL
    del plan


def test_library_has_no_oracle_dependency():
    """The CUDA library links nothing from the oracle or the input generator."""
    data = open(k.LIB_PATH, "rb").read()
    assert b"oracle_" not in data and b"synth_" not in data
    assert ctypes.CDLL(k.LIB_PATH)


def test_launch_plan_kv_rows_only():
    p = k.launch_plan(1000, 0, 152, 4)
    assert p.rows == 1000 and p.variant == k.VARIANT_SMALL and p.ctas == 500


def _ex(kv_norm=1, store=0, variant=0, q=A, kv=A, w=A, pos=A, cs=A, max_pos=4096, slot=A,
        cache=A, nb=4, bs=64, T=16, H=8, eps=1e-6, err=None):
    return k.lib().dsv4_insert_ex(store, variant, kv_norm, q, kv, w, pos, cs, max_pos, slot, cache,
                                  nb, bs, T, H, eps, err, None)


@pytest.mark.parametrize("kw,status", [
    (dict(kv_norm=2), k.ERR_VALUE), (dict(H=-1), k.ERR_SHAPE),
    (dict(q=None), k.ERR_NULL), (dict(w=None), k.ERR_NULL), (dict(kv=None), k.ERR_NULL),
    (dict(kv_norm=0, w=None, T=0), k.OK), (dict(H=0, q=None, T=0), k.OK),
    (dict(kv_norm=0, w=A + 8), k.ERR_ALIGN),
])
def test_ex_validation(kw, status):
    assert _ex(**kw) == status


def test_kv_only_and_prenormalised_entries_validate():
    lib = k.lib()
    # KV rows only: no q argument at all; weight required
    assert lib.dsv4_kv_norm_rope_insert(0, A, None, A, A, 4096, A, A, 4, 64, 16, 1e-6, None,
                                        None) == k.ERR_NULL
    assert lib.dsv4_kv_norm_rope_insert(5, A, A, A, A, 4096, A, A, 4, 64, 16, 1e-6, None,
                                        None) == k.ERR_VALUE
    assert lib.dsv4_kv_norm_rope_insert(1, A, A, A, A, 4096, A, A + 8, 4, 64, 16, 1e-6, None,
                                        None) == k.ERR_ALIGN
    assert lib.dsv4_kv_norm_rope_insert(0, A, A, A, A, 4096, A, A, 4, 64, 0, 1e-6, None,
                                        None) == k.OK
    # KV arrives normalised: no weight argument; q still required (H >= 1)
    assert lib.dsv4_qnorm_rope_kv_rope_quant_insert(A, A, A, A, 4096, A, A, 4, 64, 16, 0, 1e-6,
                                                    None, None) == k.ERR_SHAPE
    assert lib.dsv4_qnorm_rope_kv_rope_quant_insert(None, A, A, A, 4096, A, A, 4, 64, 16, 8, 1e-6,
                                                    None, None) == k.ERR_NULL
    assert lib.dsv4_qnorm_rope_kv_rope_quant_insert(A, A, A, A, 4096, A, A, 4, 64, 0, 8, 1e-6,
                                                    None, None) == k.OK


@pytest.mark.parametrize("args,status", [
    ((A, 4, 64, A, -1, A, None), k.ERR_SHAPE), ((A, 0, 64, A, 5, A, None), k.ERR_SHAPE),
    ((A, 4, 0, A, 5, A, None), k.ERR_SHAPE), ((None, 4, 64, A, 5, A, None), k.ERR_NULL),
    ((A, 4, 64, None, 5, A, None), k.ERR_NULL), ((A, 4, 64, A, 5, None, None), k.ERR_NULL),
    ((A + 4, 4, 64, A, 5, A, None), k.ERR_ALIGN), ((A, 4, 64, A + 4, 5, A, None), k.ERR_ALIGN),
    ((A, 4, 64, A, 5, A + 8, None), k.ERR_ALIGN), ((A, 4, 64, A, 5, A, A + 1), k.ERR_ALIGN),
    ((A + 8, 3, 7, A, 0, A, None), k.OK),
])
def test_gather_validation(args, status):
    assert k.lib().dsv4_dequant_gather(*args, None) == status


@pytest.mark.parametrize("kw,status", [
    (dict(m=-1), k.ERR_SHAPE), (dict(n=64), k.ERR_SHAPE), (dict(n=200), k.ERR_SHAPE),
    (dict(n=16512), k.ERR_SHAPE), (dict(eps=-1.0), k.ERR_VALUE), (dict(eps=math.nan), k.ERR_VALUE),
    (dict(x=None), k.ERR_NULL), (dict(res=None), k.ERR_NULL), (dict(g=None), k.ERR_NULL),
    (dict(out=None), k.ERR_NULL), (dict(codes=None), k.ERR_NULL), (dict(scales=None), k.ERR_NULL),
    (dict(x=A + 8), k.ERR_ALIGN), (dict(res=A + 2), k.ERR_ALIGN), (dict(g=A + 4), k.ERR_ALIGN),
    (dict(out=A + 8), k.ERR_ALIGN), (dict(codes=A + 4), k.ERR_ALIGN),
    (dict(m=0, x=None, res=None, g=None, out=None, codes=None, scales=None), k.OK),
])
def test_mxfp8_validation(kw, status):
    a = dict(x=A, res=A, g=A, m=4, n=1024, eps=1e-6, out=A, codes=A, scales=A + 1)
    a.update(kw)
    assert k.lib().dsv4_add_gemma_rmsnorm_mxfp8(a["x"], a["res"], a["g"], a["m"], a["n"], a["eps"],
                                                a["out"], a["codes"], a["scales"], None) == status


def test_mxfp8_scale_bytes():
    assert k.mxfp8_scale_bytes(1, 128) == 128 * 4
    assert k.mxfp8_scale_bytes(129, 7168) == 256 * 224
    assert k.mxfp8_scale_bytes(5, 100) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(T=-1), k.ERR_SHAPE), (dict(nb=0), k.ERR_SHAPE), (dict(bs=0), k.ERR_SHAPE),
    (dict(nb=2 ** 62), k.ERR_SHAPE),
    (dict(kp=None), k.ERR_NULL), (dict(sl=None), k.ERR_NULL), (dict(cache=None), k.ERR_NULL),
    (dict(kp=A + 8), k.ERR_ALIGN), (dict(sl=A + 4), k.ERR_ALIGN), (dict(cache=A + 2), k.ERR_ALIGN),
    (dict(err=A + 2), k.ERR_ALIGN),
    (dict(T=0, kp=None, sl=None, cache=None), k.OK),
])
def test_indexer_insert_validation(kw, status):
    a = dict(kp=A, sl=A, cache=A + 4, nb=4, bs=64, T=5, err=None)
    a.update(kw)
    assert k.lib().dsv4_indexer_k_quant_insert(a["kp"], a["sl"], a["cache"], a["nb"], a["bs"],
                                               a["T"], a["err"], None) == status


@pytest.mark.parametrize("kw,status", [
    (dict(n=-1), k.ERR_SHAPE), (dict(nb=0), k.ERR_SHAPE), (dict(bs=0), k.ERR_SHAPE),
    (dict(cache=None), k.ERR_NULL), (dict(sl=None), k.ERR_NULL), (dict(out=None), k.ERR_NULL),
    (dict(scale=None), k.ERR_NULL),
    (dict(cache=A + 2), k.ERR_ALIGN), (dict(sl=A + 4), k.ERR_ALIGN), (dict(out=A + 4), k.ERR_ALIGN),
    (dict(scale=A + 2), k.ERR_ALIGN), (dict(err=A + 1), k.ERR_ALIGN),
    (dict(n=0, cache=None, sl=None, out=None, scale=None), k.OK),
])
def test_indexer_gather_validation(kw, status):
    a = dict(cache=A + 4, nb=4, bs=3, sl=A, n=5, out=A + 8, scale=A + 4, err=None)
    a.update(kw)
    assert k.lib().dsv4_indexer_k_gather(a["cache"], a["nb"], a["bs"], a["sl"], a["n"], a["out"],
                                         a["scale"], a["err"], None) == status


def test_indexer_cache_bytes():
    assert k.indexer_cache_bytes(2048, 64) == 2048 * 64 * 132
    assert k.indexer_cache_bytes(3, 5) == 3 * 5 * 132
    assert k.indexer_cache_bytes(0, 64) == 0


def test_indexer_entries_have_no_cpu_fallback():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; covered by the GPU tests")
    assert k.lib().dsv4_indexer_k_quant_insert(A, A, A, 4, 64, 5, None, None) == k.ERR_CUDA
    assert k.lib().dsv4_indexer_k_gather(A, 4, 64, A, 5, A, A, None, None) == k.ERR_CUDA


def test_caches_beyond_two_to_the_32_slots_are_rejected():
    """num_blocks * block_size <= 2^32 for every entry that takes a cache."""
    lib = k.lib()
    nb_ok, nb_bad = (1 << 32) // 64, (1 << 32) // 64 + 1
    assert lib.dsv4_dequant_gather(A, nb_bad, 64, A, 5, A, None, None) == k.ERR_SHAPE
    assert lib.dsv4_indexer_k_quant_insert(A, A, A, nb_bad, 64, 5, None, None) == k.ERR_SHAPE
    assert lib.dsv4_indexer_k_gather(A, nb_bad, 64, A, 5, A, A, None, None) == k.ERR_SHAPE
    assert lib.dsv4_insert_ex(0, 0, 1, A, A, A, A, A, 4096, A, A, nb_bad, 64, 16, 8, 1e-6,
                              None, None) == k.ERR_SHAPE
    # exactly 2^32 slots passes the shape check (zero tokens: no launch)
    assert lib.dsv4_insert_ex(0, 0, 1, A, A, A, A, A, 4096, A, A, nb_ok, 64, 0, 8, 1e-6,
                              None, None) == k.OK
    assert lib.dsv4_indexer_k_quant_insert(A, A, A, nb_ok, 64, 0, None, None) == k.OK


@pytest.mark.parametrize("d", [2, 3, 7, 64, 100, 1000, (1 << 31) - 1, 1 << 31, (1 << 32) - 1])
def test_fast_division_identity(d):
    """The multiply-high division the kernels use (fastdiv.h): with
    M = floor((2^64 - 1) / d) + 1, n // d == (M * n) >> 64 for 32-bit n
    (Lemire, Kaser, Kurz 2019, Theorem 1), checked at the edges of n and at
    multiples of d and their neighbours."""
    m = (2**64 - 1) // d + 1
    ns = {0, 1, d - 1, d, d + 1, 2**32 - 1, 2**32 - 2, 2**31, 12345678}
    for q in (1, 2, 3, 1000, (2**32 - 1) // d):
        ns |= {q * d - 1, q * d, q * d + 1}
    for n in ns:
        if 0 <= n < 2**32:
            assert (m * n) >> 64 == n // d, (n, d)


def test_launch_plan_for_kv_rows_only_stream():
    """With no q heads STREAM runs the KV-row kernel: 4 rows per warp (one per quarter)."""
    plan = k.launch_plan(100000, 0, 152, 2, k.VARIANT_STREAM)
    assert plan.rows_per_warp == 4 and plan.threads == 256 and plan.ctas == 152 * 2
    plan = k.launch_plan(100, 0, 152, 2, k.VARIANT_STREAM)
    assert plan.ctas == 4  # 25 groups of four rows, 8 warps per CTA
    plan = k.launch_plan(100000, 8, 152, 3, k.VARIANT_STREAM)
    assert plan.rows_per_warp == 3


def test_launch_plan_half():
    """HALF: ceil(T/2) KV row pairs plus groups of 4 q rows, 8 warps per CTA."""
    plan = k.launch_plan(256, 64, 152, 3, k.VARIANT_HALF)
    items = 128 + 256 * 64 // 4
    assert plan.variant == k.VARIANT_HALF and plan.rows_per_warp == 4 and plan.threads == 256
    assert plan.ctas == min(-(-items // 8), 152 * 3)
    assert k.launch_plan(3, 1, 152, 3, k.VARIANT_HALF).ctas == 1


def test_binding_rejects_mistyped_and_misshaped_tensors():
    """Element types, contiguity, device and sizes are checked before the C call."""
    torch = pytest.importorskip("torch")
    T, H = 4, 2
    ok = dict(q=torch.zeros(T, H, 512, dtype=torch.bfloat16), kv=torch.zeros(T, 512, dtype=torch.bfloat16),
              w=torch.zeros(512, dtype=torch.bfloat16), pos=torch.zeros(T, dtype=torch.int64),
              cs=torch.zeros(8, 64), sl=torch.zeros(T, dtype=torch.int64),
              cache=torch.zeros(2 * 4 * 584, dtype=torch.uint8))

    def call(**kw):
        a = dict(ok); a.update(kw)
        k.insert(k.STORE_FP8, a["q"], a["kv"], a["w"], a["pos"], a["cs"], a["sl"], a["cache"], 2, 4, 1e-6,
                 stream=0)

    with pytest.raises(TypeError, match="positions"):
        call(pos=torch.zeros(T, dtype=torch.int32))
    with pytest.raises(TypeError, match="cos_sin_cache"):
        call(cs=torch.zeros(8, 64, dtype=torch.float64))
    with pytest.raises(TypeError, match="q"):
        call(q=torch.zeros(T, H, 512))
    with pytest.raises(ValueError, match="contiguous"):
        call(kv=torch.zeros(512, T, dtype=torch.bfloat16).t())
    with pytest.raises(ValueError, match="kv:"):
        call(kv=torch.zeros(T + 1, 512, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="kv_cache"):
        call(cache=torch.zeros(100, dtype=torch.uint8))
    with pytest.raises(ValueError, match="CUDA tensor"):
        call()
    with pytest.raises(TypeError, match="k_out"):
        k.indexer_k_gather(torch.zeros(132 * 64, dtype=torch.uint8), 1, 64, torch.zeros(3, dtype=torch.int64),
                           torch.zeros(3, 128, dtype=torch.int16), torch.zeros(3))


def test_bounded_wait_check_rejects_negative_budget():
    lib = k.lib()
    assert lib.dsv4_check_bounded_wait(-1, None, None) == k.ERR_VALUE
    with pytest.raises(ValueError):
        k.check_bounded_wait(-5)
