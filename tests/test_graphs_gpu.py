"""Every entry point can be captured into a CUDA graph and replayed.

Serving loops run decode steps as graph replays.  Each operation is run eagerly
once, then captured (after a warm-up call, as graph capture expects) and
replayed once on fresh copies of the same inputs; the replay must produce the
same bytes as the eager run.
"""
import numpy as np
import pytest

import synth
from synth import configs
from tests import harness

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import kv_norm_rope_gb300 as k  # noqa: E402

DEV = torch.device("cuda:0")


def _replay(fn, fresh):
    """fn(bufs) enqueues the operation on the current stream; fresh() returns new
    input/output buffers.  Returns the buffers of one eager run and of one replay."""
    eager = fresh()
    fn(eager)
    torch.cuda.synchronize()
    warm = fresh()
    fn(warm)  # warm-up outside the capture
    torch.cuda.synchronize()
    bufs = fresh()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn(bufs)
    g.replay()
    torch.cuda.synchronize()
    return eager, bufs


@pytest.mark.parametrize("variant", [k.VARIANT_AUTO, k.VARIANT_SMALL, k.VARIANT_STREAM,
                                     k.VARIANT_HALF])
@pytest.mark.parametrize("H", [64, 0])
def test_fused_step_in_a_graph(variant, H):
    wl = configs.generic(256, H, seed=120 + H)
    inp = harness.make_inputs(wl)

    def fresh():
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV)
        return dict(q=t(inp.q) if H else None, kv=t(inp.kv), w=t(inp.w),
                    pos=torch.from_numpy(inp.positions).to(DEV), cs=torch.from_numpy(inp.cos_sin).to(DEV),
                    sl=torch.from_numpy(inp.slots).to(DEV), cache=torch.from_numpy(inp.poison.copy()).to(DEV),
                    err=torch.zeros(1, dtype=torch.int32, device=DEV))

    def fn(b):
        k.insert(k.STORE_FP8, b["q"], b["kv"], b["w"], b["pos"], b["cs"], b["sl"], b["cache"],
                 wl.num_blocks, wl.block_size, wl.eps, device_error=b["err"], variant=variant,
                 num_heads=H)

    eager, rep = _replay(fn, fresh)
    assert torch.equal(rep["cache"], eager["cache"])
    assert int(rep["err"].item()) == int(eager["err"].item())
    if H:
        assert torch.equal(rep["q"], eager["q"])
        assert not torch.equal(rep["q"], fresh()["q"])  # the replay did run


def test_readers_and_quantisers_in_a_graph():
    # FP8 cache reader
    wl = configs.TINY
    inp = harness.make_inputs(wl)
    cache = torch.from_numpy(harness.run_gpu(inp).cache).to(DEV)
    slots = torch.from_numpy(inp.slots).to(DEV)
    eager, rep = _replay(lambda b: k.dequant_gather(cache, wl.num_blocks, wl.block_size, slots, b),
                         lambda: torch.full((wl.T, 512), 7, dtype=torch.int16, device=DEV))
    assert torch.equal(rep, eager) and not torch.equal(rep, torch.full_like(rep, 7))
    # indexer K insert and gather
    n, nb, bs = 300, 8, 64
    kb = torch.from_numpy(synth.normal_bf16(n * 128, 5, synth.TID_IDX_K).view(np.int16)).to(DEV).view(n, 128)
    sl = torch.from_numpy(synth.permutation(nb * bs, 5, synth.TID_SLOT)[:n].astype(np.int64)).to(DEV)
    poison = torch.from_numpy(synth.poison_bytes(nb * bs * 132, 5)).to(DEV)
    eager, rep = _replay(lambda c: k.indexer_k_quant_insert(kb, sl, c, nb, bs), lambda: poison.clone())
    assert torch.equal(rep, eager) and not torch.equal(rep, poison)
    def gather(b):
        k.indexer_k_gather(eager, nb, bs, sl, b[0], b[1])
    fresh = lambda: (torch.zeros((n, 128), dtype=torch.uint8, device=DEV),
                     torch.zeros(n, dtype=torch.float32, device=DEV))
    e2, r2 = _replay(gather, fresh)
    assert torch.equal(r2[0], e2[0]) and torch.equal(r2[1], e2[1]) and bool((r2[1] > 0).all())
    # MXFP8
    m, hidden = 200, 1024
    x = torch.from_numpy(synth.normal_bf16(m * hidden, 6, 1).view(np.int16)).to(DEV).view(m, hidden)
    r = torch.from_numpy(synth.normal_bf16(m * hidden, 6, 2).view(np.int16)).to(DEV).view(m, hidden)
    g = torch.from_numpy(synth.normal_bf16(hidden, 6, 3).view(np.int16)).to(DEV)
    def mx(b):
        k.add_gemma_rmsnorm_mxfp8(x, r, g, 1e-6, b[0], b[1], b[2])
    fresh = lambda: (torch.zeros((m, hidden), dtype=torch.int16, device=DEV),
                     torch.zeros((m, hidden), dtype=torch.uint8, device=DEV),
                     torch.full((k.mxfp8_scale_bytes(m, hidden),), 9, dtype=torch.uint8, device=DEV))
    e3, r3 = _replay(mx, fresh)
    for a, b in zip(r3, e3):
        assert torch.equal(a, b)
