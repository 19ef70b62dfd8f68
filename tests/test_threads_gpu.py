"""Host threads calling the library at once, each on its own CUDA stream.

The C ABI keeps per-device caches (SM count, occupancy per kernel) that are
filled on first use; several threads reaching them together, each launching on
its own stream, must get the same results as one thread calling serially.
"""
import threading

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


def _jobs():
    """(name, make() -> buffers, run(buffers, stream), result(buffers) -> numpy)"""
    jobs = []
    for i, (T, H, variant) in enumerate([(300, 8, k.VARIANT_AUTO), (1000, 64, k.VARIANT_HALF),
                                         (2000, 0, k.VARIANT_STREAM), (50, 3, k.VARIANT_SMALL)]):
        wl = configs.generic(T, H, seed=300 + i)
        inp = harness.make_inputs(wl)

        def make(inp=inp, H=H):
            t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV)
            return dict(q=t(inp.q) if H else None, kv=t(inp.kv), w=t(inp.w),
                        pos=torch.from_numpy(inp.positions).to(DEV),
                        cs=torch.from_numpy(inp.cos_sin).to(DEV),
                        sl=torch.from_numpy(inp.slots).to(DEV),
                        cache=torch.from_numpy(inp.poison.copy()).to(DEV))

        def run(b, stream, wl=wl, H=H, variant=variant):
            k.insert(k.STORE_FP8, b["q"], b["kv"], b["w"], b["pos"], b["cs"], b["sl"], b["cache"],
                     wl.num_blocks, wl.block_size, wl.eps, stream=stream, variant=variant,
                     num_heads=H)

        def result(b):
            return b["cache"].cpu().numpy()

        jobs.append((f"insert T{T} H{H} v{variant}", make, run, result))
    # the indexer insert and the MXFP8 quantiser
    n, nb, bs = 700, 16, 64
    kb = synth.normal_bf16(n * 128, 8, synth.TID_IDX_K).reshape(n, 128)
    sl = synth.permutation(nb * bs, 8, synth.TID_SLOT)[:n].astype(np.int64)

    def make_idx():
        return dict(k=torch.from_numpy(kb.view(np.int16)).to(DEV), sl=torch.from_numpy(sl).to(DEV),
                    cache=torch.zeros(nb * bs * 132, dtype=torch.uint8, device=DEV))

    jobs.append(("indexer", make_idx,
                 lambda b, s: k.indexer_k_quant_insert(b["k"], b["sl"], b["cache"], nb, bs, stream=s),
                 lambda b: b["cache"].cpu().numpy()))
    m, hid = 300, 2048
    x = synth.normal_bf16(m * hid, 9, 1).reshape(m, hid)
    r = synth.normal_bf16(m * hid, 9, 2).reshape(m, hid)
    g = synth.normal_bf16(hid, 9, 3)

    def make_mx():
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV)
        return dict(x=t(x), r=t(r), g=t(g), out=torch.zeros((m, hid), dtype=torch.int16, device=DEV),
                    codes=torch.zeros((m, hid), dtype=torch.uint8, device=DEV),
                    scales=torch.zeros(k.mxfp8_scale_bytes(m, hid), dtype=torch.uint8, device=DEV))

    jobs.append(("mxfp8", make_mx,
                 lambda b, s: k.add_gemma_rmsnorm_mxfp8(b["x"], b["r"], b["g"], 1e-6, b["out"],
                                                        b["codes"], b["scales"], stream=s),
                 lambda b: np.concatenate([b["out"].cpu().numpy().view(np.uint8).ravel(),
                                           b["codes"].cpu().numpy().ravel(),
                                           b["scales"].cpu().numpy().ravel()])))
    return jobs


def test_concurrent_host_threads_match_serial_calls():
    jobs = _jobs()
    # several rounds: the first reaches the library's empty caches from many threads
    for _ in range(3):
        bufs = [make() for _, make, _, _ in jobs]
        torch.cuda.synchronize()
        errors = []
        barrier = threading.Barrier(len(jobs))

        def worker(i):
            try:
                s = torch.cuda.Stream(DEV)
                barrier.wait()
                for _ in range(4):
                    jobs[i][2](bufs[i], s)
                s.synchronize()
            except Exception as e:  # pragma: no cover - reported below
                errors.append((jobs[i][0], repr(e)))

        threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(jobs))]
        for t in threads:
            t.start()
        for t in threads:
            t.join()
        assert not errors, errors
        for (name, make, run, result), b in zip(jobs, bufs):
            ref = make()
            s = torch.cuda.Stream(DEV)
            for _ in range(4):
                run(ref, s)
            s.synchronize()
            assert np.array_equal(result(b), result(ref)), name
