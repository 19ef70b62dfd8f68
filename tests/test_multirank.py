"""The N > 1 benchmark path on CPU: two gloo ranks.  Each rank gets an independent
batch of the same shape (token sharding, no data exchange), and the timing reduction
takes the max over ranks while the work adds up (weak scaling)."""
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    from synth import configs
    from tests import harness

    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    r, w, lr = bench.dist_env()
    assert (r, w, lr) == (rank, world, rank)
    wl = bench.rank_workload(configs.TINY, rank)
    inp = harness.make_inputs(wl)
    ref_q, ref_cache, err = harness.run_oracle(inp)
    # a rank's "step time": rank 1 is slower; the job time is the slowest rank
    t = 1.0 + rank
    bench.barrier(world)
    tmax = bench.max_over_ranks(t, world)
    tok = bench.sum_over_ranks(float(wl.T), world)
    np.savez(os.path.join(out_dir, f"rank{rank}.npz"), q=inp.q, slots=inp.slots, ref_q=ref_q,
             ref_cache=ref_cache, err=err, tmax=tmax, tok=tok, T=wl.T, H=wl.H, seed=wl.seed)
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_by_batch(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    r0 = np.load(tmp_path / "rank0.npz")
    r1 = np.load(tmp_path / "rank1.npz")
    assert int(r0["T"]) == int(r1["T"]) and int(r0["H"]) == int(r1["H"])
    assert int(r0["seed"]) != int(r1["seed"])
    assert not np.array_equal(r0["q"], r1["q"])          # independent batches
    assert float(r0["tmax"]) == float(r1["tmax"]) == 2.0  # slowest rank
    assert float(r0["tok"]) == float(r1["tok"]) == 2 * int(r0["T"])
    assert int(r0["err"]) == int(r1["err"]) == 0
    del torch


def test_rank_workload_is_a_pure_function_of_rank():
    sys.path.insert(0, ROOT)
    import bench
    from synth import configs
    a = bench.rank_workload(configs.PREFILL, 3)
    b = bench.rank_workload(configs.PREFILL, 3)
    assert a == b and a.seed == configs.PREFILL.seed + 3000
    assert np.array_equal(a.positions(), configs.PREFILL.positions())
    assert not np.array_equal(a.slot_mapping(), configs.PREFILL.slot_mapping())
    assert bench.rank_workload(configs.PREFILL, 0) is configs.PREFILL
