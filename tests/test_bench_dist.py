"""Host logic of the multi-rank bench path on CPU (gloo, world size 2): each rank
packs its own tree (weak scaling), and the timed region is the max over ranks."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist
    import bench
    import synth
    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = synth.galton_watson(seed=bench.rank_seed(rank), budget=500, seg=(5, 60))
    T = oracle.pack_ref(t.seqs)["T"]
    local = float(10 * (rank + 1))
    bench.barrier(world)
    out[rank] = (bench.reduce_max(local, world), T, [len(s) for s in t.seqs])
    dist.destroy_process_group()


def test_two_rank_max_and_distinct_trees():
    mp = torch.multiprocessing.get_context("spawn")
    mgr = mp.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [mp.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert out[0][0] == out[1][0] == 20.0          # max over ranks
    assert out[0][1] == out[1][1] == 500           # same budget per rank (weak scaling)
    assert out[0][2] != out[1][2]                  # but each rank has its own tree


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.rank_seed(3) == 3
