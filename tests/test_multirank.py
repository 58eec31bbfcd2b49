"""The N > 1 host logic of bench.py on CPU: two gloo ranks, each verifying its
own batch (weak scaling), combine their timings with a max over ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    r, w, lr = bench.dist_env()
    bench.barrier(w)
    t = bench.max_over_ranks(1.5 + rank, w)
    seeds = [bench.rank_seed(r, s) for s in range(3)]
    q.put((r, w, lr, t, seeds))
    dist.destroy_process_group()


def test_two_gloo_ranks_max_and_independent_seeds():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1] and all(r[1] == 2 for r in res)
    assert all(r[3] == 2.5 for r in res)  # max over ranks seen by every rank
    s0, s1 = set(res[0][4]), set(res[1][4])
    assert not (s0 & s1)  # each rank's batches draw different uniforms


def test_single_rank_helpers():
    import bench
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.rank_seed(0, 5) == 5 and bench.rank_seed(1, 5) == (1 << 32) + 5
    assert len(bench.source_hash()) == 64
