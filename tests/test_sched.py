"""Host-side scheduling: shards, waves, and a world-size-2 gather over gloo on
CPU (the per-rank simulator here is the CPU oracle; on GPUs it is the CUDA
library)."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as tmp

from experiment_network_simulation_gb300 import inputs as I
from experiment_network_simulation_gb300 import mv, sched
from oracle import oracle as O


def test_shard_covers_once():
    for n in (0, 1, 5, 16, 17):
        for world in (1, 2, 3, 8):
            got = [i for r in range(world) for i in sched.shard(n, r, world)]
            assert got == list(range(n))
            sizes = [len(sched.shard(n, r, world)) for r in range(world)]
            assert max(sizes) - min(sizes) <= 1


def test_waves_fit_budget_and_cover():
    b = I.config2(n_exp=40)
    one = mv.workspace_bytes(b.subset([0]).pack())
    budget = 6 * one
    waves = sched.plan_waves(b, budget, mv.workspace_bytes)
    assert [i for w in waves for i in w] == list(range(40))
    for w in waves:
        assert mv.workspace_bytes(b.subset(w).pack()) <= budget
    assert len(waves) > 1
    with pytest.raises(ValueError):
        sched.plan_waves(b, one // 4, mv.workspace_bytes)


def _worker(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = I.config1()
        res = sched.run_sharded(b, O.run, rank, world)
        if rank == 0:
            q.put({k: v for k, v in res.items()})
    finally:
        dist.destroy_process_group()


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_gloo_two_ranks_gather_equals_single_process():
    ctx = tmp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = q.get(timeout=300)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    want = O.run(I.config1().pack())
    for k in sched.PER_EXP_KEYS:
        assert np.array_equal(got[k], want[k]), k
    n = want["node_offset"][-1]
    assert np.array_equal(got["node_end"], want["node_end"][:n])
