"""Replica logic of bench.py on CPU with two gloo ranks.

Each rank owns whole matrices (no data exchange); the ranks only meet at a
barrier and a max over their step times.
"""

import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    import workloads
    r, w, local = bench.dist_env()
    dist = bench.init_dist(w)
    bench.barrier(dist)
    ms = 10.0 + 5.0 * r                       # rank 1 is the slow one
    ms_max = bench.max_over_ranks(dist, ms)
    g = workloads.gradients(1, 16, 32, bench.rank_seed_base(r), kind="lognormal_rows")
    gathered = [torch.zeros_like(g.float()) for _ in range(w)]
    dist.all_gather(gathered, g.float())      # test-only: compare the ranks' inputs
    out[r] = (ms_max, bench.aggregate_value(96, w, ms_max), bool(torch.equal(gathered[0], gathered[1])))
    dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling():
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_worker, args=(2, port, out), nprocs=2, start_method="spawn")
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0            # max over ranks
    assert res[0][1] == pytest.approx(96 * 2 / 0.015)  # whole-job matrices/s
    assert res[0][2] is False                          # each rank owns different matrices


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.init_dist(1) is None
    assert bench.max_over_ranks(None, 3.5) == 3.5
    assert bench.aggregate_value(96, 1, 30.0) == pytest.approx(3200.0)
