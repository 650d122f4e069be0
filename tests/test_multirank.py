"""The multi-rank plumbing of bench.py on CPU: two gloo ranks (127.0.0.1).

Each rank owns its own dictionaries (weak scaling, nothing exchanged on the
data path); the only collective is the max of the step time over ranks, and
the reported value is every rank's vectors over the slowest rank's time.
Each rank also runs the oracle on a slice of its own workload, the work a
rank does on its GPU, to check that ranks see different, reproducible data.
"""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from dictionary_sparse_kv_gb300 import synthetic as S
        from oracle import oracle as O
        w = bench.rank_workload(S.WORKLOADS["tiny"], rank)
        data = S.WorkloadData(w)
        x = data.inputs(0, 8)
        p = O.Params(w.N, w.d, w.n, w.s, 1e-4, 0.20, O.F32)
        res = O.encode(p, data.atoms[0], x[0])
        slow = bench.max_over_ranks(10.0 + rank)           # rank 1 is the slow one
        out[rank] = (float(np.abs(data.atoms).sum()), res.idx.copy(), slow)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
    (a0, idx0, t0), (a1, idx1, t1) = out[0], out[1]
    assert a0 != a1                                       # each rank its own dictionaries
    assert not np.array_equal(idx0, idx1)
    assert t0 == t1 == 11.0                               # the slowest rank's time everywhere
    import bench
    from dictionary_sparse_kv_gb300 import synthetic as S
    # the same rank always gets the same data
    w = bench.rank_workload(S.WORKLOADS["tiny"], 1)
    assert float(np.abs(S.WorkloadData(w).atoms).sum()) == a1
    assert bench.job_throughput(world, 20, 7168, t1) == pytest.approx(2 * 20 * 7168 / 0.011)


def test_single_process_max_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
