"""bench.py's multi-rank path on CPU: two gloo ranks on 127.0.0.1, as torchrun would
start them. The timing aggregation takes the maximum over ranks, the work the sum, the
value is the whole job's units over that time, and each rank draws its own seeds (the
replicas are independent requests)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    import torch.distributed as dist
    r, w, local = bench.dist_setup(world)
    assert (r, w, local) == (rank, world, rank) and dist.get_backend() == "gloo"
    bench.barrier(w)
    t_local = [0.25, 0.5][r]                 # seconds each rank took for its steps
    tokens_local = [64, 64][r]
    t_max = bench.max_over_ranks(t_local, w)
    tokens_all = bench.sum_over_ranks(tokens_local, w)
    cfg = bench.workload_config("tiny", 6, r)
    out[r] = (t_max, tokens_all, tokens_all / t_max, cfg.seed, cfg.steps)
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_torchrun():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][:3] == res[1][:3] == (0.5, 128.0, 256.0)   # max time, summed work, job throughput
    assert res[0][3] != res[1][3]                            # per-rank seeds: independent replicas
    assert res[0][4] >= 6 and res[1][4] >= 6
