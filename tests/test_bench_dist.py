"""The multi-GPU path of bench.py is replicas with a timing barrier and a
max-over-ranks reduction; its host logic runs here as two gloo ranks on CPU."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        env = bench.dist_env()
        bench.barrier(ws)
        mx = bench.max_over_ranks(10.0 + rank, ws)
        sm = bench.sum_over_ranks(100.0 * (rank + 1), ws)
        bench.barrier(ws)
        q.put((rank, env, mx, sm))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation():
    ws = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(ws))
    for rank, env, mx, sm in got:
        assert env == (ws, rank, rank)
        assert mx == 11.0          # max over ranks of the elapsed time
        assert sm == 300.0         # total work of all ranks


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.sum_over_ranks(2.0, 1) == 2.0
