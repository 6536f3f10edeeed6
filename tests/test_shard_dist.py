"""The multi-GPU row split's host logic on CPU, as two gloo ranks: each rank
computes the product of its row shard (the oracle stands in for the GPU
kernel, rows [g N / G, (g + 1) N / G), multiples of 128 for FP8), the shards
are all-gathered with bench.gather_shards, and the result must equal the
oracle's product of the whole matrix bit for bit (the oracle computes every
row independently)."""
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


def _worker(rank, ws, port, fmt, q_out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    import oracle as O
    from speculative_decode_verification_qmm_gb300 import shard_rows, synth
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        if fmt == "q4":
            N, K, M, align = 777, 256, 5, 1
            wb, sc, ofmt = O.q4_0_quantize(synth.weights(N, K, 70)), None, O.FMT_Q4_0
        else:
            N, K, M, align = 640, 256, 3, 128
            wb, sc = O.fp8_quantize(synth.weights(N, K, 71))
            ofmt = O.FMT_FP8
        a = synth.activations(M, K, 72, outliers=True)
        n0, n1 = shard_rows(N, ws, rank, align)
        part, _ = O.verify_rows(ofmt, wb, sc, N, K, a, rows=np.arange(n0, n1))
        full = bench.gather_shards(torch.from_numpy(part), N, ws, align).numpy()
        ref, _ = O.verify_rows(ofmt, wb, sc, N, K, a)
        q_out.put((rank, (n0, n1), bool((full.view(np.uint64) == ref.view(np.uint64)).all())))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("fmt", ["q4", "fp8"])
def test_two_rank_row_split_gathers_the_full_product(fmt):
    ws = 2
    ctx = mp.get_context("spawn")
    q_out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, fmt, q_out)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(180)
        assert p.exitcode == 0
    got = sorted(q_out.get(timeout=5) for _ in range(ws))
    assert [r for r, _, _ in got] == [0, 1]
    assert got[0][1][0] == 0 and got[0][1][1] == got[1][1][0] and all(ok for _, _, ok in got)
    if fmt == "fp8":
        assert all(b % 128 == 0 for _, (a_, b), _ in got)


def test_shard_rows_partition():
    from speculative_decode_verification_qmm_gb300 import shard_rows
    for N in (1, 7, 128, 777, 5120, 34816):
        for G in (1, 2, 3, 4, 8):
            for align in (1, 128):
                if align == 128 and N % 128:
                    continue
                cuts = [shard_rows(N, G, g, align) for g in range(G)]
                assert cuts[0][0] == 0 and cuts[-1][1] == N
                assert all(cuts[g][1] == cuts[g + 1][0] for g in range(G - 1))
                assert all(a % align == 0 and (b % align == 0 or b == N) for a, b in cuts)
