"""The multi-rank path of bench.py on CPU: two gloo ranks, each with its own time.

bench.py runs one batch per rank (weak scaling) and reports the whole job: every rank's
FLOPs over the slowest rank's time.  Here two processes join a gloo group on 127.0.0.1
and check that both see the slowest time and the same aggregate, and that the one-rank
path needs no process group.
"""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_env()
        my_ms = 10.0 + 5.0 * rank                 # rank 1 is the slow one
        ms = bench.reduce_max(my_ms, w, torch.device("cpu"))
        value = bench.aggregate_tflops(2.0e12, w, ms)
        dist.barrier()
        out_q.put((r, w, local, ms, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time_and_aggregate():
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1] and all(r[1] == 2 for r in res) and [r[2] for r in res] == [0, 1]
    for _, _, _, ms, value in res:
        assert ms == 15.0                          # both ranks see the slowest rank
        assert value == pytest.approx(2 * 2.0e12 / 15e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.reduce_max(3.5, 1, None) == 3.5
    assert bench.aggregate_tflops(1e12, 1, 1.0) == pytest.approx(1000.0)
