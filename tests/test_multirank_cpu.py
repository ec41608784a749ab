"""The bench's multi-rank path on CPU: two gloo ranks run the same rank helpers
bench.py uses under torchrun (barrier, max-over-ranks timing, whole-job throughput).
Each rank is an independent replica; nothing on the data path is exchanged."""
from __future__ import annotations

import os
import socket

import pytest

torch = pytest.importorskip("torch")
mp = torch.multiprocessing


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    import torch.distributed as dist
    w, r = bench.dist_init("gloo")
    bench.barrier()
    elapsed = 1.0 + rank            # rank 1 is the slow one
    mx = bench.reduce_max(elapsed)
    value = bench.aggregate_throughput(50, w, mx)
    q.put((r, w, mx, value))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, w, mx, value in res:
        assert w == 2 and mx == 2.0
        assert value == pytest.approx(50 * 2 / 2.0)


def test_single_rank_helpers_without_a_process_group():
    import bench
    assert bench.reduce_max(3.5) == 3.5
    assert bench.aggregate_throughput(10, 1, 2.0) == 5.0
    w = bench.wl.CONFIGS["steady_state_10k"]
    flops, byts = bench.block_work(w, 10000)
    # closed forms at the 10,000-frame steady state: N = 72*256 + 60000
    assert bench.visible_tokens(w, 10000) == 78432
    assert flops == 4 * 262 * 78432 * 16 * 64
    assert byts == (2 * 78432 + 2 * 262) * 16 * 64 * 2
