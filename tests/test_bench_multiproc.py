"""The benchmark's multi-rank logic (replicas, barrier, max-over-ranks timing) on CPU with gloo."""
import multiprocessing as mp
import os
import socket

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank), PA_BENCH_BACKEND="gloo")
    import torch.distributed as dist
    import bench
    ws_, rank_, local = bench.dist_init()
    bench.barrier(ws_)
    slowest = bench.max_over_ranks(1.5 + rank, ws_, None)   # rank 1 is the slow one
    value = bench.job_throughput(1_000_000_000, ws_, slowest)
    bench.barrier(ws_)
    q.put((rank_, ws_, slowest, value))
    dist.destroy_process_group()


def test_two_rank_timing_is_max_over_ranks():
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
    assert [r[1] for r in res] == [2, 2]
    assert all(r[2] == pytest.approx(2.5) for r in res)            # both ranks see the slowest time
    assert all(r[3] == pytest.approx(2 * 1e9 / 2.5e-3 / 1e9) for r in res)  # both ranks' bytes / max time


def test_single_rank_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.0, 1, None) == 3.0
    assert bench.job_throughput(4_000_000_000, 1, 2.0) == pytest.approx(2000.0)


def test_timing_protocol_batches():
    """K timed steps are cut into 5 batches (fewer when K < 5) that add up to exactly K."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.batch_sizes(250) == [50] * 5
    assert bench.batch_sizes(20) == [4] * 5
    assert bench.batch_sizes(3) == [1, 1, 1]
    for K in range(1, 300):
        b = bench.batch_sizes(K)
        assert sum(b) == K and len(b) == min(5, K) and max(b) - min(b) <= 1
