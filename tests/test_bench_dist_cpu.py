"""The multi-rank path of bench.py (one independent replica per rank, a
barrier around the timed region, the slowest rank's time) with world size 2
over gloo on the CPU."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE="2", LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=2)
    import bench
    ws, r, local = bench._dist()
    bench._barrier(ws)
    slowest = bench._max_over_ranks(10.0 + 5.0 * rank, ws)   # step times 10 and 15 ms
    rate = bench._job_rate(1e9, slowest, ws)
    bench._barrier(ws)
    q.put((r, ws, local, slowest, rate))
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_step_and_sum_the_replicas():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1] and all(o[1] == 2 for o in out)
    assert [o[2] for o in out] == [0, 1]
    for _, _, _, slowest, rate in out:
        assert slowest == 15.0                     # both ranks see the slowest rank
        assert rate == pytest.approx(2 * 1e9 / 15e-3)  # two replicas in 15 ms


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench._max_over_ranks(3.0, 1) == 3.0
    assert bench._job_rate(100.0, 1000.0, 1) == pytest.approx(100.0)
