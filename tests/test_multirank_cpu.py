"""The N > 1 path of bench.py on CPU: two gloo ranks (one process per GPU in a
real run) each process their own units with no data-path collective; the
reported throughput is every rank's units over the slowest rank's time, and
the reference arm prints from rank 0 only."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, ws: int, port: int, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(ws), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist
    import bench
    got_ws, got_rank = bench.init_dist("gloo")
    # rank r takes (r + 1) seconds for its 10 units: the job takes 2 s for 20 units
    value, tmax = bench.aggregate(10.0, float(rank + 1))
    slowest = bench.max_over_ranks(float(rank + 1))
    bench.barrier()
    q.put((rank, got_ws, got_rank, value, tmax, slowest))
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_weak_scaling():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got_ws, got_rank, value, tmax, slowest in results:
        assert (got_ws, got_rank) == (ws, rank)
        assert tmax == pytest.approx(2.0) and slowest == pytest.approx(2.0)
        assert value == pytest.approx(20.0 / 2.0)


def _ref_worker(rank: int, ws: int, port: int, q):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(ws), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench

    class Args:
        steps, warmup, gpus = 1, 0, ws
    called = []
    bench.oracle_prepare = lambda names: {n: None for n in names}
    bench.oracle_run = lambda preps, pairs, seconds, max_pairs=None: (called.append(1) or (1e9, 0.5, ["q@M4"]))
    line = bench.run_reference(Args())
    q.put((rank, line is not None, len(called)))


def test_reference_arm_runs_on_rank_zero_only():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_ref_worker, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert results[0] == (0, True, 1)
    assert results[1] == (1, False, 0)
