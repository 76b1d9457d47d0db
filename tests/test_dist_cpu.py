"""The multi-rank host logic of bench.py on CPU: two gloo ranks.

With N GPUs the benchmark runs N independent replicas of the workload (the
path shards over batches, heads and sequences with no exchange).  Its only
collectives are the barrier around the timed region and the max of the
per-rank times; the reported value is the work of all ranks divided by the
slowest rank's time.  This checks that logic with world size 2 on gloo.
"""

import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    d = bench.Dist(world, backend="gloo")
    try:
        assert d.world == world and d.rank == rank
        d.barrier()
        ms = 2.0 + rank  # rank 1 is the slower one
        ms_max = d.max(ms)
        value = bench.whole_job_rate(1e12, d.world, ms_max, 1e12)
        d.barrier()
        out.put((rank, ms_max, value))
    finally:
        d.close()


def test_two_gloo_ranks_take_the_max_time_and_aggregate_the_work():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    codes = [p.exitcode for p in procs]
    for p in procs:
        if p.is_alive():
            p.kill()
    assert codes == [0, 0], codes
    res = sorted(out.get(timeout=5) for _ in range(world))
    for rank, ms_max, value in res:
        assert ms_max == pytest.approx(3.0)
        # 2 ranks x 1e12 units in 3 ms -> 666.67 (units/s / 1e12)
        assert value == pytest.approx(2e12 / 3e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    saved = {k: os.environ.pop(k, None) for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    try:
        d = bench.Dist(1)
        assert d.world == 1 and d.pg is None
        assert d.max(4.5) == 4.5
        assert bench.whole_job_rate(6e9, 1, 1.0, 1e9) == pytest.approx(6000.0)
    finally:
        for k, v in saved.items():
            if v is not None:
                os.environ[k] = v
