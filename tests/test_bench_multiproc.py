"""The multi-GPU path of bench.py is replicas: each rank runs the same step on
its own GPU, the job's time is the slowest rank's (all-reduce MAX after a
barrier), and the value is the units all ranks processed over that time.  The
rank reduction and the throughput are checked here with two gloo ranks on the
CPU (no GPU, no NCCL)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist

    r, w, local = bench.setup_distributed(world, backend="gloo")
    assert (r, w, local) == (rank, world, rank)
    ms = bench.job_time(times[rank], w)
    out[rank] = (ms, bench.job_value(100.0, w, ms))
    dist.destroy_process_group()


def test_replica_job_time_is_the_slowest_rank_and_value_counts_all_ranks():
    world, times = 2, [3.0, 5.0]
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_rank, args=(r, world, PORT, times, out))
                 for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        ms, value = res[r]
        assert ms == 5.0  # every rank sees the slowest rank's time
        assert value == pytest.approx(2 * 100.0 / 5e-3)


def test_single_process_needs_no_collective():
    import bench

    assert bench.job_time(4.0, 1) == 4.0
    assert bench.job_value(10.0, 1, 2.0) == pytest.approx(5000.0)


PORT = _free_port()


def test_gate_up_traffic_is_null_once_the_sources_change(monkeypatch):
    """The recorded DRAM traffic of the gate_up GEMM belongs to the sources it was
    captured on: bench.py reports it only while their hash matches."""
    import bench

    assert bench.gate_up_traffic() in (bench.GATE_UP_TRAFFIC["bytes"], None)
    monkeypatch.setitem(bench.GATE_UP_TRAFFIC, "sources_sha256", "0" * 64)
    assert bench.gate_up_traffic() is None


def test_job_value_counts_all_ranks_units():
    import bench

    assert bench.job_value(1e12, 4, 2.0) == 4 * 1e12 / 2e-3
    assert bench.job_time(3.0, 1) == 3.0
