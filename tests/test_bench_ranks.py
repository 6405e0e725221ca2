"""The multi-GPU path of bench.py is replicas only (the op needs no exchange):
each rank times the same workload and the job reports the slowest rank's time
and the whole-job throughput.  This checks that host-side logic with two gloo
ranks on the CPU (no GPU involved)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [2.0, 3.5][rank]  # rank 1 is the slow one
        slowest = bench.max_over_ranks(ms, world, "cpu")
        out[rank] = (slowest, bench.job_tflops(1e12, world, slowest))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        res = dict(out)
    for r in range(2):
        slowest, tflops = res[r]
        assert slowest == pytest.approx(3.5)
        # 2 replicas x 1e12 FLOP in 3.5 ms
        assert tflops == pytest.approx(2 * 1e12 / 3.5e-3 / 1e12)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(4.25, 1) == 4.25
    assert bench.job_tflops(2e12, 1, 2.0) == pytest.approx(1000.0)
