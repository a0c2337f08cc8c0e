"""The multi-rank path of the benchmark on CPU (gloo, world size 2): the job
reports the maximum of the ranks' timed-region lengths and whole-job
throughput = ranks x per-rank work / that time (replicas, weak scaling)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [12.5, 20.0][rank]
    ms = bench.reduce_step_time(local_ms, world)
    results[rank] = (ms, bench.job_tflops(bench.STEP_FLOPS, ms / 10, world))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_reduction_gloo():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        import bench
        for r in range(2):
            ms, tf = results[r]
            assert ms == 20.0
            assert tf == pytest.approx(2 * bench.STEP_FLOPS / (2.0e-3) / 1e12)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_step_time(3.25, 1) == 3.25
    assert bench.job_tflops(1e12, 1.0, 1) == pytest.approx(1000.0)
