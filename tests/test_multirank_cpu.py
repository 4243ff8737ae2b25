"""The bench's multi-rank host logic on CPU: two gloo ranks (one process per
rank, as the bench runs one per GPU) agree on the slowest rank's time and on
the whole-job rate.  The attention path itself shards by sample and head with
no exchange step, so ranks run independent replicas and only these timing
reductions cross ranks."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        import bench
        got_ws, got_rank, got_local = bench.dist_env()
        bench.barrier(ws)
        ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        ms_max = bench.barrier_max(ms, ws)
        rate = bench.whole_job_tflops(2.0e12, 4, ws, ms_max)
        out.put((rank, got_ws, got_rank, got_local, ms_max, rate))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time_and_job_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ws, got_rank, local, ms_max, rate in res:
        assert (ws, got_rank, local) == (2, rank, rank)
        assert ms_max == 15.0
        # 2 ranks x 4 steps x 2e12 flops in 15 ms
        assert rate == pytest.approx(2 * 4 * 2.0e12 / 15e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.barrier_max(3.5, 1) == 3.5
    bench.barrier(1)
    assert bench.whole_job_tflops(1e12, 2, 1, 1.0) == pytest.approx(2000.0)
