"""The bench's multi-rank logic on CPU: two gloo ranks run the same barrier,
max-over-ranks and whole-job throughput code that the GPU replicas use."""
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


def _rank_main(rank, ws, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        got_ws, got_rank, got_local = bench.dist_setup()
        bench.barrier(ws)
        mine = 10.0 + 5.0 * rank                # this rank's total milliseconds
        slowest = bench.max_over_ranks(mine, ws, "cpu")
        value = bench.whole_job_tflops(ws, 1e12, 4, slowest)
        bench.barrier(ws)
        q.put((rank, got_ws, got_rank, got_local, slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time_and_job_value():
    ws = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, got_ws, got_rank, got_local, slowest, value in res:
        assert (got_ws, got_rank, got_local) == (ws, rank, rank)
        assert slowest == 15.0                  # the max over ranks, seen by every rank
        # both ranks' work (2 x 4 steps x 1e12 flops) over the slowest rank's 15 ms
        assert value == pytest.approx(2 * 4 * 1e12 / 0.015 / 1e12)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    bench.barrier(1)
    assert bench.whole_job_tflops(1, 2e12, 10, 1000.0) == pytest.approx(20.0)


def test_reference_arm_other_ranks_do_no_work(capsys):
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        steps, warmup, gpus = 3, 3, 2

    assert bench.run_reference(Args, 2, 1) == 0
    assert capsys.readouterr().out == ""
