"""The N > 1 path of bench.py on CPU: two gloo ranks, each with its own replica timings."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r's replica took (r + 1) x as long on one part, and less on another
        mine = {"sliding_prefill": 10.0 * (rank + 1), "global_prefill": 40.0 - rank, "decode_global": 3.0}
        got = bench.max_over_ranks(mine, dist, "cpu")
        dist.barrier()
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_of_every_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    want = {"sliding_prefill": 20.0, "global_prefill": 40.0, "decode_global": 3.0}
    assert out[0] == want and out[1] == want


def test_job_value_counts_every_replica():
    # two replicas each doing 1e12 flops per step for 10 steps in a max-over-ranks 20 ms
    assert bench.job_tflops(1e12, 10, 2, 20.0) == pytest.approx(1000.0)
    assert bench.job_tflops(1e12, 10, 1, 20.0) == pytest.approx(500.0)
    assert bench.job_tflops(1e12, 10, 2, 0.0) is None


def test_reference_arm_prints_on_rank_zero_only(capsys):
    class Args:
        steps, warmup = 1, 1
    assert bench.run_reference(Args(), rank=1, world=2) == 0
    assert capsys.readouterr().out == ""
