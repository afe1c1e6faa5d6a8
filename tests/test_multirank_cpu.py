"""The N > 1 benchmark logic on CPU: two gloo ranks on 127.0.0.1.

Ranks run independent batches (sequence sharding, no data-path exchange); the only
collective is the max of the timed region and the sum of accepted tokens.  The
reference arm runs on rank 0 alone."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [5.0, 7.5][rank]                   # rank 1 is the slower one
        tok = [180.0, 200.0][rank]
        ms_max = bench.reduce_over_ranks(ms, dist, "cpu", "max")
        tok_sum = bench.reduce_over_ranks(tok, dist, "cpu", "sum")
        out[rank] = (ms_max, tok_sum, bench.step_throughput(world, ms_max))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation_takes_slowest_rank_and_total_tokens():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(2, _free_port(), out), nprocs=2, join=True,
                           start_method="spawn")
        res = dict(out)
    for r in (0, 1):
        ms_max, tok_sum, thr = res[r]
        assert ms_max == 7.5 and tok_sum == 380.0
        assert thr == pytest.approx(2 * 1000.0 / 7.5)


def test_single_rank_reduction_is_identity():
    assert bench.reduce_over_ranks(3.25, None, "cpu", "max") == 3.25
    assert bench.step_throughput(1, 4.0) == 250.0


def test_reference_arm_runs_on_rank_zero_only():
    class A:
        steps, warmup = 1, 1
    assert bench.run_reference(A(), rank=1, world=2) is None
