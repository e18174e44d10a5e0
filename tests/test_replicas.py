"""The multi-GPU path of bench.py runs independent replicas (heads shard with
no exchange step): each rank draws its own inputs, the job's time is the
slowest rank's and its throughput counts every rank's tokens.  Exercised with
two gloo processes on the CPU (no GPU, no NCCL)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r's step takes 1 + r ms, its dominant kernel 0.5 + 2 r ms
        ms, dom = bench.max_over_ranks([1.0 + rank, 0.5 + 2 * rank], dist, "cpu")
        seeds = [None] * world
        dist.all_gather_object(seeds, bench.rank_inputs_seed(7, rank))
        q.put((rank, ms, dom, bench.job_throughput(1000, world, ms), seeds))
    finally:
        dist.destroy_process_group()


def test_two_rank_replicas_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    results = sorted(q.get() for _ in range(world))
    for rank, ms, dom, value, seeds in results:
        assert ms == 2.0 and dom == 2.5            # the maxima over the two ranks
        assert value == pytest.approx(2 * 1000 / 2e-3)
        assert seeds == [7, 1007]                  # distinct inputs per replica


def test_single_process_is_unchanged():
    import bench
    assert bench.max_over_ranks([3.0, 4.0], None, "cpu") == [3.0, 4.0]
    assert bench.job_throughput(500, 1, 2.0) == pytest.approx(250000.0)


@pytest.mark.parametrize("workload", ["causal8k", "decode8k", "causal8k_bwd"])
def test_reference_arm_runs_on_rank_zero_only(workload, monkeypatch, capsys):
    import argparse
    import bench
    monkeypatch.setenv("RANK", "1")
    args = argparse.Namespace(workload=workload, steps=1, warmup=3, gpus=2, impl="reference",
                              no_cpu_baseline=True)
    fn = {"causal8k": bench.run_reference, "decode8k": bench.run_decode_reference,
          "causal8k_bwd": bench.run_backward_reference}[workload]
    assert fn(args) == 0
    assert capsys.readouterr().out == ""
