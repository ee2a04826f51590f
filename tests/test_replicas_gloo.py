"""The multi-GPU path of bench.py is replicas (no exchange in the layer):
each rank draws its own tokens, the job's time is the slowest rank's and
its rate counts every rank's tokens; only rank 0 runs the oracle arm.  The
rank logic is checked here with two gloo processes on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from workloads import CONFIGS

        cfg = CONFIGS[1]
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, world, "cpu")
        seed = bench.rank_seed(cfg, rank)
        ref = bench.run_reference(None, cfg, rank, world) if rank != 0 else "rank0"
        out.put((rank, ms, seed, ref))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_slowest_rank_and_distinct_tokens():
    world = 2
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, ms0, s0, ref0), (r1, ms1, s1, ref1) = res
    assert ms0 == ms1 == 15.0          # both ranks time the job by its slowest rank
    assert s0 != s1                    # replicas draw different tokens
    assert ref1 is None                # the oracle arm runs on rank 0 only


def test_job_rate_counts_every_rank():
    import bench
    assert bench.job_rate(1, 1000, 10.0) == 100000.0
    assert bench.job_rate(4, 1000, 10.0) == 400000.0
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
