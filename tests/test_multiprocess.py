"""The N-GPU launch of bench.py, on CPU: world-size-2 gloo ranks.

Every call of the path runs on one GPU, so N GPUs run N independent replicas
of the decode step with no data-path collective; the only cross-rank steps
are the barrier and the max-over-ranks of the step time, and the whole-job
rate counts every rank's tokens.  These tests run those steps on two gloo
processes (no GPU), plus the reference arm's rank handling.
"""

import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        ms = 10.0 + 5.0 * rank                 # the slower rank sets the step time
        worst = bench.max_over_ranks(ms)
        dist.barrier()
        rate = bench.whole_job_rate(1000, worst, w)
        q.put((r, w, local, worst, rate))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_count_all_tokens():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, (r, w, local, worst, rate) in enumerate(res):
        assert (r, w, local) == (rank, 2, rank)
        assert worst == 15.0                   # max over ranks, on every rank
        assert rate == pytest.approx(2 * 1000 / 15e-3)


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_rate(500, 2.0, 1) == pytest.approx(250000.0)


def test_reference_arm_runs_on_rank_zero_only():
    sys.path.insert(0, ROOT)
    import argparse
    import bench
    from kv_cache_quantization_random_gb300 import workloads as WL
    w = WL.scaled(WL.get("llama8b_32k"), n_q_heads=4, n_kv_heads=1, context=300, window=16)
    args = argparse.Namespace(warmup=3, steps=2, reference_max_steps=2)
    assert bench.run_reference(args, w, 1, 2) is None
    line = bench.run_reference(args, w, 0, 2)
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle" and line["value"] > 0
