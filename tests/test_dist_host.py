"""The benchmark's multi-rank host logic on CPU: two gloo ranks (no GPU).

Each rank runs its own replica of the step (the path does not shard across GPUs); the
job's time is the slowest rank's and its throughput counts every rank's units. These
are the helpers bench.py uses for that, run here in two processes over gloo.
"""

import multiprocessing as mp
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, q):
    try:
        os.environ.update(RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                          MASTER_PORT=str(port))
        import torch
        import torch.distributed as dist

        import bench
        r, world, local = bench.dist_setup(2, backend="gloo")
        cpu = torch.device("cpu")
        bench.barrier(world)
        slowest = bench.max_over_ranks([1.5, 4.0][r], world, cpu)
        rate = bench.job_rate(1000, [2.0, 4.0][r], world, cpu)  # 1000 units a rank
        pre = {"T": 512, "ms_per_step": [0.3, 0.5][r], "e2e": [1.0e6, 2.0e6][r], "value": 0.0}
        bench.reduce_prefill(pre, world, cpu)
        seeds = [bench.layer_seed(r, i) for i in range(64)]
        q.put((r, world, local, slowest, rate, pre, seeds))
        dist.destroy_process_group()
    except Exception as e:  # reported to the parent
        q.put((rank, "error", repr(e)))


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    try:
        for _ in range(2):
            item = q.get(timeout=120)
            assert item[1] != "error", item
            res[item[0]] = item
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert sorted(res) == [0, 1]
    for r in (0, 1):
        _, world, local, slowest, rate, pre, _ = res[r]
        assert world == 2 and local == r
        assert slowest == 4.0                       # the slowest rank's time, on both ranks
        assert rate == pytest.approx(2 * 1000 / 4.0)  # every rank's units over the slowest time
        assert pre["ms_per_step"] == 0.5
        assert pre["value"] == pytest.approx(2 * 512 / 0.5e-3, rel=1e-6)
        # e2e: 512 tokens at 1e6 and 2e6 tokens/s -> the slower rank's step time, both ranks' tokens
        assert pre["e2e"] == pytest.approx(2 * 512 / (512 / 1.0e6), rel=1e-6)
    assert not set(res[0][6]) & set(res[1][6])      # the ranks draw different layers
