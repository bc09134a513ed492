"""Host logic of bench.py's replica mode, on CPU with two gloo ranks (no GPU).

The layer runs as independent replicas, one per GPU (no data-path collective);
the bench times every replica, takes the slowest as the job's time and reports
the tokens of all replicas over that time. These tests run the rank aggregation
over a real two-process gloo group and check the whole-job arithmetic and that
the reference arm's non-zero ranks do no work and print nothing."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, queue):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank r's step, forward and end-to-end times (ms): each entry is slowest on a different rank
        got = bench.max_over_ranks([10.0 + rank, 7.0 - rank, 3.5])
        queue.put((rank, got, bench.dist_env()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = {}
    for _ in procs:
        rank, got, env = queue.get(timeout=120)
        results[rank] = (got, env)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in (0, 1):
        got, env = results[rank]
        assert got == [11.0, 7.0, 3.5]          # every rank sees the slowest replica's times
        assert env == (2, rank, 0)              # world size, rank, local rank from the environment


def test_max_over_ranks_alone_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2]) == [1.5, 2.0]


def test_job_throughput_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench
    # 2 replicas x 4096 tokens x 10 steps over the slowest replica's 100 ms
    assert bench.job_tokens_per_s(2, 4096, 10, 100.0) == pytest.approx(819200.0)
    assert bench.job_tokens_per_s(1, 4096, 10, 100.0) == pytest.approx(409600.0)


def test_reference_arm_other_ranks_do_nothing(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    import workloads as WL
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")

    class Args:
        steps, warmup, gpus = 1, 1, 2
    called = []
    monkeypatch.setattr(bench, "oracle_step", lambda *a, **k: called.append(1) or 1.0)
    assert bench.run_reference(Args(), WL.TINY) is None
    assert called == [] and capsys.readouterr().out == ""
