"""bench.py's multi-process path on CPU: two gloo ranks check the timing
barrier, the max over ranks and the whole-job aggregation, and that the
reference arm does no work on ranks other than 0."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        elapsed = 1.0 + rank                       # rank 1 is the slow one
        mx = bench.max_over_ranks(elapsed, world)
        value = bench.aggregate_value(1e12, 10, world, mx)
        q.put((rank, mx, value, bench.dist_env()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_bench():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, mx, value, env in res:
        assert mx == 2.0                           # max over ranks, on every rank
        assert value == pytest.approx(1e12 * 10 * 2 / 2.0 / 1e12)   # all ranks' FLOPs / slowest time
        assert env == (2, rank, rank)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    import bench
    import workloads
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps, warmup = 5, 3

    called = []
    monkeypatch.setattr(bench, "oracle_sample_rate", lambda *a, **k: called.append(1) or (1.0, 1.0))
    assert bench.run_reference(Args(), workloads.BY_LABEL["0"]) == 0
    assert not called
