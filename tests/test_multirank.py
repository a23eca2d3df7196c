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


def _column_worker(rank, world, port, q, M, N, K):
    """One rank of the column-parallel split, on the CPU: its slice of W1
    and W2's columns through the oracle, gathered on rank 0."""
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import bench
    import oracle
    import workloads
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        A, W1, W2 = workloads.random_case(M, N, K, seed=31)
        c0, c1 = bench.column_slice(N, world, rank)
        Yr = oracle.swiglu_up(A, W1[:, c0:c1].copy(), W2[:, c0:c1].copy())["Y"]
        parts = [None] * world
        dist.all_gather_object(parts, (c0, c1, Yr))
        if rank == 0:
            q.put(parts)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("N", [520, 1000])
def test_column_split_over_two_gloo_ranks_reassembles_the_whole_result(N, oracle_mod):
    """Two ranks each compute Y[:, slice] from their slice of the weights;
    the slices tile [0, N) and, put side by side, equal the oracle's whole Y
    bit for bit (columns of Y are independent, no collective is needed)."""
    import numpy as np

    import workloads
    world, port = 2, _free_port()
    M, K = 9, 72
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_column_worker, args=(r, world, port, q, M, N, K))
             for r in range(world)]
    for p in procs:
        p.start()
    parts = q.get(timeout=120)
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert parts[0][0] == 0 and parts[-1][1] == N
    for (a0, a1, _), (b0, b1, _) in zip(parts, parts[1:]):
        assert a1 == b0
    for c0, c1, Yr in parts:
        assert (c1 - c0) % 8 == 0 and c1 > c0 and Yr.shape == (M, c1 - c0)
    whole = oracle_mod.swiglu_up(*workloads.random_case(M, N, K, seed=31))["Y"]
    assert np.array_equal(np.concatenate([Yr for _, _, Yr in parts], axis=1), whole)


def test_column_slice_arithmetic():
    import bench
    for N in (8, 136, 520, 4864, 8960, 18944, 27648, 29568):
        tiles = -(-N // 128)
        for world in (1, 2, 3, 4, 8):
            if world > tiles:
                with pytest.raises(ValueError):
                    bench.column_slice(N, world, 0)
                continue
            s = [bench.column_slice(N, world, r) for r in range(world)]
            assert s[0][0] == 0 and s[-1][1] == N
            assert all(a[1] == b[0] for a, b in zip(s, s[1:]))
            widths = [c1 - c0 for c0, c1 in s]
            assert all(wd > 0 and wd % 8 == 0 for wd in widths)
            assert all(c0 % 128 == 0 for c0, _ in s)       # slices start on tile boundaries
            assert max(widths) - min(widths) <= 128          # whole tiles dealt evenly


def test_gpus_flag_starts_ranks_or_must_match_world(monkeypatch):
    """`--gpus N` outside torchrun re-launches under torch.distributed.run
    with N processes on 127.0.0.1; under torchrun it must equal WORLD_SIZE."""
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    seen = []
    monkeypatch.setattr(bench.subprocess, "call", lambda cmd: seen.append(cmd) or 0)
    assert bench.main(["--gpus", "4", "--steps", "5", "--warmup", "3"]) == 0
    cmd = seen[0]
    assert cmd[1:4] == ["-m", "torch.distributed.run", "--nnodes=1"]
    assert "--nproc-per-node=4" in cmd and "127.0.0.1" in cmd
    assert cmd[-6:] == ["--gpus", "4", "--steps", "5", "--warmup", "3"]
    monkeypatch.setenv("WORLD_SIZE", "2")
    with pytest.raises(SystemExit):
        bench.main(["--gpus", "4"])
