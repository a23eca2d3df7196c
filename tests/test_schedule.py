"""Host-side checks of the persistent / stream-K work schedule (no GPU):
compiles tests/schedule_check.cpp against schedule.cuh with g++ and runs it
over every workload shape and a sweep of small and ragged shapes."""
import os
import subprocess

import numpy as np
import pytest

import workloads

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    exe = str(tmp_path_factory.mktemp("sched") / "schedule_check")
    subprocess.run(["g++", "-O1", "-std=c++17", "-Wall", os.path.join(HERE, "schedule_check.cpp"),
                    "-o", exe], check=True)
    return exe


def _cases():
    cases = []
    for w in workloads.WORKLOADS:
        mt, nt, kb = -(-w.M // 128), -(-w.N // 128), -(-w.K // 64)
        for sms in (152, 148, 132):
            cases.append((mt, nt, kb, sms, 8, int(w.M <= 128)))
            cases.append((-(-w.M // 256), nt, kb, sms // 2, 8, 0))   # CTA-pair kernel
    rng = np.random.Generator(np.random.PCG64(3))
    for _ in range(400):
        cases.append((int(rng.integers(1, 40)), int(rng.integers(1, 40)), int(rng.integers(1, 30)),
                      int(rng.integers(1, 200)), int(rng.integers(1, 10)), int(rng.integers(0, 2))))
    cases += [(1, 1, 1, 152, 8, 1), (1, 1, 200, 152, 8, 0), (1, 152, 3, 152, 8, 1),
              (2, 152, 5, 152, 8, 0), (1, 153, 7, 152, 1, 1), (64, 231, 128, 152, 8, 0),
              # the forced-schedule GPU parity shape (M=1300, N=2000; BF16 and FP8 k-blocks)
              (11, 16, 33, 152, 4, 0), (6, 16, 33, 76, 4, 0), (11, 16, 17, 152, 4, 0),
              (6, 16, 17, 76, 4, 0)]
    return cases


MODES = {"auto": 0, "dp": 1, "split": 2, "sk": 3, "sk-tail": 4}
WIDE_MODES = {"auto": 10, "dp": 11, "sk": 13, "sk-tail": 14, "sk-aligned": 15}


@pytest.mark.parametrize("mode", sorted(MODES))
def test_schedule_covers_every_iteration_once_and_balances(checker, mode):
    cases = [c + (MODES[mode],) for c in _cases()]
    inp = "\n".join(" ".join(map(str, c)) for c in cases) + "\n"
    r = subprocess.run([checker], input=inp, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout[-3000:]
    assert r.stdout.count("\n") == len(cases)


def _wide_cases():
    """The wide down-projection planner: tiles of 256 rows x 512 output
    columns of every workload's down-projection (out [M, K] = Y [M, N] x
    W3 [N, K]: k-blocks over N), on 76, 74 and 66 pairs, and random shapes."""
    cases = []
    for w in workloads.WORKLOADS:
        mt, nt, kb = -(-w.M // 256), -(-w.K // 512), -(-w.N // 64)
        for pairs in (76, 74, 66):
            cases.append((mt, nt, kb, pairs, 8, 0))
    rng = np.random.Generator(np.random.PCG64(4))
    for _ in range(400):
        cases.append((int(rng.integers(1, 40)), int(rng.integers(1, 20)), int(rng.integers(1, 500)),
                      int(rng.integers(1, 100)), 8, 0))
    cases += [(8, 3, 140, 76, 8, 0), (6, 4, 33, 76, 8, 0), (12, 7, 76, 76, 8, 0),
              (12, 7, 32, 76, 8, 0), (2, 7, 296, 76, 8, 0), (1, 1, 1, 76, 8, 0)]
    return cases


@pytest.mark.parametrize("mode", sorted(WIDE_MODES))
def test_wide_down_schedule_covers_every_iteration_once(checker, mode):
    """Coverage, k order and slot checks of plan_down_wide's plans; its
    aligned form (each tile cut into equal K ranges) gives every pair one
    unit."""
    cases = [c + (WIDE_MODES[mode],) for c in _wide_cases()]
    inp = "\n".join(" ".join(map(str, c)) for c in cases) + "\n"
    r = subprocess.run([checker], input=inp, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout[-3000:]
    assert r.stdout.count("\n") == len(cases)


def test_wide_down_plans_of_the_workload_shapes(checker):
    """The forms of the wide planner at the down-projection shapes on 76
    pairs: the aligned split cuts the 1.5B shape's 24 tiles in three K
    ranges on 72 pairs and the 7B M=512 shape's 14 tiles in five on 70;
    whole tiles (the automatic form) keep one pair per tile."""
    want = [("1", 15, 72, 0), ("5", 15, 70, 0), ("7", 10, 76, 224), ("11", 10, 76, 512)]
    for label, mode, grid, dp in want:
        w = workloads.BY_LABEL[label]
        case = (-(-w.M // 256), -(-w.K // 512), -(-w.N // 64), 76, 8, 0, mode)
        r = subprocess.run([checker], input=" ".join(map(str, case)) + "\n", capture_output=True,
                           text=True)
        assert r.returncode == 0, r.stdout
        assert "grid=%d dp=%d " % (grid, dp) in r.stdout, (label, r.stdout)


def test_stream_k_grid_search(checker):
    """plan_stream_k_grid: coverage and k order on random few-tile shapes,
    and the 1.5B down-projection shape (48 tiles of 256 x 256, 140 k-blocks,
    76 pairs) lands on 72 pairs (two per tile)."""
    rng = np.random.Generator(np.random.PCG64(5))
    cases = [(int(rng.integers(1, 10)), int(rng.integers(1, 10)), int(rng.integers(1, 400)),
              int(rng.integers(2, 100)), 8, 0, 20) for _ in range(300)]
    cases.append((8, 6, 140, 76, 8, 0, 20))
    inp = "\n".join(" ".join(map(str, c)) for c in cases) + "\n"
    r = subprocess.run([checker], input=inp, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout[-3000:]
    last = r.stdout.strip().splitlines()[-1]
    assert "grid=72 " in last and "max_contrib=2" in last, last


def test_decode_splits(checker):
    """The decode down-projection kernel's K ranges per tile: range checks on
    random shapes, and with the cluster capacities measured on GB300 the
    choices at the workloads' decode shapes (tiles of 128 output columns,
    k-blocks over the intermediate size): for long weight streams the
    smallest split that puts two thirds of the 152 SMs to work in one wave
    (7B: 28 tiles in 4, 112 CTAs; 72B: 64 in 2; 32B: 40 in 3), for short
    ranges the most CTAs in one wave (1.5B M=16: 12 tiles in 10; 0.5B: 7 in
    16), whole tiles for 152 tiles or more."""
    rng = np.random.Generator(np.random.PCG64(7))
    cases = [(1, int(rng.integers(1, 400)), int(rng.integers(1, 600)), 152, 8,
              int(rng.integers(0, 2)), 30) for _ in range(500)]
    inp = "\n".join(" ".join(map(str, c)) for c in cases) + "\n"
    r = subprocess.run([checker], input=inp, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout[-3000:]
    assert r.stdout.count("\n") == len(cases)
    want = {"3": 4, "10": 2, "8": 3, "0": 16}
    for label, j in want.items():
        w = workloads.BY_LABEL[label]
        case = (1, -(-w.K // 128), -(-w.N // 64), 152, 8, 1, 30)
        r = subprocess.run([checker], input=" ".join(map(str, case)) + "\n", capture_output=True,
                           text=True)
        assert r.returncode == 0 and "splits=%d\n" % j in r.stdout, (label, r.stdout)
    for case, j in [((1, 12, 140, 152, 8, 1, 30), 10), ((1, 152, 296, 152, 8, 1, 30), 1),
                    ((1, 7, 3, 152, 8, 1, 30), 1)]:
        r = subprocess.run([checker], input=" ".join(map(str, case)) + "\n", capture_output=True,
                           text=True)
        assert r.returncode == 0 and "splits=%d\n" % j in r.stdout, (case, r.stdout)
