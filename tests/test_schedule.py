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


@pytest.mark.parametrize("mode", sorted(MODES))
def test_schedule_covers_every_iteration_once_and_balances(checker, mode):
    cases = [c + (MODES[mode],) for c in _cases()]
    inp = "\n".join(" ".join(map(str, c)) for c in cases) + "\n"
    r = subprocess.run([checker], input=inp, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout[-3000:]
    assert r.stdout.count("\n") == len(cases)
