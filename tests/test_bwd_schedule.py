"""Host-only check of how the backward main kernel splits its iterations over
persistent CTAs (csrc/bwd_sched.cuh), by brute force over many shapes: built
from the same header with the host compiler and run on the CPU."""
import os
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "..", "exact_io_aware_26_gb300", "csrc")


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    exe = str(tmp_path_factory.mktemp("sched") / "sched_check")
    subprocess.run(["g++", "-O1", "-std=c++17", "-I", CSRC, os.path.join(HERE, "sched_check.cpp"),
                    "-o", exe], check=True)
    return exe


CASES = [
    # n, BH, causal, G
    (16, 48, 0, 152), (16, 48, 1, 152),        # the B=4 H=12 N=2048 workload
    (183, 12, 1, 152), (64, 1, 0, 152),        # N = 23400 causal, N = 8192 one head
    (128, 32, 0, 152), (1, 1, 0, 1), (1, 1, 1, 1), (2, 1, 1, 3),
    (3, 1, 1, 6), (8, 3, 0, 7), (8, 3, 1, 7), (5, 2, 1, 13), (5, 2, 0, 50),
    (9, 5, 1, 160), (16, 2, 0, 160), (40, 1, 1, 17), (7, 7, 0, 49),
]


@pytest.mark.parametrize("n,BH,causal,G", CASES)
def test_schedule_covers_every_iteration_once(checker, n, BH, causal, G):
    r = subprocess.run([checker, str(n), str(BH), str(causal), str(G)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr + r.stdout
