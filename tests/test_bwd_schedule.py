"""Host-only check of how the backward main kernel splits its iterations over
persistent CTAs (csrc/bwd_sched.cuh), and of the head-group grid order of the
one-CTA-per-tile launches, by brute force over many shapes: built from the same
header with the host compiler and run on the CPU."""
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
    # n, BH, causal, G, u0 (first split unit; the units before it run one CTA each)
    (16, 48, 0, 152, 0), (16, 48, 1, 152, 0),
    (16, 48, 0, 152, 456),                     # B=4 H=12 N=2048: the last 2 waves' worth split
    (64, 12, 0, 152, 608), (183, 12, 1, 152, 0),
    (64, 1, 0, 152, 0), (64, 1, 1, 152, 0),    # one head, N = 8192
    (128, 32, 0, 152, 3800), (1, 1, 0, 1, 0), (1, 1, 1, 1, 0), (2, 1, 1, 3, 0),
    (3, 1, 1, 6, 0), (8, 3, 0, 7, 0), (8, 3, 1, 7, 5), (5, 2, 1, 13, 0), (5, 2, 0, 50, 0),
    (9, 5, 1, 160, 0), (16, 2, 0, 16, 16), (40, 1, 1, 17, 3), (7, 7, 0, 49, 0),
    (7, 4, 0, 3, 24), (7, 4, 0, 5, 20), (7, 4, 0, 9, 18), (5, 3, 1, 4, 11),
]


@pytest.mark.parametrize("n,BH,causal,G,u0", CASES)
def test_schedule_covers_every_iteration_once(checker, n, BH, causal, G, u0):
    r = subprocess.run([checker, str(n), str(BH), str(causal), str(G), str(u0)], capture_output=True,
                       text=True)
    assert r.returncode == 0, r.stderr + r.stdout


GROUP_CASES = [
    # tiles, BH, group, tail
    (183, 12, 12, 0), (183, 12, 7, 0), (183, 12, 1, 0), (128, 32, 11, 0), (128, 32, 5, 0),
    (16, 48, 48, 0), (1, 1, 1, 0), (3, 5, 2, 0), (7, 9, 4, 0), (2, 3, 3, 0), (5, 7, 6, 0), (4, 4, 1, 0),
    # the last heads as one more group (causal launches run head by head)
    (183, 12, 1, 5), (183, 12, 1, 12), (183, 12, 1, 2), (128, 32, 1, 7), (7, 9, 4, 3), (5, 7, 2, 6),
    (1, 3, 1, 3), (3, 2, 1, 1),
]


@pytest.mark.parametrize("tiles,BH,group,tail", GROUP_CASES)
def test_group_order_visits_every_tile_once_group_by_group(checker, tiles, BH, group, tail):
    r = subprocess.run([checker, "group", str(tiles), str(BH), str(group), str(tail)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr + r.stdout
