"""Host-only check of how the backward main kernel spreads its work over CTAs
(csrc/bwd_sched.cuh: whole key tiles, or slices of their query tiles), and of the
head-group grid order of the one-CTA-per-tile launches, by brute force over many
shapes: built from the same header with the host compiler and run on the CPU."""
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
    # n, BH, causal, G (CTAs per wave)
    (64, 1, 0, 152), (64, 1, 1, 152),            # one head, N = 8192
    (16, 48, 0, 152), (16, 48, 1, 152),          # B=4 H=12 N=2048: a last wave of 8 key tiles
    (183, 12, 1, 152), (183, 12, 0, 152),        # one trading day, 12 heads
    (16, 10, 0, 152), (16, 11, 0, 152), (16, 14, 0, 152), (8, 20, 0, 152), (5, 31, 0, 152),
    (16, 16, 0, 152), (128, 32, 0, 152), (32, 2, 0, 152), (32, 2, 1, 152),
    (1, 1, 0, 152), (1, 1, 1, 152), (2, 1, 1, 3), (3, 1, 1, 6), (8, 3, 0, 7), (8, 3, 1, 7),
    (5, 2, 1, 13), (5, 2, 0, 50), (9, 5, 1, 160), (16, 2, 0, 16), (40, 1, 1, 17), (7, 7, 0, 49),
    (7, 4, 0, 3), (7, 4, 0, 5), (7, 4, 0, 9), (5, 3, 1, 4), (4, 7, 0, 9), (3, 2, 0, 160),
    (28, 1, 0, 50), (7, 4, 1, 50), (27, 1, 1, 40), (4, 37, 0, 152), (100, 1, 1, 152),
]


@pytest.mark.parametrize("n,BH,causal,G", CASES)
def test_slices_cover_every_tile_pair_once(checker, n, BH, causal, G):
    r = subprocess.run([checker, "slices", str(n), str(BH), str(causal), str(G)], capture_output=True,
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
