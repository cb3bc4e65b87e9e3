"""Pins of the oracle's window geometry ("Window-Aligned Sequence Parallelism
(SeedVR2)", section "Window layouts")."""

import json
import math
import os
import random

import pytest

import oracle
from oracle.geometry import axis_intervals, window_size

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# Closed forms worked out by hand for each workload grid.  Where H*W = 3600*k^2
# the scale is exactly 1/k, so round(H*scale) and round(W*scale) are exact.
@pytest.mark.parametrize("grid,expect", [
    # H*W = 144 -> scale = 5: round(45) = 45, round(80) = 80; 45/9 = 5, 80/16 = 5; ceil(4/2) = 2
    ((4, 9, 16, 2, 9, 16), (2, 5, 5)),
    # H*W = 3600 -> scale = 1: ceil(45/3) = 15, ceil(80/3) = 27, ceil(21/4) = 6
    ((21, 45, 80, 4, 3, 3), (6, 15, 27)),
    # scale = sqrt(3600/8160) = 0.6642..: 68*scale = 45.17 -> 45, 120*scale = 79.70 -> 80
    ((21, 68, 120, 4, 3, 3), (6, 15, 27)),
    # temporal cap: ceil(min(31, 30)/4) = ceil(7.5) = 8
    ((31, 45, 80, 4, 3, 3), (8, 15, 27)),
    # H*W = 14400 -> scale = 1/2 exactly: 45, 80
    ((21, 90, 160, 4, 3, 3), (6, 15, 27)),
])
def test_window_size_closed_forms(grid, expect):
    assert window_size(*grid) == expect


def test_scale_irrational_hand_values():
    # 1080p-scale grid: check the two products against hand arithmetic.
    s = math.sqrt(3600 / (68 * 120))
    assert 45.16 < 68 * s < 45.17 and 79.70 < 120 * s < 79.71


def test_round_half_even_reading():
    # H*W = 14400 gives scale 1/2 exactly; H = 45 makes H*scale = 22.5, a tie.
    # Python's round (half-to-even) gives 22; C's round() would give 23.
    assert window_size(1, 45, 320, 1, 1, 1) == (1, 22, 160)
    # 225 * 0.5 = 112.5 -> 112; 9 * 0.5 = 4.5 -> 4; 75 * 0.5 = 37.5 -> 38
    assert window_size(1, 225, 64, 1, 1, 1) == (1, 112, 32)
    assert window_size(1, 9, 1600, 1, 1, 1) == (1, 4, 800)
    assert window_size(1, 75, 192, 1, 1, 1) == (1, 38, 96)


def test_temporal_cap_only_limits_size():
    # T = 31: window size 8 from min(T, 30) = 30, yet the cuts tile all 31 frames.
    assert axis_intervals(31, 8, False) == [(0, 8), (8, 16), (16, 24), (24, 31)]


@pytest.mark.parametrize("bad", [
    (0, 9, 16, 2, 9, 16), (4, 0, 16, 2, 9, 16), (4, 9, -1, 2, 9, 16),
    (4, 9, 16, 0, 9, 16), (4, 9, 16, 2, 0, 16), (4, 9, 16, 2, 9, 0),
])
def test_invalid_inputs_raise(bad):
    with pytest.raises(ValueError):
        window_size(*bad)


def test_zero_window_raises():
    # Extreme aspect ratio: H = 1, W = 100000 -> scale ~ 0.19, round(0.19) = 0 -> wh = 0.
    with pytest.raises(ValueError):
        window_size(1, 1, 100000, 1, 1, 1)


def test_hand_cut_lists():
    g = json.load(open(os.path.join(GOLDEN, "tiny_worked_example.json")))
    def cuts(iv):
        return [iv[0][0]] + [b for (_, b) in iv]
    assert cuts(axis_intervals(4, 2, False)) == g["regular"]["t_cuts"]
    assert cuts(axis_intervals(9, 5, False)) == g["regular"]["h_cuts"]
    assert cuts(axis_intervals(16, 5, False)) == g["regular"]["w_cuts"]
    assert cuts(axis_intervals(4, 2, True)) == g["shifted"]["t_cuts"]
    assert cuts(axis_intervals(9, 5, True)) == g["shifted"]["h_cuts"]
    assert cuts(axis_intervals(16, 5, True)) == g["shifted"]["w_cuts"]


def test_degenerate_axes():
    # w >= size: a single window, shifted or not (no interior cut to move).
    assert axis_intervals(5, 5, True) == [(0, 5)]
    assert axis_intervals(4, 8, True) == [(0, 4)]
    # w == 1: floor(1/2) = 0, the shifted layout equals the regular one (empty
    # first interval dropped).
    assert axis_intervals(3, 1, True) == [(0, 1), (1, 2), (2, 3)]
    # w == 2, odd size: shifted cuts at 1, 3, clipped end
    assert axis_intervals(5, 2, True) == [(0, 1), (1, 3), (3, 5)]


def test_interval_properties_random():
    rng = random.Random(7)
    for _ in range(2000):
        size = rng.randint(1, 200)
        w = rng.randint(1, 60)
        for shifted in (False, True):
            iv = axis_intervals(size, w, shifted)
            assert iv[0][0] == 0 and iv[-1][1] == size
            assert all(b > a for a, b in iv)
            assert all(iv[i][1] == iv[i + 1][0] for i in range(len(iv) - 1))
            lens = [b - a for a, b in iv]
            if not shifted or size <= w:
                assert all(n == w for n in lens[:-1]) and lens[-1] <= w
                assert len(iv) == -(-size // w)
            else:
                # first window is half a window (or absent when w // 2 == 0),
                # interior windows are full, the last is clipped.
                if w // 2 > 0:
                    assert lens[0] == min(w // 2, size)
                    inner = lens[1:-1]
                else:
                    inner = lens[:-1]
                assert all(n == w for n in inner) and 0 < lens[-1] <= w


def test_enumeration_order_w_outermost():
    ws = oracle.windows(4, 9, 16, 2, 5, 5, False)
    # t varies fastest, then h, then w
    assert [w[0] for w in ws[:2]] == [0, 2]
    assert ws[2][2] == 5 and ws[2][0] == 0
    assert ws[4][4] == 5 and ws[4][2] == 0
