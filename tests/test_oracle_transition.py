"""Pins of the oracle's layout transition ("Window-Aligned Sequence Parallelism
(SeedVR2)", sections "Motivation" and "Plan A redistribution": with one rank a
layout change is a local permutation of rows)."""

import numpy as np
import pytest

import oracle
from wsa_inputs import WORKLOADS

SMALL = [(4, 9, 16, 2, 9, 16), (7, 5, 11, 3, 2, 4), (21, 45, 80, 4, 3, 3)]


@pytest.mark.parametrize("grid", SMALL)
def test_round_trip_identity(grid):
    reg = oracle.make_plan(*grid, 0)
    sft = oracle.make_plan(*grid, 1)
    rng = np.random.default_rng(3)
    x = rng.standard_normal((reg.num_tokens, 5)).astype(np.float32)
    y = oracle.transition(oracle.transition(x, reg, sft), sft, reg)
    assert np.array_equal(x, y)


@pytest.mark.parametrize("grid", SMALL)
def test_labels_follow_tokens(grid):
    # Rows labelled with their canonical id in the source packing must come out
    # labelled with the destination packing's ids.
    reg = oracle.make_plan(*grid, 0)
    sft = oracle.make_plan(*grid, 1)
    out = oracle.transition(reg.ids.reshape(-1, 1), reg, sft)
    assert np.array_equal(out[:, 0], sft.ids)
    back = oracle.transition(sft.ids.reshape(-1, 1), sft, reg)
    assert np.array_equal(back[:, 0], reg.ids)


@pytest.mark.parametrize("grid", SMALL)
def test_canonical_composition(grid):
    # Independent route: pack a canonical array with each plan's ids directly.
    reg = oracle.make_plan(*grid, 0)
    sft = oracle.make_plan(*grid, 1)
    rng = np.random.default_rng(5)
    canon = rng.standard_normal((reg.num_tokens, 3))
    assert np.array_equal(oracle.transition(canon[reg.ids], reg, sft), canon[sft.ids])


def test_same_layout_is_copy():
    reg = oracle.make_plan(4, 9, 16, 2, 9, 16, 0)
    x = np.arange(reg.num_tokens * 2).reshape(-1, 2)
    assert np.array_equal(oracle.transition(x, reg, reg), x)


def test_grid_mismatch_raises():
    a = oracle.make_plan(4, 9, 16, 2, 9, 16, 0)
    b = oracle.make_plan(4, 9, 17, 2, 9, 16, 1)
    with pytest.raises(ValueError):
        oracle.gather_table(a, b)


def test_gather_is_permutation_all_workloads():
    for w in WORKLOADS.values():
        a = oracle.make_plan(w.T, w.H, w.W, w.nt, w.nh, w.nw, 0)
        b = oracle.make_plan(w.T, w.H, w.W, w.nt, w.nh, w.nw, 1)
        g = oracle.gather_table(a, b)
        assert np.array_equal(np.sort(g), np.arange(a.num_tokens))
        assert not np.array_equal(g, np.arange(a.num_tokens))
