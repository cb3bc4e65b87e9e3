"""Pins of the Plan A redistribution oracle ("Window-Aligned Sequence
Parallelism (SeedVR2)", sections "Planner" and "Plan A redistribution")."""

import numpy as np
import pytest

import oracle
from oracle import sp
from wsa_inputs import WORKLOADS

GRIDS = [(4, 9, 16, 2, 9, 16), (7, 5, 11, 3, 2, 4), (21, 45, 80, 4, 3, 3)]


@pytest.mark.parametrize("grid", GRIDS)
@pytest.mark.parametrize("ranks", [1, 2, 3, 5])
def test_exchange_equals_single_rank_transition(grid, ranks):
    # The rows every rank ends with are exactly the destination layout's rows
    # of its windows, in destination-local order: the single-rank transition
    # restricted to that rank.
    src = oracle.make_plan(*grid, 0)
    dst = oracle.make_plan(*grid, 1)
    x = np.random.default_rng(ranks).standard_normal((src.num_tokens, 3))
    out, sched = sp.simulate(x, src, dst, ranks)
    full = oracle.transition(x[src.ids], src, dst)  # dst packed order
    pos = np.empty(src.num_tokens, dtype=np.int64)
    pos[dst.ids] = np.arange(src.num_tokens)
    for d in range(ranks):
        rows = sched["dst_rows"][d]
        assert np.array_equal(out[d], full[pos[rows]])
        assert np.array_equal(out[d], x[rows])
    assert sched["counts"].sum() == src.num_tokens


def test_split_sizes_are_rows_and_columns():
    src = oracle.make_plan(21, 45, 80, 4, 3, 3, 0)
    dst = oracle.make_plan(21, 45, 80, 4, 3, 3, 1)
    sched = sp.plan_a(src, dst, 4)
    c = sched["counts"]
    for r in range(4):
        assert c[r].sum() == sched["src_rows"][r].size   # rank r sends all its rows
        assert c[:, r].sum() == sched["dst_rows"][r].size  # and receives all its new rows


def test_segments_in_destination_local_order():
    src = oracle.make_plan(7, 5, 11, 3, 2, 4, 1)
    dst = oracle.make_plan(7, 5, 11, 3, 2, 4, 0)
    sched = sp.plan_a(src, dst, 3)
    pos = {}
    for d in range(3):
        for i, c in enumerate(sched["dst_rows"][d]):
            pos[int(c)] = i
    for r in range(3):
        sent = sched["src_rows"][r][sched["send_index"][r]]
        b = np.concatenate([[0], np.cumsum(sched["counts"][r])])
        for d in range(3):
            seg = [pos[int(c)] for c in sent[b[d]:b[d + 1]]]
            assert seg == sorted(seg)


def test_same_layout_needs_no_network():
    p = oracle.make_plan(21, 45, 80, 4, 3, 3, 0)
    sched = sp.plan_a(p, p, 4)
    assert not sched["network_exchange_required"]
    assert np.array_equal(sched["counts"], np.diag(np.diag(sched["counts"])))
    src = oracle.make_plan(21, 45, 80, 4, 3, 3, 0)
    dst = oracle.make_plan(21, 45, 80, 4, 3, 3, 1)
    assert sp.plan_a(src, dst, 4)["network_exchange_required"]
    assert not sp.plan_a(src, dst, 1)["network_exchange_required"]  # SP = 1: local permutation


def test_more_ranks_than_windows():
    # A rank with no window holds and receives nothing; the others still agree.
    src = oracle.make_plan(2, 3, 4, 1, 1, 1, 0)
    dst = oracle.make_plan(2, 3, 4, 1, 1, 1, 1)
    assert src.num_windows == 1
    x = np.arange(src.num_tokens, dtype=np.float64)[:, None]
    out, sched = sp.simulate(x, src, dst, 3)
    assert [o.shape[0] for o in out] == [src.num_tokens, 0, 0]
    assert np.array_equal(out[0][:, 0], dst.ids.astype(np.float64))


def test_owner_hand_example():
    # tiny regular windows: sizes 50,50,40,40 repeated for w 0..2 and 10,10,8,8
    # for the last w column; LPT over 2 ranks balances token counts
    p = oracle.make_plan(4, 9, 16, 2, 9, 16, 0)
    own = sp.owners(p, 2)
    n = np.diff(p.offsets)
    loads = [n[own == r].sum() for r in range(2)]
    assert sum(loads) == 576 and abs(loads[0] - loads[1]) <= n.max()
    assert own[0] == 0 and own[1] == 1  # the two largest windows (ties by id) go to ranks 0, 1
