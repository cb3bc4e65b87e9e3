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


# ---- Plan B (halo exchange) evaluation counts -------------------------------

def _brute_plan_b(reg, sft, ranks):
    # independent restatement: for each shifted window, count rows by holder
    own = sp.owners(reg, ranks)
    holder = {}
    for w in range(reg.num_windows):
        for c in reg.ids[reg.offsets[w]:reg.offsets[w + 1]]:
            holder[int(c)] = int(own[w])
    moved, comp = 0, []
    for w in range(sft.num_windows):
        rows = [int(c) for c in sft.ids[sft.offsets[w]:sft.offsets[w + 1]]]
        counts = [sum(1 for c in rows if holder[c] == r) for r in range(ranks)]
        best = max(range(ranks), key=lambda r: (counts[r], -r))
        comp.append(best)
        moved += len(rows) - counts[best]
    return moved, comp


@pytest.mark.parametrize("grid", GRIDS)
@pytest.mark.parametrize("ranks", [1, 2, 3, 5])
def test_plan_b_against_brute_force(grid, ranks):
    reg, sft = oracle.make_plan(*grid, 0), oracle.make_plan(*grid, 1)
    got = sp.plan_b(reg, sft, ranks)
    moved, comp = _brute_plan_b(reg, sft, ranks)
    assert list(got["owner"]) == comp
    assert got["halo_in"].sum() == moved == got["halo_out"].sum()
    assert got["tokens"].sum() == reg.num_tokens
    assert got["work"].sum() == pytest.approx(float(np.sum(np.diff(sft.offsets).astype(np.float64) ** 2)))


def test_plan_b_one_rank_and_one_window_move_nothing():
    reg, sft = oracle.make_plan(21, 45, 80, 4, 3, 3, 0), oracle.make_plan(21, 45, 80, 4, 3, 3, 1)
    assert sp.plan_b(reg, sft, 1)["halo_in"].sum() == 0
    g = (2, 3, 4, 1, 1, 1)  # a single window in both layouts
    assert sp.plan_b(oracle.make_plan(*g, 0), oracle.make_plan(*g, 1), 4)["halo_in"].sum() == 0


def test_plan_b_hand_example():
    # (T, H, W) = (1, 45, 80) at scale 1 with nw = 4: windows 45 x 20 columns.
    # Regular column cuts 0,20,40,60,80 -> LPT over 2 ranks (all 900 tokens,
    # ties to the lower rank): r0, r1, r0, r1.  Shifted cuts move by 10 on w
    # only (H equals its window): 0,10,30,50,70,80.  Windows [10,30), [30,50)
    # and [50,70) straddle two owners with 450 rows each -> computed by r0
    # (tie), 450 halo rows each; [0,10) is r0's, [70,80) is r1's.
    reg, sft = oracle.make_plan(1, 45, 80, 1, 1, 4, 0), oracle.make_plan(1, 45, 80, 1, 1, 4, 1)
    assert [b[4:] for b in sft.boxes] == [(0, 10), (10, 30), (30, 50), (50, 70), (70, 80)]
    got = sp.plan_b(reg, sft, 2)
    assert list(got["owner"]) == [0, 0, 0, 0, 1]
    assert list(got["halo_in"]) == [1350, 0] and list(got["halo_out"]) == [0, 1350]
    assert list(got["tokens"]) == [3150, 450]
    assert list(got["work"]) == [450.0 ** 2 + 3 * 900.0 ** 2, 450.0 ** 2]
    # Plan A: shifted LPT sizes 450,900,900,900,450 -> owners r1,r0,r1,r0,r1;
    # columns 0-9, 20-29, 40-49 and 60-69 change rank: 4 x 450 rows.
    assert list(sp.owners(sft, 2)) == [1, 0, 1, 0, 1]
    assert sp.plan_a_rows_moved(reg, sft, 2) == 1800
