"""The library's Plan A host planner (wsa_sp_owners, wsa_sp_local_rows,
wsa_sp_plan_a; no GPU) against the oracle ("Window-Aligned Sequence
Parallelism (SeedVR2)", sections "Planner" and "Plan A redistribution").
Integer tables: bit-exact."""

import numpy as np
import pytest

import oracle
from oracle import sp as osp
from wsa_inputs import WORKLOADS

GRIDS = {
    "tiny": (4, 9, 16, 2, 9, 16),
    "odd": (7, 5, 11, 3, 2, 4),
    "720p": (21, 45, 80, 4, 3, 3),
    "1080p": (21, 68, 120, 4, 3, 3),
}


@pytest.fixture(scope="module")
def sp():
    import __graft_entry__
    __graft_entry__.build()
    import shifted_window_attention_gb300.sp as m
    return m


@pytest.mark.parametrize("name", list(GRIDS))
@pytest.mark.parametrize("ranks", [1, 2, 3, 8])
@pytest.mark.parametrize("layouts", [(0, 1), (1, 0), (1, 1)])
def test_plan_a_matches_oracle(sp, name, ranks, layouts):
    grid = GRIDS[name]
    src, dst = oracle.make_plan(*grid, layouts[0]), oracle.make_plan(*grid, layouts[1])
    ref = osp.plan_a(src, dst, ranks)
    assert np.array_equal(sp.owners(*grid, layouts[0], ranks), osp.owners(src, ranks))
    for r in range(ranks):
        pa = sp.PlanA(*grid, *layouts, ranks, r)
        assert np.array_equal(pa.counts, ref["counts"])
        assert pa.input_split_sizes == list(ref["counts"][r])
        assert pa.output_split_sizes == list(ref["counts"][:, r])
        assert np.array_equal(pa.send_index, ref["send_index"][r])
        assert np.array_equal(pa.recv_index, ref["recv_index"][r])
        assert pa.network_exchange_required == ref["network_exchange_required"]
        assert np.array_equal(sp.local_rows(*grid, layouts[0], ranks, r), ref["src_rows"][r])


def test_host_exchange_reproduces_destination_rows(sp):
    # Run the schedule on the host (index arithmetic only): every rank ends
    # with exactly its destination rows.
    grid, R = GRIDS["720p"], 4
    x = np.arange(75600, dtype=np.int64)
    plans = [sp.PlanA(*grid, 0, 1, R, r) for r in range(R)]
    local = [x[sp.local_rows(*grid, 0, R, r)] for r in range(R)]
    sends = [local[r][plans[r].send_index] for r in range(R)]
    bounds = [np.concatenate([[0], np.cumsum(p.input_split_sizes)]) for p in plans]
    for d in range(R):
        recv = np.concatenate([sends[r][bounds[r][d]:bounds[r][d + 1]] for r in range(R)])
        assert np.array_equal(recv[plans[d].recv_index], sp.local_rows(*grid, 1, R, d))


def test_same_layout_is_local(sp):
    grid = GRIDS["720p"]
    for r in range(3):
        pa = sp.PlanA(*grid, 1, 1, 3, r)
        assert not pa.network_exchange_required
        assert pa.input_split_sizes[r] == pa.n_send and sum(pa.input_split_sizes) == pa.n_send
        # the composed fast-path index is the identity: nothing moves
        assert np.array_equal(pa.send_index[pa.recv_index], np.arange(pa.n_send))


def test_more_ranks_than_windows(sp):
    grid = (2, 3, 4, 1, 1, 1)  # one window in either layout
    plans = [sp.PlanA(*grid, 0, 1, 3, r) for r in range(3)]
    assert [p.n_send for p in plans] == [24, 0, 0] and [p.n_recv for p in plans] == [24, 0, 0]
    assert not plans[1].network_exchange_required


def test_errors(sp):
    import ctypes
    from shifted_window_attention_gb300 import WsaError
    with pytest.raises(WsaError, match="INVALID_ARG"):
        sp.PlanA(*GRIDS["tiny"], 0, 1, 0, 0)
    with pytest.raises(WsaError, match="INVALID_ARG"):
        sp.PlanA(*GRIDS["tiny"], 0, 1, 2, 2)
    with pytest.raises(WsaError, match="INVALID_ARG"):
        sp.PlanA(*GRIDS["tiny"], 0, 7, 2, 0)
    with pytest.raises(WsaError, match="INVALID_ARG"):
        sp.owners(0, 9, 16, 2, 9, 16, 0, 2)
    lib = sp.lib
    n_send, n_recv, cross = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    small = (ctypes.c_int * 3)()
    st = lib.wsa_sp_plan_a(*GRIDS["tiny"], 0, 1, 30, 2, 0, None, small, 3, None, 0, None, 0, ctypes.byref(n_send),
                           ctypes.byref(n_recv), ctypes.byref(cross))
    assert st == -1 and n_send.value > 3
    n = ctypes.c_int()
    assert lib.wsa_sp_local_rows(*GRIDS["tiny"], 0, 30, 2, 0, small, 3, ctypes.byref(n)) == -1
    assert lib.wsa_gather_rows(None, 0, None, None, 0, 8, 0, None) == 0   # rows == 0: no-op
    assert lib.wsa_gather_rows(None, 4, None, None, 4, 8, 0, None) == -1  # null pointers
    assert lib.wsa_gather_rows(None, 4, None, None, 4, 0, 0, None) == -1  # channels


@pytest.mark.parametrize("name", list(GRIDS))
@pytest.mark.parametrize("ranks", [1, 2, 3, 8])
def test_plan_b_matches_oracle(sp, name, ranks):
    grid = GRIDS[name]
    ref = osp.plan_b(oracle.make_plan(*grid, 0), oracle.make_plan(*grid, 1), ranks)
    got = sp.plan_b(*grid, ranks)
    assert np.array_equal(got["window_rank"], ref["owner"])
    for k in ("halo_in", "halo_out", "tokens"):
        assert np.array_equal(got[k], ref[k]), k
    assert np.array_equal(got["work"], ref["work"])


def test_crossover_hand_grid(sp):
    # the hand-worked grid of the oracle pin: Plan A moves 1800 rows at each of
    # the two boundaries, Plan B 1350 halo rows in and 1350 outputs back.
    c = sp.crossover(1, 45, 80, 1, 1, 4, 2, channels=3072)
    row = 3072 * 2
    assert c["plan_a_bytes"] == 2 * 1800 * row
    assert c["plan_b_bytes"] == 2 * 1350 * row
    assert c["plan_b_max_rank_bytes"] == 2 * 1350 * row
    assert c["plan_b_shifted_imbalance"] > c["plan_a_shifted_imbalance"]


def test_plan_b_errors(sp):
    import ctypes
    from shifted_window_attention_gb300 import WsaError
    with pytest.raises(WsaError, match="INVALID_ARG"):
        sp.plan_b(*GRIDS["tiny"], 0)
    n = ctypes.c_int()
    small = (ctypes.c_int * 2)()
    assert sp.lib.wsa_sp_plan_b(*GRIDS["tiny"], 30, 2, small, 2, ctypes.byref(n), None, None, None, None) == -1
    assert n.value == 36


@pytest.mark.parametrize("name", list(GRIDS))
@pytest.mark.parametrize("layouts", [(0, 1), (1, 1)])
def test_local_index_is_the_composed_fast_path(sp, name, layouts):
    # one rank (and any boundary where no row changes rank): the planner's
    # local_index equals send_index[recv_index] of the oracle's schedule
    grid = GRIDS[name]
    src, dst = oracle.make_plan(*grid, layouts[0]), oracle.make_plan(*grid, layouts[1])
    ref = osp.plan_a(src, dst, 1)
    pa = sp.PlanA(*grid, *layouts, 1, 0)
    assert not pa.network_exchange_required
    assert np.array_equal(pa.local_index, ref["send_index"][0][ref["recv_index"][0]])
    # with ranks that exchange rows there is no fast-path table
    assert sp.PlanA(*grid, 0, 1, 3, 1).local_index.size == 0


@pytest.mark.parametrize("name", ["tiny", "odd", "720p"])
@pytest.mark.parametrize("ranks", [1, 2, 4, 8])
def test_crossover_figures_from_the_oracle(sp, name, ranks):
    # every byte and imbalance figure recomputed from the oracle's Plan A
    # matrices, LPT owners and Plan B counts
    grid = GRIDS[name]
    reg, sft = oracle.make_plan(*grid, 0), oracle.make_plan(*grid, 1)
    row = 3072 * 2
    a_rows = a_max = 0
    for s, d in ((reg, sft), (sft, reg)):
        c = osp.plan_a(s, d, ranks)["counts"]
        off = c - np.diag(np.diag(c))
        a_rows += int(off.sum())
        a_max += int(max(off.sum(axis=1).max(), off.sum(axis=0).max()))
    b = osp.plan_b(reg, sft, ranks)
    n = np.diff(sft.offsets).astype(np.float64)
    a_work = np.bincount(osp.owners(sft, ranks), weights=n * n, minlength=ranks)
    got = sp.crossover(*grid, ranks, channels=3072, shifted_ms=2.0)
    assert got["plan_a_bytes"] == a_rows * row and got["plan_a_max_rank_bytes"] == a_max * row
    assert got["plan_b_bytes"] == 2 * int(b["halo_in"].sum()) * row
    assert got["plan_b_max_rank_bytes"] == 2 * int(max(b["halo_in"].max(), b["halo_out"].max())) * row
    assert np.isclose(got["plan_a_shifted_imbalance"], a_work.max() / a_work.mean())
    assert np.isclose(got["plan_b_shifted_imbalance"], b["work"].max() / np.mean(b["work"]))
    ta, tb = 2.0 * a_work.max() / a_work.sum(), 2.0 * b["work"].max() / a_work.sum()
    assert np.isclose(got["plan_a_shifted_ms_max_rank"], ta) and np.isclose(got["plan_b_shifted_ms_max_rank"], tb)
    dbytes = (a_max - 2 * int(max(b["halo_in"].max(), b["halo_out"].max()))) * row
    if tb > ta and dbytes > 0:
        assert np.isclose(got["crossover_link_gbs"], dbytes / ((tb - ta) * 1e-3) / 1e9)
    else:
        assert got["crossover_link_gbs"] is None
