"""Pins of the LPT planner ("Window-Aligned Sequence Parallelism (SeedVR2)",
section "Planner")."""

import numpy as np

import oracle


def test_hand_example():
    # sorted by (-tokens, id): 0(5) 1(3) 2(3) 3(2) 4(2) 5(1)
    # 0->r0 (5,0); 1->r1 (5,3); 2->r1 (5,6); 3->r0 (7,6); 4->r1 (7,8); 5->r0 (8,8)
    owned, load = oracle.lpt_assign([5, 3, 3, 2, 2, 1], 2)
    assert owned == [[0, 3, 5], [1, 2, 4]]
    assert load == [8, 8]


def test_ties_go_to_lower_rank_and_id():
    owned, load = oracle.lpt_assign([4, 4, 4, 4], 4)
    assert owned == [[0], [1], [2], [3]]
    owned, _ = oracle.lpt_assign([1, 1], 3)
    assert owned == [[0], [1], []]


def test_partition_and_bound_random():
    rng = np.random.default_rng(0)
    for _ in range(200):
        n = int(rng.integers(1, 60))
        r = int(rng.integers(1, 9))
        tok = rng.integers(1, 3000, size=n).tolist()
        owned, load = oracle.lpt_assign(tok, r)
        flat = sorted(i for o in owned for i in o)
        assert flat == list(range(n))
        assert all(o == sorted(o) for o in owned)
        assert load == [sum(tok[i] for i in o) for o in owned]
        # greedy list-scheduling bound: the last window placed on the fullest
        # rank found it at or below the mean, so max load <= mean + largest.
        assert max(load) <= sum(tok) / r + max(tok)
        # LPT never leaves a rank idle while another holds two windows
        if n >= r:
            assert all(len(o) > 0 for o in owned)
