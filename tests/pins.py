"""Checks that pin the oracle's plan construction to what the window note fixes.

Each check takes a plan-building function with the signature of
``oracle.make_plan`` and returns a list of failure strings (empty = pinned).
The same checks are run against deliberately broken variants of the oracle in
``test_oracle_mutants.py`` to show that each plausible mistake is caught.

Source: "Window-Aligned Sequence Parallelism (SeedVR2)", section "Window
layouts" (exact partition, shifted differs from regular, clipped not rolled,
w-outermost / t-innermost enumeration, row-major tokens inside a window,
canonical id (t*H+h)*W+w, ragged edge windows).
"""

import bisect

import numpy as np


def _decode(ids, H, W):
    ids = np.asarray(ids, dtype=np.int64)
    return ids // (H * W), (ids // W) % H, ids % W


def partition_failures(plan):
    fails = []
    N = plan.T * plan.H * plan.W
    ids = np.asarray(plan.ids, dtype=np.int64)
    if ids.size != N or not np.array_equal(np.sort(ids), np.arange(N)):
        fails.append("ids is not a permutation of arange(N)")
    if int(plan.offsets[0]) != 0 or int(plan.offsets[-1]) != N:
        fails.append("offsets do not run from 0 to N")
    if np.any(np.diff(plan.offsets) <= 0):
        fails.append("empty or negative window")
    pos = np.asarray(plan.pos, dtype=np.int64)
    if ids.size == N and not np.array_equal(pos[ids], np.arange(N)):
        fails.append("pos is not the inverse of ids")
    return fails


def box_failures(plan):
    """Every window's ids form exactly its box, row-major inside the window."""
    fails = []
    t, h, w = _decode(plan.ids, plan.H, plan.W)
    for k in range(len(plan.offsets) - 1):
        a, b = int(plan.offsets[k]), int(plan.offsets[k + 1])
        t0, t1, h0, h1, w0, w1 = (int(x) for x in plan.dims[k])
        if (t1 - t0) * (h1 - h0) * (w1 - w0) != b - a:
            fails.append(f"window {k}: size {b - a} != box volume")
            continue
        tt, hh, ww = np.meshgrid(np.arange(t0, t1), np.arange(h0, h1), np.arange(w0, w1),
                                 indexing="ij")
        expect = ((tt * plan.H + hh) * plan.W + ww).ravel()
        if not np.array_equal(np.asarray(plan.ids[a:b], dtype=np.int64), expect):
            fails.append(f"window {k}: ids are not the row-major box")
        if t[a:b].min() < t0 or t[a:b].max() >= t1 or h[a:b].min() < h0 or w[a:b].max() >= w1:
            fails.append(f"window {k}: token outside its box")
    return fails


def _cuts_of(dims, lo, hi):
    return sorted({int(d[lo]) for d in dims} | {int(d[hi]) for d in dims})


def enumeration_failures(plan):
    """Independent construction: label each token with its window number
    (iw * nH + ih) * nT + it found by interval search on the cut lists, then a
    stable sort of the canonical ids by label must give ``ids``."""
    fails = []
    dims = np.asarray(plan.dims)
    tc, hc, wc = _cuts_of(dims, 0, 1), _cuts_of(dims, 2, 3), _cuts_of(dims, 4, 5)
    nT, nH, nW = len(tc) - 1, len(hc) - 1, len(wc) - 1
    if nT * nH * nW != len(dims):
        return ["window count is not the product of per-axis counts"]
    N = plan.T * plan.H * plan.W
    t, h, w = _decode(np.arange(N), plan.H, plan.W)
    it = np.array([bisect.bisect_right(tc, x) - 1 for x in range(plan.T)])[t]
    ih = np.array([bisect.bisect_right(hc, x) - 1 for x in range(plan.H)])[h]
    iw = np.array([bisect.bisect_right(wc, x) - 1 for x in range(plan.W)])[w]
    label = (iw * nH + ih) * nT + it
    expect = np.argsort(label, kind="stable")
    if not np.array_equal(np.asarray(plan.ids, dtype=np.int64), expect):
        fails.append("ids differ from the label-sort construction (order or membership)")
    counts = np.bincount(label, minlength=len(dims))
    if not np.array_equal(counts, np.diff(np.asarray(plan.offsets, dtype=np.int64))):
        fails.append("offsets differ from per-window token counts")
    return fails


def regular_cut_failures(plan):
    """Regular cuts sit at multiples of the window size, the last one clipped."""
    fails = []
    dims = np.asarray(plan.dims)
    for (lo, hi, size, w) in ((0, 1, plan.T, plan.wt), (2, 3, plan.H, plan.wh),
                              (4, 5, plan.W, plan.ww)):
        expect = sorted(set(range(0, size, w)) | {size})
        if _cuts_of(dims, lo, hi) != expect:
            fails.append(f"regular cuts on axis {lo // 2} are {_cuts_of(dims, lo, hi)}, not {expect}")
    return fails


def shifted_cut_failures(plan):
    """Shifted cuts: every regular cut moved by floor(w/2), clipped to [0, size]."""
    fails = []
    dims = np.asarray(plan.dims)
    for (lo, hi, size, w) in ((0, 1, plan.T, plan.wt), (2, 3, plan.H, plan.wh),
                              (4, 5, plan.W, plan.ww)):
        if size > w:
            moved = {min(max(c + w // 2, 0), size) for c in range(-w, size + w, w)}
            expect = sorted(moved | {0, size})
        else:
            expect = [0, size]
        if _cuts_of(dims, lo, hi) != expect:
            fails.append(f"shifted cuts on axis {lo // 2} are {_cuts_of(dims, lo, hi)}, not {expect}")
    return fails


def not_rolled_failures(plan):
    """Clipped shifting: along every axis a window covers one contiguous range
    of coordinates.  A cyclic roll would give a wrapped window holding both
    ends of an axis ({0..a} and {size-b..size-1}), which is not contiguous."""
    fails = []
    t, h, w = _decode(plan.ids, plan.H, plan.W)
    for k in range(len(plan.offsets) - 1):
        a, b = int(plan.offsets[k]), int(plan.offsets[k + 1])
        for coord in (t, h, w):
            c = coord[a:b]
            if len(np.unique(c)) != c.max() - c.min() + 1:
                fails.append(f"window {k} is not contiguous along an axis (wrapped)")
    return fails


def all_plan_failures(make_plan, T, H, W, nt, nh, nw, max_temporal=30):
    reg = make_plan(T, H, W, nt, nh, nw, 0, max_temporal)
    sft = make_plan(T, H, W, nt, nh, nw, 1, max_temporal)
    fails = []
    for name, p in (("regular", reg), ("shifted", sft)):
        for f in (partition_failures(p) + box_failures(p) + enumeration_failures(p)
                  + not_rolled_failures(p)):
            fails.append(f"{name}: {f}")
    fails += ["regular: " + f for f in regular_cut_failures(reg)]
    fails += ["shifted: " + f for f in shifted_cut_failures(sft)]
    # A shifted axis differs from the regular one when it has an interior cut
    # to move (size > w) and the move is not zero (w >= 2).
    movable = any(size > w >= 2 for size, w in ((T, reg.wt), (H, reg.wh), (W, reg.ww)))
    if movable and np.array_equal(reg.ids, sft.ids) and np.array_equal(reg.offsets, sft.offsets):
        fails.append("shifted layout equals the regular one")
    return fails
