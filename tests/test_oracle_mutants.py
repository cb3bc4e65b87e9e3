"""Planted mistakes in copies of the oracle, on the CPU: each plausible error
in the plan construction must trip at least one pin in ``tests/pins.py``."""

import numpy as np
import pytest

import oracle
from oracle import geometry, plan as plan_mod
from tests import pins

GRID = (4, 9, 16, 2, 9, 16)


def _make_plan_with(windows_fn=None, ids_fn=None):
    """A copy of the oracle's make_plan with one step replaced."""
    def make(T, H, W, nt, nh, nw, layout, max_temporal=30):
        wt, wh, ww = geometry.window_size(T, H, W, nt, nh, nw, max_temporal)
        boxes = (windows_fn or geometry.windows)(T, H, W, wt, wh, ww, layout == 1)
        grid = np.arange(T * H * W).reshape(T, H, W)
        pieces = [(ids_fn or (lambda g, b: g[b[0]:b[1], b[2]:b[3], b[4]:b[5]].ravel()))(grid, b)
                  for b in boxes]
        ids = np.concatenate(pieces)
        pos = np.full(T * H * W, -1, dtype=np.int64)
        pos[ids] = np.arange(ids.size)
        return plan_mod.Plan(T, H, W, wt, wh, ww, layout, boxes,
                             plan_mod.cu_seqlens([x.size for x in pieces]).astype(np.int32),
                             np.asarray(boxes, dtype=np.int32).reshape(-1, 6),
                             ids.astype(np.int32), pos.astype(np.int32))
    return make


def test_real_oracle_passes():
    assert pins.all_plan_failures(oracle.make_plan, *GRID) == []


def _t_outermost(T, H, W, wt, wh, ww, shifted):
    ti = geometry.axis_intervals(T, wt, shifted)
    hi = geometry.axis_intervals(H, wh, shifted)
    wi = geometry.axis_intervals(W, ww, shifted)
    return [(t0, t1, h0, h1, w0, w1) for (t0, t1) in ti for (h0, h1) in hi for (w0, w1) in wi]


def _ceil_half_shift(T, H, W, wt, wh, ww, shifted):
    def iv(size, w):
        if shifted and size > w:
            cuts = [0] + list(range((w + 1) // 2, size, w)) + [size]
        else:
            cuts = list(range(0, size, w)) + [size]
        return [(a, b) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]
    return [(t0, t1, h0, h1, w0, w1) for (w0, w1) in iv(W, ww) for (h0, h1) in iv(H, wh)
            for (t0, t1) in iv(T, wt)]


def _rolled(T, H, W, wt, wh, ww, shifted):
    # boxes of the regular layout; ids taken from a cyclically rolled grid below
    return geometry.windows(T, H, W, wt, wh, ww, False)


def _shift_not_clipped_last(T, H, W, wt, wh, ww, shifted):
    # forgets the clipped tail window on every axis
    def iv(size, w):
        cuts = [0] + list(range(w // 2, size, w)) if shifted and size > w else list(range(0, size, w)) + [size]
        return [(a, b) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]
    return [(t0, t1, h0, h1, w0, w1) for (w0, w1) in iv(W, ww) for (h0, h1) in iv(H, wh)
            for (t0, t1) in iv(T, wt)]


@pytest.mark.parametrize("mutant", [
    _make_plan_with(windows_fn=_t_outermost),
    _make_plan_with(windows_fn=_ceil_half_shift),
    _make_plan_with(windows_fn=_shift_not_clipped_last),
    # column-major tokens inside a window
    _make_plan_with(ids_fn=lambda g, b: g[b[0]:b[1], b[2]:b[3], b[4]:b[5]].transpose(2, 1, 0).ravel()),
    # cyclic roll instead of clipping for the shifted layout
    _make_plan_with(windows_fn=_rolled, ids_fn=lambda g, b: np.roll(g, (-1, -2, -2), (0, 1, 2))
                    [b[0]:b[1], b[2]:b[3], b[4]:b[5]].ravel()),
])
def test_mutant_is_caught(mutant):
    assert pins.all_plan_failures(mutant, *GRID) != []


def test_attention_mutants_caught_by_brute_force():
    p = oracle.make_plan(*GRID, 1)
    rng = np.random.default_rng(9)
    q, k, v = (rng.standard_normal((p.num_tokens, 2, 8)) for _ in range(3))
    brute = oracle.masked_full_attention(q, k, v, p)
    good = oracle.window_attention(q, k, v, p)
    assert np.allclose(good, brute, atol=1e-12)
    # planted mistakes: softmax over the query axis; missing 1/sqrt(d); V of
    # the wrong head; K transposed role (Q K^T -> K Q^T)
    def variant(kind):
        out = np.empty_like(q)
        for w in range(p.num_windows):
            r = p.ids[p.offsets[w]:p.offsets[w + 1]]
            for h in range(2):
                s = q[r, h] @ k[r, h].T
                if kind != "noscale":
                    s = s / np.sqrt(8)
                if kind == "transpose":
                    s = s.T
                ax = 0 if kind == "axis" else 1
                e = np.exp(s - s.max(axis=ax, keepdims=True))
                pm = e / e.sum(axis=ax, keepdims=True)
                out[r, h] = pm @ v[r, 1 - h if kind == "head" else h]
        return out
    for kind in ("axis", "noscale", "head", "transpose"):
        assert not np.allclose(variant(kind), brute, atol=1e-6), kind
