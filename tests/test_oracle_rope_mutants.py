"""Planted mistakes in copies of the RoPE oracle, on the CPU: each plausible
error must trip at least one independent check (complex arithmetic per
pair, hand-worked window-local positions, window restarts)."""

import numpy as np

import oracle
from oracle import rope

TINY = (4, 9, 16, 2, 9, 16)


def _complex_reference(x, pos, rope_dim=128, theta=10000.0):
    y = np.array(x, dtype=np.float64, copy=True)
    da = rope_dim // 3
    for a in range(3):
        for j in range(da // 2):
            c0 = a * da + 2 * j
            z = (y[..., c0] + 1j * y[..., c0 + 1]) * np.exp(1j * pos[:, a] * theta ** (-2.0 * j / da))[:, None]
            y[..., c0], y[..., c0 + 1] = z.real, z.imag
    return y


def failures(apply_fn, positions_fn):
    out = []
    rng = np.random.default_rng(9)
    x = rng.standard_normal((16, 2, 128))
    pos = rng.integers(0, 200, size=(16, 3))
    if not np.allclose(apply_fn(x, pos), _complex_reference(x, pos), atol=1e-10):
        out.append("complex formulation")
    reg = positions_fn(oracle.make_plan(*TINY, 0), 0)
    sft = positions_fn(oracle.make_plan(*TINY, 1), 77)
    if tuple(reg[179]) != (1, 2, 3) or tuple(sft[179]) != (77, 0, 1):
        out.append("hand positions")
    p = oracle.make_plan(*TINY, 1)
    pp = positions_fn(p, 3)
    for w in range(p.num_windows):
        if tuple(pp[p.ids[p.offsets[w]]]) != (3, 0, 0):
            out.append("restart")
            break
    return out


def _apply(mut):
    def f(x, pos, rope_dim=128, theta=10000.0):
        x = np.array(x, dtype=np.float64, copy=True)
        da = rope_dim // 3
        fr = rope.inv_freq(rope_dim, theta)
        for a in range(3):
            ang = pos[:, a:a + 1] * fr[None, :]
            c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
            lo, hi = a * da, (a + 1) * da
            if mut == "half_split":  # pairs (j, j + da/2) instead of (2j, 2j+1)
                x0, x1 = x[..., lo:lo + da // 2].copy(), x[..., lo + da // 2:hi].copy()
                x[..., lo:lo + da // 2], x[..., lo + da // 2:hi] = x0 * c - x1 * s, x0 * s + x1 * c
                continue
            x0, x1 = x[..., lo:hi:2].copy(), x[..., lo + 1:hi:2].copy()
            if mut == "sin_sign":
                s = -s
            if mut == "axis_order" and a < 2:
                ang = pos[:, 1 - a:2 - a] * fr[None, :]
                c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
            x[..., lo:hi:2], x[..., lo + 1:hi:2] = x0 * c - x1 * s, x0 * s + x1 * c
        return x
    return f


def _positions(mut):
    def f(plan, text_len):
        pos = np.zeros((plan.num_tokens, 3), dtype=np.int64)
        for w, (t0, t1, h0, h1, w0, w1) in enumerate(plan.boxes):
            rows = plan.ids[plan.offsets[w]:plan.offsets[w + 1]]
            tt, hh, ww = np.meshgrid(np.arange(t0, t1), np.arange(h0, h1), np.arange(w0, w1), indexing="ij")
            if mut == "global":  # grid coordinates, no restart
                pos[rows] = np.stack([text_len + tt.ravel(), hh.ravel(), ww.ravel()], 1)
            elif mut == "offset_on_w":  # text offset on the last axis
                pos[rows] = np.stack([tt.ravel() - t0, hh.ravel() - h0, text_len + ww.ravel() - w0], 1)
            else:
                pos[rows] = np.stack([text_len + tt.ravel() - t0, hh.ravel() - h0, ww.ravel() - w0], 1)
        return pos
    return f


def test_real_oracle_passes():
    assert failures(rope.apply_rope, rope.window_positions) == []
    assert failures(_apply(None), _positions(None)) == []  # the un-mutated copies


def test_each_mutant_is_caught():
    for m in ("half_split", "sin_sign", "axis_order"):
        assert failures(_apply(m), rope.window_positions), m
    for m in ("global", "offset_on_w"):
        assert failures(rope.apply_rope, _positions(m)), m
