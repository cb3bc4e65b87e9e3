"""Pins of the window-local 3D RoPE oracle ("Window-Aligned Sequence
Parallelism (SeedVR2)", section "Reference quirks reproduced on purpose";
the readings of the oracle's header).  Each pin uses a formulation other
than the oracle's own (complex arithmetic, an explicit rotation matrix), a
hand-worked position, or an invariant that RoPE guarantees by construction."""

import numpy as np
import pytest

import oracle
from oracle import rope

TINY = (4, 9, 16, 2, 9, 16)


def _complex_rope(x, pos, rope_dim=128, theta=10000.0):
    # pair j of axis a as the complex number x[2j] + i x[2j+1], times e^{i angle}
    y = np.array(x, dtype=np.float64, copy=True)
    da = rope_dim // 3
    for a in range(3):
        for j in range(da // 2):
            c0 = a * da + 2 * j
            z = y[..., c0] + 1j * y[..., c0 + 1]
            ang = pos[:, a].astype(np.float64) * theta ** (-2.0 * j / da)
            z = z * np.exp(1j * ang)[:, None]
            y[..., c0], y[..., c0 + 1] = z.real, z.imag
    return y


def _rotation_matrix(p, d=128, rope_dim=128, theta=10000.0):
    R = np.eye(d)
    da = rope_dim // 3
    for a in range(3):
        for j in range(da // 2):
            ang = p[a] * theta ** (-2.0 * j / da)
            c0 = a * da + 2 * j
            R[c0:c0 + 2, c0:c0 + 2] = [[np.cos(ang), -np.sin(ang)], [np.sin(ang), np.cos(ang)]]
    return R


def test_inv_freq_closed_form():
    f = rope.inv_freq(128)
    assert f.shape == (21,)
    assert f[0] == 1.0
    assert f[1] == pytest.approx(10000.0 ** (-2.0 / 42.0), rel=1e-15)
    assert f[-1] == pytest.approx(10000.0 ** (-40.0 / 42.0), rel=1e-15)


def test_matches_complex_formulation():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((50, 3, 128))
    pos = rng.integers(0, 600, size=(50, 3))
    np.testing.assert_allclose(rope.apply_rope(x, pos), _complex_rope(x, pos), atol=1e-12)


def test_matches_rotation_matrix():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((7, 2, 128))
    pos = rng.integers(0, 40, size=(7, 3))
    got = rope.apply_rope(x, pos)
    for n in range(7):
        R = _rotation_matrix(pos[n])
        np.testing.assert_allclose(got[n], x[n] @ R.T, atol=1e-12)


def test_norm_preserved_and_tail_passes_through():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((20, 4, 128))
    pos = rng.integers(0, 300, size=(20, 3))
    y = rope.apply_rope(x, pos)
    np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)
    assert np.array_equal(y[..., 126:], x[..., 126:])  # 3 * (128 // 3) = 126 rotated channels
    assert np.array_equal(rope.apply_rope(x, np.zeros((20, 3), dtype=np.int64)), x)


def test_scores_depend_on_position_difference_only():
    rng = np.random.default_rng(4)
    q, k = rng.standard_normal((1, 1, 128)), rng.standard_normal((1, 1, 128))
    pq, pk = np.array([[5, 3, 9]]), np.array([[2, 7, 1]])
    base = float(np.sum(rope.apply_rope(q, pq) * rope.apply_rope(k, pk)))
    for shift in ([1, 0, 0], [0, 11, 0], [0, 0, 4], [37, 2, 19]):
        s = np.array([shift])
        got = float(np.sum(rope.apply_rope(q, pq + s) * rope.apply_rope(k, pk + s)))
        assert got == pytest.approx(base, abs=1e-12)


def test_hand_worked_positions_tiny():
    # token (t, h, w) = (1, 2, 3), canonical id (1*9 + 2)*16 + 3 = 179.
    # regular windows (wt, wh, ww) = (2, 5, 5): it is in box t[0,2) h[0,5) w[0,5) -> (1, 2, 3)
    # shifted cuts t {0,1,3,4}, h {0,2,7,9}, w {0,2,7,12,16}: box t[1,3) h[2,7) w[2,7) -> (0, 0, 1)
    reg = rope.window_positions(oracle.make_plan(*TINY, 0), text_len=0)
    sft = rope.window_positions(oracle.make_plan(*TINY, 1), text_len=0)
    assert tuple(reg[179]) == (1, 2, 3)
    assert tuple(sft[179]) == (0, 0, 1)
    assert tuple(rope.window_positions(oracle.make_plan(*TINY, 1), text_len=77)[179]) == (77, 0, 1)


@pytest.mark.parametrize("layout", [0, 1])
def test_every_window_restarts_at_zero(layout):
    p = oracle.make_plan(21, 45, 80, 4, 3, 3, layout)
    pos = rope.window_positions(p, text_len=5)
    for w, (t0, t1, h0, h1, w0, w1) in enumerate(p.boxes):
        rows = p.ids[p.offsets[w]:p.offsets[w + 1]]
        assert tuple(pos[rows[0]]) == (5, 0, 0)
        assert tuple(pos[rows[-1]]) == (5 + t1 - t0 - 1, h1 - h0 - 1, w1 - w0 - 1)


def test_text_positions_diagonal():
    assert rope.text_positions(3).tolist() == [[0, 0, 0], [1, 1, 1], [2, 2, 2]]


def test_text_len_does_not_change_video_attention():
    # text_len shifts the first axial index of every video token of a window
    # by the same amount, so window attention (video only) cannot change.
    plan = oracle.make_plan(4, 9, 16, 2, 3, 3, 1)
    rng = np.random.default_rng(5)
    q, k, v = (rng.standard_normal((plan.num_tokens, 2, 128)) for _ in range(3))
    outs = []
    for tl in (0, 256):
        pos = rope.window_positions(plan, text_len=tl)
        outs.append(oracle.window_attention(rope.apply_rope(q, pos), rope.apply_rope(k, pos), v, plan))
    np.testing.assert_allclose(outs[0], outs[1], atol=1e-12)
    pos = rope.window_positions(plan, text_len=0)
    plain = oracle.window_attention(q, k, v, plan)
    assert np.max(np.abs(plain - outs[0])) > 1e-3  # and RoPE does change the result
