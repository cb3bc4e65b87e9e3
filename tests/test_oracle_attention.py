"""Pins of the oracle's window attention ("Window-Aligned Sequence Parallelism
(SeedVR2)", section "Motivation": attention only inside a window, no global
attention) against brute force, library routines and closed forms."""

import numpy as np
import pytest
import torch

import oracle


def _qkv(n, heads, d, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return tuple(rng.standard_normal((n, heads, d)) * scale for _ in range(3))


@pytest.mark.parametrize("grid,layout", [
    ((4, 9, 16, 2, 9, 16), 0), ((4, 9, 16, 2, 9, 16), 1),
    ((3, 7, 10, 2, 3, 4), 0), ((3, 7, 10, 2, 3, 4), 1),
])
def test_matches_masked_full_attention(grid, layout):
    p = oracle.make_plan(*grid, layout)
    q, k, v = _qkv(p.num_tokens, 2, 16, 1)
    a = oracle.window_attention(q, k, v, p)
    b = oracle.masked_full_attention(q, k, v, p)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_single_window_is_sdpa():
    # nt = nh = nw = 1 with T <= 30 and a small H*W: one window covers the grid,
    # so the result is plain scaled-dot-product attention (library routine).
    p = oracle.make_plan(3, 6, 10, 1, 1, 1, 0)
    assert p.num_windows == 1
    q, k, v = _qkv(p.num_tokens, 3, 32, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(
        *(torch.from_numpy(x).permute(1, 0, 2) for x in (q, k, v))).permute(1, 0, 2).numpy()
    np.testing.assert_allclose(oracle.window_attention(q, k, v, p), ref, rtol=0, atol=1e-12)


def test_one_token_windows_return_v_exactly():
    # wt = wh = ww = 1: every window holds one token, softmax of one score is 1,
    # so O = V bit for bit.
    p = oracle.make_plan(2, 3, 4, 2, 52, 69, 0)
    assert (p.wt, p.wh, p.ww) == (1, 1, 1) and p.num_windows == p.num_tokens
    q, k, v = _qkv(p.num_tokens, 2, 8, 3)
    assert np.array_equal(oracle.window_attention(q, k, v, p), v)


def test_constant_keys_give_mean_of_values():
    p = oracle.make_plan(4, 9, 16, 2, 9, 16, 1)
    q, k, v = _qkv(p.num_tokens, 2, 8, 4)
    k = np.ones_like(k) * 0.3
    out = oracle.window_attention(q, k, v, p)
    for w in range(p.num_windows):
        rows = p.ids[p.offsets[w]:p.offsets[w + 1]]
        np.testing.assert_allclose(out[rows], np.broadcast_to(v[rows].mean(axis=0), out[rows].shape),
                                   rtol=0, atol=1e-13)


def test_isolation_between_windows():
    # Change one window's inputs: only that window's outputs may change, and the
    # other windows stay bit-identical (the isolation test of the diffusion-runtime
    # blog, section 5.1, applied to windows).
    p = oracle.make_plan(4, 9, 16, 2, 9, 16, 0)
    q, k, v = _qkv(p.num_tokens, 2, 8, 5)
    base = oracle.window_attention(q, k, v, p)
    rows = p.ids[p.offsets[3]:p.offsets[4]]
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    q2[rows] += 1.0
    k2[rows] *= -1.0
    v2[rows] += 2.0
    out = oracle.window_attention(q2, k2, v2, p)
    other = np.setdiff1d(np.arange(p.num_tokens), rows)
    assert np.array_equal(out[other], base[other])
    assert not np.allclose(out[rows], base[rows])


def test_rows_helper_and_packed_order():
    p = oracle.make_plan(3, 7, 10, 2, 3, 4, 1)
    q, k, v = _qkv(p.num_tokens, 3, 8, 6)
    full = oracle.window_attention(q, k, v, p)
    w = p.num_windows // 2
    n = int(p.offsets[w + 1] - p.offsets[w])
    sel = [0, n // 2, n - 1]
    got = oracle.window_attention_rows(q, k, v, p, w, 1, sel)
    rows = p.ids[p.offsets[w]:p.offsets[w + 1]][sel]
    np.testing.assert_allclose(got, full[rows, 1, :], rtol=0, atol=1e-13)
    # packed order: row p holds packed position p
    packed = oracle.window_attention(q[p.ids], k[p.ids], v[p.ids], p, canonical=False)
    np.testing.assert_allclose(packed, full[p.ids], rtol=0, atol=1e-13)


def test_explicit_scale():
    p = oracle.make_plan(4, 9, 16, 2, 9, 16, 0)
    q, k, v = _qkv(p.num_tokens, 1, 4, 7)
    a = oracle.window_attention(q, k, v, p, scale=0.25)
    b = oracle.window_attention(q * 0.5, k, v, p)  # 1/sqrt(4) = 0.5 -> 0.25 total
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)
