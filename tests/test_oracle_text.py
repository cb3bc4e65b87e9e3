"""Pins of the oracle's text segment ("Window-Aligned Sequence Parallelism
(SeedVR2)", sections "Text stream" and "SeedVR2 integration")."""

import numpy as np
import pytest
import torch

import oracle


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


@pytest.mark.parametrize("layout", [0, 1])
def test_no_text_is_video_attention(layout):
    p = oracle.make_plan(4, 9, 16, 2, 9, 16, layout)
    q, k, v = (_rand((p.num_tokens, 2, 8), s) for s in (1, 2, 3))
    e = np.zeros((0, 2, 8))
    out, txt = oracle.window_attention_text(q, k, v, e, e, e, p)
    np.testing.assert_allclose(out, oracle.window_attention(q, k, v, p), rtol=0, atol=1e-13)
    assert txt.shape == (0, 2, 8)


def test_single_window_is_sdpa_over_video_then_text():
    # One window covers the grid: the segment is [all video tokens, text], and
    # both outputs are rows of one scaled-dot-product attention (library routine).
    p = oracle.make_plan(3, 6, 10, 1, 1, 1, 0)
    assert p.num_windows == 1
    n_text = 7
    q, k, v = (_rand((p.num_tokens, 2, 16), s) for s in (4, 5, 6))
    qt, kt, vt = (_rand((n_text, 2, 16), s) for s in (7, 8, 9))
    out, txt = oracle.window_attention_text(q, k, v, qt, kt, vt, p)
    seq = [torch.from_numpy(np.concatenate([a, b])).permute(1, 0, 2) for a, b in ((q, qt), (k, kt), (v, vt))]
    ref = torch.nn.functional.scaled_dot_product_attention(*seq).permute(1, 0, 2).numpy()
    np.testing.assert_allclose(out, ref[:p.num_tokens], rtol=0, atol=1e-12)
    np.testing.assert_allclose(txt, ref[p.num_tokens:], rtol=0, atol=1e-12)


def test_matches_masked_attention_on_replicated_sequence():
    # Independent construction: lay all segments end to end ([window w, text copy
    # w] for every w), run one dense attention with a block-diagonal segment mask,
    # read the video rows back and average the text copies.
    p = oracle.make_plan(4, 9, 16, 2, 9, 16, 1)
    n_text, heads, d = 5, 2, 8
    q, k, v = (_rand((p.num_tokens, heads, d), s) for s in (10, 11, 12))
    qt, kt, vt = (_rand((n_text, heads, d), s) for s in (13, 14, 15))
    seg, idx = [], []
    for w in range(p.num_windows):
        rows = p.ids[p.offsets[w]:p.offsets[w + 1]]
        idx.append(np.concatenate([rows, -1 - np.arange(n_text)]))
        seg.append(np.full(rows.size + n_text, w))
    idx, seg = np.concatenate(idx), np.concatenate(seg)
    def gather(x, xt):
        return np.where((idx >= 0)[:, None, None], x[np.maximum(idx, 0)], xt[np.maximum(-1 - idx, 0)])
    Q, K, V = gather(q, qt), gather(k, kt), gather(v, vt)
    mask = seg[:, None] == seg[None, :]
    o = np.empty_like(Q)
    for h in range(heads):
        s = np.where(mask, (Q[:, h] @ K[:, h].T) / np.sqrt(d), -np.inf)
        s = np.exp(s - s.max(axis=1, keepdims=True))
        o[:, h] = (s / s.sum(axis=1, keepdims=True)) @ V[:, h]
    out, txt = oracle.window_attention_text(q, k, v, qt, kt, vt, p)
    vid = idx >= 0
    ref_out = np.empty_like(q)
    ref_out[idx[vid]] = o[vid]
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    ref_txt = np.zeros((n_text, heads, d))
    for t in range(n_text):
        ref_txt[t] = o[idx == -1 - t].mean(axis=0)
    np.testing.assert_allclose(txt, ref_txt, rtol=0, atol=1e-12)


def test_divides_by_global_window_count_not_tokens():
    # Identical windows (constant video inputs, so every segment is the same up to
    # its length) -- the text output is a plain mean over windows, not weighted by
    # window size: windows of different sizes give different T_w and the result
    # is their unweighted average.
    p = oracle.make_plan(4, 9, 16, 2, 9, 16, 1)
    n_text = 3
    q = np.ones((p.num_tokens, 1, 4)) * 0.2
    k = np.ones_like(q) * 0.5
    v = np.ones_like(q) * 2.0
    qt = np.ones((n_text, 1, 4)) * 0.2
    kt = np.ones((n_text, 1, 4)) * 0.5
    vt = np.zeros((n_text, 1, 4))
    out, txt = oracle.window_attention_text(q, k, v, qt, kt, vt, p)
    # every score is equal, so T_w = (2 n_w + 0 n_text) / (n_w + n_text)
    n = np.diff(p.offsets).astype(np.float64)
    expect = np.mean(2.0 * n / (n + n_text))
    np.testing.assert_allclose(txt, expect, rtol=0, atol=1e-13)
    # a token-weighted mean would differ on this ragged layout
    assert abs(expect - (2.0 * n.sum() / (n + n_text).sum())) > 1e-3


def test_isolation_with_text():
    # Changing one window's video inputs changes that window's video rows and the
    # text output, never another window's video rows.
    p = oracle.make_plan(4, 9, 16, 2, 9, 16, 0)
    q, k, v = (_rand((p.num_tokens, 2, 8), s) for s in (20, 21, 22))
    qt, kt, vt = (_rand((4, 2, 8), s) for s in (23, 24, 25))
    out, txt = oracle.window_attention_text(q, k, v, qt, kt, vt, p)
    rows = p.ids[p.offsets[2]:p.offsets[3]]
    v2 = v.copy()
    v2[rows] += 1.0
    out2, txt2 = oracle.window_attention_text(q, k, v2, qt, kt, vt, p)
    other = np.setdiff1d(np.arange(p.num_tokens), rows)
    assert np.array_equal(out2[other], out[other])
    assert not np.allclose(out2[rows], out[rows])
    assert not np.allclose(txt2, txt)
