"""Per-window softmax attention in fp64.

"Window-Aligned Sequence Parallelism (SeedVR2)", section "Motivation": every
layer partitions the video tokens into windows and attends only inside a
window (no global attention).  For window w and head h:

    O[w, h] = softmax(Q[w, h] K[w, h]^T * scale) V[w, h],   scale = 1/sqrt(d)

with no mask inside a window and no term across windows.  Inputs are upcast
exactly to fp64 and every step runs in fp64.  Q, K, V and O are [N, heads, d]
arrays in canonical token order (row = canonical id), or in the plan's packed
order when ``canonical=False`` (row = packed position).
"""

import math

import numpy as np


def _as64(x):
    return np.asarray(x, dtype=np.float64)


def _softmax_rows(s):
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    return p / p.sum(axis=-1, keepdims=True)


def _scale(d, scale):
    return 1.0 / math.sqrt(d) if (scale is None or scale <= 0) else float(scale)


def _rows_of_window(plan, w, canonical):
    a, b = int(plan.offsets[w]), int(plan.offsets[w + 1])
    if canonical:
        return plan.ids[a:b].astype(np.int64)
    return np.arange(a, b, dtype=np.int64)


def window_attention(q, k, v, plan, scale=None, canonical=True):
    """Full per-window attention over every window and head; returns fp64."""
    q, k, v = _as64(q), _as64(k), _as64(v)
    n_tok, heads, d = q.shape
    if n_tok != plan.num_tokens or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q/k/v shapes do not match the plan")
    c = _scale(d, scale)
    out = np.empty_like(q)
    for w in range(plan.num_windows):
        rows = _rows_of_window(plan, w, canonical)
        qw, kw, vw = q[rows], k[rows], v[rows]
        for h in range(heads):
            p = _softmax_rows((qw[:, h, :] @ kw[:, h, :].T) * c)
            out[rows, h, :] = p @ vw[:, h, :]
    return out


def window_attention_rows(q, k, v, plan, window, head, rows_in_window,
                          scale=None, canonical=True):
    """Attention output of selected query rows of one (window, head).

    ``rows_in_window`` are positions inside the window (0 .. n_w - 1).  Used to
    check sampled outputs at sizes where the full oracle is too slow."""
    q, k, v = np.asarray(q), np.asarray(k), np.asarray(v)
    d = q.shape[2]
    c = _scale(d, scale)
    rows = _rows_of_window(plan, window, canonical)
    sel = rows[np.asarray(rows_in_window, dtype=np.int64)]
    qs = _as64(q[sel, head, :])
    kw = _as64(k[rows, head, :])
    vw = _as64(v[rows, head, :])
    p = _softmax_rows((qs @ kw.T) * c)
    return p @ vw


def masked_full_attention(q, k, v, plan, scale=None, canonical=True):
    """Brute force: dense N x N attention per head with a block-diagonal mask
    that keeps only same-window pairs.  Tiny grids only (O(N^2) memory)."""
    q, k, v = _as64(q), _as64(k), _as64(v)
    n_tok, heads, d = q.shape
    c = _scale(d, scale)
    label = np.empty(n_tok, dtype=np.int64)
    for w in range(plan.num_windows):
        label[_rows_of_window(plan, w, canonical)] = w
    same = label[:, None] == label[None, :]
    out = np.empty_like(q)
    for h in range(heads):
        s = (q[:, h, :] @ k[:, h, :].T) * c
        s = np.where(same, s, -np.inf)
        out[:, h, :] = _softmax_rows(s) @ v[:, h, :]
    return out


def window_attention_text(q, k, v, q_txt, k_txt, v_txt, plan, scale=None, canonical=True):
    """Window attention over packed segments [video window, replicated text].

    "Window-Aligned Sequence Parallelism (SeedVR2)", sections "SeedVR2
    integration" and "Text stream": every window's attention is one segment
    made of the window's video tokens followed by the text tokens (the same
    text for every window); each window yields a text output, and the layer's
    text output is the sum of the per-window text outputs divided by the
    global window count of the layout:  T = (sum_w T_w) / W.

    q, k, v: [N, heads, d] (canonical or packed rows); q_txt, k_txt, v_txt:
    [n_text, heads, d].  Returns (video output [N, heads, d], text output
    [n_text, heads, d]), both fp64."""
    q, k, v = _as64(q), _as64(k), _as64(v)
    qt, kt, vt = _as64(q_txt), _as64(k_txt), _as64(v_txt)
    n_tok, heads, d = q.shape
    n_text = qt.shape[0]
    c = _scale(d, scale)
    out = np.empty_like(q)
    t_sum = np.zeros((n_text, heads, d))
    for w in range(plan.num_windows):
        rows = _rows_of_window(plan, w, canonical)
        n = rows.size
        for h in range(heads):
            qs = np.concatenate([q[rows, h, :], qt[:, h, :]])
            ks = np.concatenate([k[rows, h, :], kt[:, h, :]])
            vs = np.concatenate([v[rows, h, :], vt[:, h, :]])
            o = _softmax_rows((qs @ ks.T) * c) @ vs
            out[rows, h, :] = o[:n]
            t_sum[:, h, :] += o[n:]
    return out, t_sum / plan.num_windows
