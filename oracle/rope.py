"""Window-local 3D rotary position embedding (RoPE), fp64 oracle.

"Window-Aligned Sequence Parallelism (SeedVR2)", section "Reference quirks
reproduced on purpose":
* positions are window-local: a video token at window-local (dt, dh, dw)
  takes the axial indices (text_len + dt, dh, dw); every window restarts at 0;
* the rotary span is 3 * (rope_dim // 3) channels (126 of 128), so the last
  channels pass through unrotated.

Readings where the page is silent (each stated again where the library
documents the call):
* axis a in (t, h, w) owns channels [a * da, (a + 1) * da), da = rope_dim // 3;
* within an axis, channels (2j, 2j + 1) form rotation pair j, turned by the
  angle pos_a * theta ** (-2j / da), theta = 10000:
      (x0, x1) -> (x0 cos - x1 sin, x0 sin + x1 cos);
* text token i takes the axial indices (i, i, i), which is why the video's
  first index starts at text_len.

Test infrastructure only: nothing on the product path imports this module.
"""

import numpy as np

from .plan import Plan

DEFAULT_THETA = 10000.0


def inv_freq(rope_dim, theta=DEFAULT_THETA):
    """theta ** (-2j / da) for the da // 2 pairs of one axis, da = rope_dim // 3."""
    da = rope_dim // 3
    return theta ** (-(2.0 * np.arange(da // 2)) / da)


def window_positions(plan: Plan, text_len=0):
    """pos[id] = (text_len + dt, dh, dw) of canonical token id in its window."""
    pos = np.zeros((plan.num_tokens, 3), dtype=np.int64)
    for w, (t0, t1, h0, h1, w0, w1) in enumerate(plan.boxes):
        rows = plan.ids[plan.offsets[w]:plan.offsets[w + 1]]
        dt, dh, dw = np.meshgrid(np.arange(t1 - t0), np.arange(h1 - h0), np.arange(w1 - w0), indexing="ij")
        pos[rows] = np.stack([text_len + dt.ravel(), dh.ravel(), dw.ravel()], axis=1)
    return pos


def text_positions(n_text):
    """Text token i at (i, i, i)."""
    i = np.arange(n_text, dtype=np.int64)
    return np.stack([i, i, i], axis=1)


def apply_rope(x, pos, rope_dim=None, theta=DEFAULT_THETA):
    """Rotate x [n, heads, d] (fp64 copy) by the axial positions pos [n, 3]."""
    x = np.array(x, dtype=np.float64, copy=True)
    d = x.shape[-1]
    rope_dim = d if rope_dim is None else rope_dim
    da = rope_dim // 3
    f = inv_freq(rope_dim, theta)
    for a in range(3):
        ang = pos[:, a:a + 1].astype(np.float64) * f[None, :]  # [n, da/2]
        c, s = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
        x0 = x[..., a * da:(a + 1) * da:2].copy()
        x1 = x[..., a * da + 1:(a + 1) * da:2].copy()
        x[..., a * da:(a + 1) * da:2] = x0 * c - x1 * s
        x[..., a * da + 1:(a + 1) * da:2] = x0 * s + x1 * c
    return x
