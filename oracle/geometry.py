"""Window geometry: window size, per-axis cuts, window enumeration.

Follows "Window-Aligned Sequence Parallelism (SeedVR2)", section "Window
layouts":

* the window size is normalised to a 720p reference area of 45 x 80 post-patch
  tokens: scale = sqrt(45*80 / (H*W)), wh = ceil(round(H*scale) / nh),
  ww = ceil(round(W*scale) / nw), wt = ceil(min(T, 30) / nt);
* the regular layout cuts each axis at multiples of the window size, the last
  window clipped to the axis end;
* the shifted layout moves every cut by half a window and clips at both ends
  (max(.., 0) / min(.., size)) -- it is not a cyclic roll;
* windows are enumerated with w outermost and t innermost.

Readings where the note is silent:

* ``round`` is Python's round-half-to-even on the fp64 product ``H * scale``
  (the note's pseudocode is Python).
* "half a window" for an odd size is floor(w / 2).
* An axis whose size is not larger than its window size is not shifted: there
  is no interior cut to move, so it keeps the single window [0, size).
* An empty interval (e.g. w == 1 gives a first shifted cut at 0) is dropped:
  a partition has no empty block.
* Only the window *size* uses min(T, 30); the cuts tile the whole T axis.
"""

import math

# 720p reference area in post-patch tokens (45 x 80), section "Window layouts".
WINDOW_REF_AREA = 45 * 80
# Temporal cap on the window size (BYTEDANCE_MAX_TEMPORAL_WINDOW in the note).
MAX_TEMPORAL = 30


def _ceil_div(a, b):
    return -(-a // b)


def window_size(T, H, W, nt, nh, nw, max_temporal=MAX_TEMPORAL):
    """Return (wt, wh, ww) for a post-patch grid (T, H, W).

    Raises ValueError when an input is not positive or a size computes to 0
    (the formula is undefined there).
    """
    for name, v in (("T", T), ("H", H), ("W", W), ("nt", nt), ("nh", nh),
                    ("nw", nw), ("max_temporal", max_temporal)):
        if int(v) != v or v <= 0:
            raise ValueError(f"{name} must be a positive integer, got {v!r}")
    scale = math.sqrt(WINDOW_REF_AREA / (H * W))
    resized_h = round(H * scale)
    resized_w = round(W * scale)
    wh = _ceil_div(resized_h, nh)
    ww = _ceil_div(resized_w, nw)
    wt = _ceil_div(min(T, max_temporal), nt)
    if wt <= 0 or wh <= 0 or ww <= 0:
        raise ValueError(f"window size computes to zero: wt={wt} wh={wh} ww={ww}")
    return wt, wh, ww


def axis_intervals(size, w, shifted):
    """Half-open intervals [a, b) that cut one axis of length ``size``.

    Regular: cuts at 0, w, 2w, ... and ``size``.
    Shifted: cuts at 0, floor(w/2), floor(w/2) + w, ... (< size) and ``size``.
    """
    if size <= 0 or w <= 0:
        raise ValueError("size and window must be positive")
    if shifted and size > w:
        cuts = [0] + list(range(w // 2, size, w)) + [size]
    else:
        cuts = list(range(0, size, w)) + [size]
    return [(a, b) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]


def windows(T, H, W, wt, wh, ww, shifted):
    """All windows of one layout as (t0, t1, h0, h1, w0, w1), in the note's
    enumeration order: w outermost, then h, t innermost."""
    ti = axis_intervals(T, wt, shifted)
    hi = axis_intervals(H, wh, shifted)
    wi = axis_intervals(W, ww, shifted)
    out = []
    for (w0, w1) in wi:
        for (h0, h1) in hi:
            for (t0, t1) in ti:
                out.append((t0, t1, h0, h1, w0, w1))
    return out
