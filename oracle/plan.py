"""One layout's window plan: ragged offsets, window boxes and token-id tables.

"Window-Aligned Sequence Parallelism (SeedVR2)", section "Window layouts":
tokens inside a window are row-major in (t, h, w) and the canonical token id
is (t*H + h)*W + w, which is what windowing ``arange`` gives.  The packed
order of a layout is the concatenation of its windows in enumeration order;
``offsets`` are the segment boundaries in the ``cu_seqlens`` convention of the
vLLM-Omni diffusion-runtime blog, section 4.2 (prefix sums, first entry 0,
last entry the total).
"""

from dataclasses import dataclass

import numpy as np

from .geometry import window_size, windows, MAX_TEMPORAL

REGULAR = 0
SHIFTED = 1


def cu_seqlens(lengths):
    """Prefix-sum boundaries of packed segments, starting at 0.

    A zero-length segment repeats the previous boundary (blog section 4.2:
    lengths 60, 4, 64, 0 give [0, 60, 64, 128, 128])."""
    out = [0]
    for n in lengths:
        if n < 0:
            raise ValueError("segment length must be >= 0")
        out.append(out[-1] + int(n))
    return np.asarray(out, dtype=np.int64)


@dataclass
class Plan:
    T: int
    H: int
    W: int
    wt: int
    wh: int
    ww: int
    layout: int            # REGULAR or SHIFTED
    boxes: list            # [(t0, t1, h0, h1, w0, w1)] in enumeration order
    offsets: np.ndarray    # int32 [num_windows + 1]
    dims: np.ndarray       # int32 [num_windows, 6]
    ids: np.ndarray        # int32 [N]: canonical id of packed position p
    pos: np.ndarray        # int32 [N]: packed position of canonical id

    @property
    def num_tokens(self):
        return self.T * self.H * self.W

    @property
    def num_windows(self):
        return len(self.boxes)

    @property
    def max_window_tokens(self):
        return int(np.max(np.diff(self.offsets)))


def make_plan(T, H, W, nt, nh, nw, layout, max_temporal=MAX_TEMPORAL):
    """Build the plan of one layout (REGULAR=0 or SHIFTED=1)."""
    if layout not in (REGULAR, SHIFTED):
        raise ValueError("layout must be 0 (regular) or 1 (shifted)")
    wt, wh, ww = window_size(T, H, W, nt, nh, nw, max_temporal)
    boxes = windows(T, H, W, wt, wh, ww, layout == SHIFTED)
    grid = np.arange(T * H * W, dtype=np.int64).reshape(T, H, W)
    pieces = [grid[t0:t1, h0:h1, w0:w1].ravel() for (t0, t1, h0, h1, w0, w1) in boxes]
    ids = np.concatenate(pieces)
    offsets = cu_seqlens([p.size for p in pieces])
    pos = np.empty_like(ids)
    pos[ids] = np.arange(ids.size, dtype=np.int64)
    return Plan(T=T, H=H, W=W, wt=wt, wh=wh, ww=ww, layout=layout, boxes=boxes,
                offsets=offsets.astype(np.int32),
                dims=np.asarray(boxes, dtype=np.int32).reshape(-1, 6),
                ids=ids.astype(np.int32), pos=pos.astype(np.int32))
