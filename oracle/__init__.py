"""Oracle for NaDiT-style 3D regular/shifted window attention.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously correct CPU
restatement of what the library computes, written in numpy with fp64 arithmetic.
Only the test-suite, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import it.  The product path
(``shifted_window_attention_gb300``) never imports or calls anything here, and
this package imports nothing from the product: the two share no code.  The only
module both sides use is ``wsa_inputs`` (seeded synthetic inputs, no method
arithmetic).

Source of truth: the vllm-omni design note "Window-Aligned Sequence Parallelism
(SeedVR2)", sections "Window layouts" (geometry, cuts, enumeration, token ids),
"Planner" (LPT assignment) and "Motivation" (attention only inside a window),
plus the vLLM-Omni diffusion-runtime blog, section 4.2 (``cu_seqlens``
convention for packed segments).

Every function is pinned by ``tests/test_oracle_*.py`` against closed forms,
hand-derived worked examples, invariants the note states, brute force on tiny
grids and library routines; none is "parity unpinned".
"""

from .geometry import window_size, axis_intervals, windows, WINDOW_REF_AREA
from .plan import Plan, make_plan, cu_seqlens
from .transition import transition, gather_table
from .attention import (window_attention, masked_full_attention, window_attention_rows,
                        window_attention_text)
from .planner import lpt_assign
from . import sp
from . import rope

__all__ = [
    "WINDOW_REF_AREA",
    "window_size",
    "axis_intervals",
    "windows",
    "Plan",
    "make_plan",
    "cu_seqlens",
    "transition",
    "gather_table",
    "window_attention",
    "window_attention_rows",
    "masked_full_attention",
    "window_attention_text",
    "lpt_assign",
    "sp",
    "rope",
]
