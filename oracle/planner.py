"""Deterministic LPT assignment of windows to ranks.

"Window-Aligned Sequence Parallelism (SeedVR2)", section "Planner": windows
are taken in order of (-token count, window id); each goes to the rank with
the smallest (assigned tokens, rank id); every rank then lists its windows in
ascending window id.
"""


def lpt_assign(window_tokens, ranks):
    """Return (per-rank window lists, per-rank token totals)."""
    if ranks <= 0:
        raise ValueError("ranks must be positive")
    order = sorted(range(len(window_tokens)), key=lambda i: (-int(window_tokens[i]), i))
    load = [0] * ranks
    owned = [[] for _ in range(ranks)]
    for i in order:
        r = min(range(ranks), key=lambda j: (load[j], j))
        owned[r].append(i)
        load[r] += int(window_tokens[i])
    return [sorted(o) for o in owned], load
