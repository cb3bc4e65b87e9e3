"""Full-size attention parity against the fp64 oracle, spread over host cores.

Test infrastructure.  The oracle itself is unchanged: every (window, head)
problem goes through ``oracle.window_attention_rows`` exactly as the smaller
tests call it.  What this module adds is only distribution: one task per
window, run by a pool of single-threaded worker processes (a problem of a few
thousand rows is too small for a multithreaded BLAS to pay off, so one
process per core finishes a layer several times faster).

The pool is started with the ``spawn`` method, so no worker is ever forked
from a process that holds a CUDA context.  Workers import numpy and the oracle
only.

Tensors travel as raw bf16 bits (uint16) to halve the bytes sent through the
pool's pipes; a worker widens them to fp32 exactly (a bf16 value is the upper
16 bits of the fp32 with the same value) before handing them to the oracle,
which upcasts to fp64.
"""

import os
import types

import numpy as np

_POOL = None
_TASK_TIMEOUT_S = 300  # one window's heads take seconds; anything near this is a stuck pool


def _bf16_bits_to_f32(a):
    return (a.astype(np.uint16).astype(np.uint32) << 16).view(np.float32)


def _one_window_plan(n):
    # the window's rows, already gathered in packed order: one window [0, n)
    return types.SimpleNamespace(offsets=np.array([0, n], dtype=np.int64), ids=np.arange(n, dtype=np.int64),
                                 num_windows=1, num_tokens=n)


def _compare_window(task):
    """Worker: oracle output of every listed head of one window against the
    GPU output rows; returns (max |diff|, sum diff^2, sum ref^2, elements,
    head of the max)."""
    import oracle

    win, q, k, v, o, heads, scale = task
    q, k, v, o = (_bf16_bits_to_f32(x) for x in (q, k, v, o))
    n = q.shape[0]
    plan = _one_window_plan(n)
    rows = np.arange(n)
    worst, worst_head, ssd, ssr, count = 0.0, -1, 0.0, 0.0, 0
    for j, h in enumerate(heads):
        ref = oracle.window_attention_rows(q[:, j:j + 1, :], k[:, j:j + 1, :], v[:, j:j + 1, :], plan, 0, 0, rows,
                                           scale=scale)
        diff = o[:, j, :].astype(np.float64) - ref
        m = float(np.max(np.abs(diff)))
        if m > worst:
            worst, worst_head = m, int(h)
        ssd += float(np.sum(diff * diff))
        ssr += float(np.sum(ref * ref))
        count += diff.size
    return win, worst, ssd, ssr, count, worst_head


def _compare_text_window(task):
    """Worker: the oracle's [video window, text] segment attention of one
    window for every listed head; returns the video-row error sums (as
    _compare_window) and the window's text output T_w [n_text, heads, d]."""
    import oracle

    win, q, k, v, o, qt, kt, vt, heads, scale = task
    q, k, v, o, qt, kt, vt = (_bf16_bits_to_f32(x) for x in (q, k, v, o, qt, kt, vt))
    n = q.shape[0]
    plan = _one_window_plan(n)
    ref, t_w = oracle.window_attention_text(q, k, v, qt, kt, vt, plan, scale=scale)  # one window: T_w itself
    diff = o.astype(np.float64) - ref
    worst_head = int(heads[int(np.argmax(np.abs(diff).max(axis=(0, 2))))]) if diff.size else -1
    return (win, float(np.max(np.abs(diff))), float(np.sum(diff * diff)), float(np.sum(ref * ref)), diff.size,
            worst_head, t_w)


def pool():
    """The shared spawn pool (one single-threaded worker per usable core)."""
    global _POOL
    if _POOL is None:
        import multiprocessing as mp
        try:
            cores = len(os.sched_getaffinity(0))
        except AttributeError:
            cores = os.cpu_count() or 1
        saved = {key: os.environ.get(key) for key in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")}
        for key in saved:
            os.environ[key] = "1"  # inherited by the spawned workers only
        try:
            _POOL = mp.get_context("spawn").Pool(processes=max(1, cores))
            # a worker that cannot start would be respawned forever: fail fast instead
            _POOL.apply_async(os.getpid).get(timeout=_TASK_TIMEOUT_S)
        except Exception:
            if _POOL is not None:
                _POOL.terminate()
                _POOL = None
            raise
        finally:
            for key, val in saved.items():
                if val is None:
                    os.environ.pop(key, None)
                else:
                    os.environ[key] = val
    return _POOL


def close():
    global _POOL
    if _POOL is not None:
        _POOL.terminate()
        _POOL.join()
        _POOL = None


def _bits(t):
    """bf16 CPU tensor -> uint16 numpy view of its bits (no copy)."""
    import torch
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def compare_layer(q, k, v, o, plan, windows=None, heads=None, canonical=True, scale=None):
    """Compares the GPU output ``o`` of one layer with the oracle on the given
    windows (all by default) and heads (all by default).

    q, k, v, o: bf16 CPU tensors [N, heads, d] (rows canonical, or in the
    packed order of ``plan`` when canonical=False); plan: an oracle plan.
    Returns (max_abs, rel_rms, worst (window, head), elements compared), with
    rel_rms = sqrt(sum diff^2 / sum ref^2) over every compared element."""
    qb, kb, vb, ob = (_bits(t) for t in (q, k, v, o))
    all_heads = q.shape[1]
    hsel = np.arange(all_heads) if heads is None else np.asarray(heads)
    wsel = range(plan.num_windows) if windows is None else windows

    def tasks():
        for win in wsel:
            a, b = int(plan.offsets[win]), int(plan.offsets[win + 1])
            rows = plan.ids[a:b].astype(np.int64) if canonical else np.arange(a, b)
            yield (int(win), qb[rows][:, hsel], kb[rows][:, hsel], vb[rows][:, hsel], ob[rows][:, hsel],
                   [int(h) for h in hsel], scale)

    worst, where, ssd, ssr, count = 0.0, None, 0.0, 0.0, 0
    results = pool().imap_unordered(_compare_window, tasks(), chunksize=1)
    while True:
        try:
            win, m, d2, r2, c, h = results.next(timeout=_TASK_TIMEOUT_S)
        except StopIteration:
            break
        if where is None or m > worst:
            worst, where = m, (win, h)
        ssd += d2
        ssr += r2
        count += c
    rel = float(np.sqrt(ssd / max(ssr, 1e-300)))
    return worst, rel, where, count


def compare_text_layer(q, k, v, o, q_txt, k_txt, v_txt, o_txt, plan, scale=None):
    """The [video window, replicated text] layer (oracle.window_attention_text)
    compared in full: every video row of every window and head, and the text
    output T = (sum over windows of T_w) / W.  bf16 CPU tensors; canonical
    rows.  Returns ((video max_abs, rel_rms, worst (window, head)), (text
    max_abs, rel_rms))."""
    qb, kb, vb, ob = (_bits(t) for t in (q, k, v, o))
    tb = tuple(_bits(t) for t in (q_txt, k_txt, v_txt))
    heads = list(range(q.shape[1]))

    def tasks():
        for win in range(plan.num_windows):
            a, b = int(plan.offsets[win]), int(plan.offsets[win + 1])
            rows = plan.ids[a:b].astype(np.int64)
            yield (win, qb[rows], kb[rows], vb[rows], ob[rows], *tb, heads, scale)

    worst, where, ssd, ssr = 0.0, None, 0.0, 0.0
    t_sum = None
    results = pool().imap_unordered(_compare_text_window, tasks(), chunksize=1)
    while True:
        try:
            win, m, d2, r2, _, h, t_w = results.next(timeout=_TASK_TIMEOUT_S)
        except StopIteration:
            break
        if where is None or m > worst:
            worst, where = m, (win, h)
        ssd += d2
        ssr += r2
        t_sum = t_w if t_sum is None else t_sum + t_w
    t_ref = t_sum / plan.num_windows
    t_got = o_txt.float().numpy().astype(np.float64)
    t_diff = t_got - t_ref
    text = (float(np.max(np.abs(t_diff))), float(np.sqrt(np.sum(t_diff ** 2) / max(np.sum(t_ref ** 2), 1e-300))))
    return (worst, float(np.sqrt(ssd / max(ssr, 1e-300))), where), text

