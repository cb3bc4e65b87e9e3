"""The 32-layer alternating schedule run as one chain on the GPU.

"Window-Aligned Sequence Parallelism (SeedVR2)", sections "Motivation" and
"Window layouts": regular and shifted layouts alternate at every layer of the
32-layer model, so the hidden state goes through 31 layout transitions, and
ensure_layout(current, required) derives each one from the layer schedule.
Section "SeedVR2 integration": the runtime owns the entry distribution into
the first layer's packed order and the final reconstruction back to
canonical token order, and attention is a packed call over each window's rows.

The chain here has no weights.  The hidden state h [N, 3072] enters layer 0's
packed order by a gather through that plan's ids table; before every later
layer, ensure_layout moves it into the layer's packed order.  Each layer
attends with fresh seeded Q and K and V = h + Z, Z fresh seeded noise (Q, K
and Z put into the layer's packed order on the test side; the add is
tokenwise, so it runs in packed order, as the note says of the residual and
MLP), on packed rows (full tiles by TMA); the attention output is the next
layer's h.  So every layer's attention consumes rows that the previous
transition produced, while the values stay of order one (a plain residual
h + O would double each window's mean every layer and push the outputs to
magnitudes where bf16 rounding alone exceeds the absolute tolerance).

Checks: every transition against the oracle's gather table (bit for bit);
layers 0, 1, 15 and 31 against the fp64 oracle on a seeded sample of windows
(all heads), given the same input rows; the final reconstruction through pos
against the oracle's ids.
"""

import numpy as np
import pytest
import torch

import oracle
import wsa_inputs
from tests import oracle_pool
from tests.helpers import BF16_MAX_ABS, BF16_REL_RMS
from wsa_inputs import WORKLOADS

pytestmark = pytest.mark.gpu

CHECKED_LAYERS = (0, 1, 15, 31)


def _sample_windows(op, count, seed):
    n = np.diff(op.offsets)
    rng = np.random.default_rng(seed)
    picks = {int(np.argmin(n)), int(np.argmax(n))}
    picks |= set(int(x) for x in rng.choice(op.num_windows, size=min(count, op.num_windows), replace=False))
    return sorted(picks)


def test_32layer_chain_through_transitions():
    import shifted_window_attention_gb300 as wsa

    w = WORKLOADS["32layer"]
    g = (w.T, w.H, w.W, w.nt, w.nh, w.nw)
    N, heads, d = w.num_tokens, w.heads, w.head_dim
    C = heads * d
    # the model's layer list: NaDiT alternates the two window methods
    layer_layouts = [(wsa.REGULAR, wsa.SHIFTED)[l % 2] for l in range(w.layers)]
    plans = {lay: wsa.Plan(*g, lay) for lay in set(layer_layouts)}
    oplans = {lay: oracle.make_plan(*g, lay) for lay in set(layer_layouts)}
    ids_dev = {lay: torch.from_numpy(oplans[lay].ids.astype(np.int64)).cuda() for lay in oplans}
    gather = {(a, b): torch.from_numpy(oracle.gather_table(oplans[a], oplans[b])).cuda()
              for a in oplans for b in oplans if a != b}

    # entry distribution: canonical rows -> packed order of layer 0's layout
    x = wsa_inputs.activation(w, device="cuda")
    cur = layer_layouts[0]
    h = wsa.gather_rows(x, plans[cur].tables()[2])
    assert torch.equal(h, x[ids_dev[cur]])

    moves = 0
    for l, req in enumerate(layer_layouts):
        prev = h
        h = wsa.ensure_layout(plans[cur], plans[req], h)
        if h is not prev:
            moves += 1
            assert torch.equal(h, prev[gather[(cur, req)]]), f"transition before layer {l}"
        else:
            assert req == cur
        cur = req
        q_c, k_c, z_c = wsa_inputs.qkv(w, layer=l, device="cuda")
        q = q_c[ids_dev[cur]].contiguous()
        k = k_c[ids_dev[cur]].contiguous()
        v = (h.view(N, heads, d).float() + z_c[ids_dev[cur]].float()).to(torch.bfloat16)
        o = wsa.attention(plans[cur], q, k, v, canonical=False)
        if l in CHECKED_LAYERS:
            assert plans[cur].device_status() == 0
            wins = _sample_windows(oplans[cur], 8, 500 + l)
            max_abs, rel_rms, where, count = oracle_pool.compare_layer(
                q.cpu(), k.cpu(), v.cpu(), o.cpu(), oplans[cur], windows=wins, canonical=False)
            print(f"chain layer {l}: {len(wins)} windows x {heads} heads, {count} elements, "
                  f"max-abs {max_abs:.3e} at {where}, rel-RMS {rel_rms:.3e}")
            assert max_abs <= BF16_MAX_ABS and rel_rms <= BF16_REL_RMS, f"layer {l}: {max_abs:.3e}, {rel_rms:.3e}"
        h = o.view(N, C)
    assert moves == w.layers - 1 == 31
    for p in plans.values():
        assert p.device_status() == 0

    # final reconstruction back to canonical token order through pos
    out = wsa.gather_rows(h, plans[cur].tables()[3])
    assert torch.equal(out[ids_dev[cur]], h)
    assert bool(torch.isfinite(out.float()).all())
