"""The pooled full-size comparison (tests/oracle_pool.py) against the
single-process one: same maximum error and relative RMS on a grid the
oracle runs whole, and a planted error is found in the right window."""

import numpy as np
import torch

import oracle
import wsa_inputs
from tests import oracle_pool
from tests.helpers import errors

MID = wsa_inputs.custom(8, 24, 40, 2, 2, 2, heads=2, head_dim=128, name="mid")


def _grid(w):
    return (w.T, w.H, w.W, w.nt, w.nh, w.nw)


def test_pooled_errors_equal_the_plain_computation():
    w = MID
    for layout in (0, 1):
        q, k, v = wsa_inputs.qkv(w, layer=layout)
        p = oracle.make_plan(*_grid(w), layout)
        ref = oracle.window_attention(q.double().numpy(), k.double().numpy(), v.double().numpy(), p)
        o = torch.from_numpy(ref).to(torch.bfloat16)  # a stand-in output: the oracle rounded to bf16
        max_abs, rel_rms, _, count = oracle_pool.compare_layer(q, k, v, o, p)
        m2, r2 = errors(o.double().numpy(), ref)
        assert count == o.numel()
        assert np.isclose(max_abs, m2, rtol=0, atol=1e-12) and np.isclose(rel_rms, r2, rtol=1e-9)
        # packed rows give the same figures
        ids = torch.from_numpy(p.ids.astype(np.int64))
        packed = oracle_pool.compare_layer(q[ids], k[ids], v[ids], o[ids], p, canonical=False)
        assert np.isclose(packed[0], max_abs, rtol=0, atol=1e-12) and np.isclose(packed[1], rel_rms, rtol=1e-9)


def test_pooled_comparison_finds_a_planted_error():
    w = MID
    q, k, v = wsa_inputs.qkv(w, layer=1)
    p = oracle.make_plan(*_grid(w), 1)
    ref = oracle.window_attention(q.double().numpy(), k.double().numpy(), v.double().numpy(), p)
    o = torch.from_numpy(ref).to(torch.bfloat16)
    row = int(p.ids[p.offsets[5] + 3])
    o[row, 1, 9] += 0.25
    max_abs, _, where, _ = oracle_pool.compare_layer(q, k, v, o, p)
    assert max_abs > 0.2 and where == (5, 1)
    # a comparison that leaves that window out does not see it
    assert oracle_pool.compare_layer(q, k, v, o, p, windows=[4, 6])[0] < 0.02


def test_pooled_text_comparison_equals_the_plain_computation():
    # the text output is the mean over every window's text rows: the pooled
    # per-window sums must reproduce the oracle's whole-layer result
    w = wsa_inputs.custom(4, 9, 16, 2, 9, 16, heads=2, head_dim=128, name="tiny-bf16")
    p = oracle.make_plan(*_grid(w), 1)
    q, k, v = wsa_inputs.qkv(w)
    qt, kt, vt = (wsa_inputs.randn((20, 2, 128), 77 + j).to(torch.bfloat16) for j in range(3))
    ref, ref_t = oracle.window_attention_text(*(t.double().numpy() for t in (q, k, v, qt, kt, vt)), p)
    o, ot = torch.from_numpy(ref).to(torch.bfloat16), torch.from_numpy(ref_t).to(torch.bfloat16)
    (vmax, vrel, _), (tmax, trel) = oracle_pool.compare_text_layer(q, k, v, o, qt, kt, vt, ot, p)
    assert np.isclose(vmax, errors(o.double().numpy(), ref)[0], rtol=0, atol=1e-12)
    assert np.isclose(tmax, errors(ot.double().numpy(), ref_t)[0], rtol=0, atol=1e-12)
    assert np.isclose(trel, errors(ot.double().numpy(), ref_t)[1], rtol=1e-9)
    ot2 = ot.clone()
    ot2[3, 1, 5] += 0.5
    assert oracle_pool.compare_text_layer(q, k, v, o, qt, kt, vt, ot2, p)[1][0] > 0.4
