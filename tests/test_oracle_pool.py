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
