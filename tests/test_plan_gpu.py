"""GPU plans against the oracle, bit for bit: offsets, window boxes, ids, pos
("Window-Aligned Sequence Parallelism (SeedVR2)", section "Window layouts")."""

import numpy as np
import pytest
import torch

import oracle
from wsa_inputs import WORKLOADS

pytestmark = pytest.mark.gpu

GRIDS = [(w.T, w.H, w.W, w.nt, w.nh, w.nw) for w in WORKLOADS.values()] + [
    (1, 1, 1, 1, 1, 1), (2, 3, 4, 2, 52, 69), (7, 5, 11, 3, 2, 4), (40, 12, 30, 9, 4, 5),
    (3, 6, 10, 1, 1, 1), (64, 90, 160, 4, 3, 3),
]


@pytest.fixture(scope="module")
def wsa():
    import shifted_window_attention_gb300 as m
    return m


@pytest.mark.parametrize("grid", GRIDS)
@pytest.mark.parametrize("layout", [0, 1])
def test_tables_bit_exact(wsa, grid, layout):
    ref = oracle.make_plan(*grid, layout)
    p = wsa.Plan(*grid, layout)
    assert (p.wt, p.wh, p.ww) == (ref.wt, ref.wh, ref.ww)
    assert p.num_windows == ref.num_windows and p.num_tokens == ref.num_tokens
    assert p.max_window_tokens == ref.max_window_tokens
    offsets, dims, ids, pos = (t.cpu().numpy() for t in p.tables())
    assert np.array_equal(offsets, ref.offsets)
    assert np.array_equal(dims.reshape(-1, 6), ref.dims)
    assert np.array_equal(ids, ref.ids)
    assert np.array_equal(pos, ref.pos)
    assert p.device_status() == 0
    p.destroy()


def test_plan_on_side_stream(wsa):
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        p = wsa.Plan(21, 45, 80, 4, 3, 3, 1, stream=s)
        ids = p.tables()[2].clone()
    s.synchronize()
    assert np.array_equal(ids.cpu().numpy(), oracle.make_plan(21, 45, 80, 4, 3, 3, 1).ids)


def test_invalid_plan_arguments(wsa):
    for bad in [(0, 9, 16, 2, 9, 16, 0), (4, 9, 16, 2, 9, 16, 5), (1, 1, 100000, 1, 1, 1, 0)]:
        with pytest.raises(wsa.WsaError) as e:
            wsa.Plan(*bad)
        assert e.value.name == "WSA_ERR_INVALID_ARG"
