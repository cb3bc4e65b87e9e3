"""Plan A on the device: wsa_gather_rows packs and unpacks, and the library's
schedule drives them ("Window-Aligned Sequence Parallelism (SeedVR2)",
section "Plan A redistribution").  The ranks are emulated in one process on
one GPU: each rank's pack runs, the all_to_all_single is replaced by slicing
the send buffers into receive buffers, and each rank unpacks.  Every rank
must hold exactly its destination rows; the expected rows come from the
oracle's rank-local orders.  Pure data movement: bit-exact."""

import numpy as np
import pytest
import torch

import oracle
import wsa_inputs
from oracle import sp as osp
from wsa_inputs import WORKLOADS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wsa():
    import shifted_window_attention_gb300 as m
    import shifted_window_attention_gb300.sp  # noqa: F401
    return m


def _grid(w):
    return (w.T, w.H, w.W, w.nt, w.nh, w.nw)


def _emulate(sp, grid, layouts, R, x):
    """Returns every rank's destination rows after pack / exchange / unpack."""
    plans = [sp.PlanA(*grid, *layouts, R, r) for r in range(R)]
    src = oracle.make_plan(*grid, layouts[0])
    locals_ = [x[torch.from_numpy(osp.local_rows(src, R, r)).to(x.device)] for r in range(R)]
    sends = [plans[r].pack(locals_[r]) for r in range(R)]
    bounds = [np.concatenate([[0], np.cumsum(p.input_split_sizes)]) for p in plans]
    outs = []
    for d in range(R):
        recv = torch.cat([sends[r][bounds[r][d]:bounds[r][d + 1]] for r in range(R)]).contiguous()
        outs.append(plans[d].unpack(recv))
    return outs, plans


@pytest.mark.parametrize("R", [2, 3, 8])
@pytest.mark.parametrize("layouts", [(0, 1), (1, 0)])
def test_emulated_exchange_720p_hidden(wsa, R, layouts):
    w = WORKLOADS["720p"]
    grid = _grid(w)
    x = wsa_inputs.activation(w, device="cuda")  # [N, 3072] bf16, canonical rows
    outs, plans = _emulate(wsa.sp, grid, layouts, R, x)
    dst = oracle.make_plan(*grid, layouts[1])
    for d in range(R):
        want = x[torch.from_numpy(osp.local_rows(dst, R, d)).cuda()]
        assert torch.equal(outs[d], want), f"rank {d}"
    assert plans[0].network_exchange_required


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("channels", [1, 3, 8, 130])
def test_emulated_exchange_ragged_channels(wsa, dtype, channels):
    grid = (7, 5, 11, 3, 2, 4)
    N = 7 * 5 * 11
    x = wsa_inputs.randn((N, channels), 31 + channels, "cuda").to(dtype)
    outs, _ = _emulate(wsa.sp, grid, (1, 0), 3, x)
    dst = oracle.make_plan(*grid, 0)
    for d in range(3):
        assert torch.equal(outs[d].cpu(), x.cpu()[torch.from_numpy(osp.local_rows(dst, 3, d))])


def test_one_rank_fast_path_equals_transition(wsa):
    # SP = 1: nothing crosses ranks; the exchange is the local permutation,
    # the same rows the layout transition produces.
    w = WORKLOADS["720p"]
    grid = _grid(w)
    src, dst = wsa.Plan(*grid, 0), wsa.Plan(*grid, 1)
    x = wsa_inputs.activation(w, device="cuda")
    ids_src = torch.from_numpy(oracle.make_plan(*grid, 0).ids.astype(np.int64)).cuda()
    x_src = x[ids_src].contiguous()
    pa = wsa.sp.PlanA(*grid, 0, 1, 1, 0)
    assert not pa.network_exchange_required
    assert torch.equal(pa.exchange(x_src), wsa.transition(src, dst, x_src))


def test_same_layout_exchange_is_identity(wsa):
    grid = (21, 45, 80, 4, 3, 3)
    for r in range(4):
        pa = wsa.sp.PlanA(*grid, 1, 1, 4, r)
        x = wsa_inputs.randn((pa.n_send, 64), 5 + r, "cuda").to(torch.bfloat16)
        assert torch.equal(pa.exchange(x), x)


def test_gather_rows_bounds_and_empty(wsa):
    x = wsa_inputs.randn((10, 8), 3, "cuda")
    idx = torch.tensor([9, 0, -1, 10, 4, 1 << 30], dtype=torch.int32, device="cuda")
    out = torch.full((6, 8), 7.0, device="cuda")
    wsa.gather_rows(x, idx, out=out)
    got, xc = out.cpu(), x.cpu()
    assert torch.equal(got[0], xc[9]) and torch.equal(got[1], xc[0]) and torch.equal(got[4], xc[4])
    for i in (2, 3, 5):  # outside [0, 10): row left unwritten
        assert torch.all(got[i] == 7.0)
    empty = wsa.gather_rows(x, torch.zeros(0, dtype=torch.int32, device="cuda"))
    assert empty.shape == (0, 8)
