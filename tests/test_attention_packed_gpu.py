"""Window attention on rows in plan-packed order ("Window-Aligned Sequence
Parallelism (SeedVR2)", section "Motivation": attention only inside a window;
the packed order is the one the layout transition produces).

Full 128-row tiles of packed rows reach the tensor-core kernel by TMA tile
loads, a window's last partial tile by the zero-filling gather.  The tile
contents are the same as in canonical order, so packed and canonical outputs
must agree bit for bit; the oracle checks both within the bf16 tolerance
(max-abs 2e-2, relative RMS 1e-2)."""

import numpy as np
import pytest
import torch

import oracle
import wsa_inputs
from tests.helpers import assert_bf16_close, to64
from wsa_inputs import WORKLOADS

pytestmark = pytest.mark.gpu

# every regular window a whole number of 128-row tiles (1024..1920 rows): all TMA
WHOLE_TILES = wsa_inputs.custom(8, 44, 76, 1, 4, 4, heads=2, head_dim=128, name="whole-tiles")
MID = wsa_inputs.custom(8, 24, 40, 2, 2, 2, heads=2, head_dim=128, name="mid")
SMALL = wsa_inputs.custom(4, 9, 16, 2, 9, 16, heads=3, head_dim=128, name="tiny-bf16")  # 4..50 rows: no TMA tile


@pytest.fixture(scope="module")
def wsa():
    import shifted_window_attention_gb300 as m
    return m


def _grid(w):
    return (w.T, w.H, w.W, w.nt, w.nh, w.nw)


def _packed(t, ids):
    return t[ids].contiguous()


def test_whole_tile_grid_is_all_whole_tiles():
    op = oracle.make_plan(*_grid(WHOLE_TILES), 0)
    sizes = np.diff(op.offsets)
    assert np.all(sizes % 128 == 0) and op.num_windows == 16


@pytest.mark.parametrize("w", [SMALL, MID, WHOLE_TILES], ids=lambda w: w.name)
@pytest.mark.parametrize("layout", [0, 1])
def test_packed_matches_oracle_and_canonical(wsa, w, layout):
    g = _grid(w)
    p = wsa.Plan(*g, layout)
    op = oracle.make_plan(*g, layout)
    q, k, v = wsa_inputs.qkv(w, device="cuda")
    ids = torch.from_numpy(op.ids.astype(np.int64)).cuda()
    o_can = wsa.attention(p, q, k, v)
    o_pk = torch.full_like(q, float("nan"))
    wsa.attention(p, _packed(q, ids), _packed(k, ids), _packed(v, ids), out=o_pk, canonical=False)
    assert p.device_status() == 0
    assert torch.equal(o_pk, o_can[ids])
    ref = oracle.window_attention(to64(q), to64(k), to64(v), op)[op.ids]
    assert_bf16_close(to64(o_pk), ref, f"{w.name} packed layout {layout}")


@pytest.mark.parametrize("name", ["720p", "1080p", "long"])
@pytest.mark.parametrize("layout", [0, 1])
def test_full_size_packed_bit_identical(wsa, name, layout):
    # The launch configuration of the packed-order bench leg, full size: the
    # packed output is the canonical output permuted, bit for bit, and sampled
    # (window, head) problems agree with the oracle.
    w = WORKLOADS[name]
    g = _grid(w)
    p = wsa.Plan(*g, layout)
    op = oracle.make_plan(*g, layout)
    q, k, v = wsa_inputs.qkv(w, device="cuda")
    ids = torch.from_numpy(op.ids.astype(np.int64)).cuda()
    o_can = wsa.attention(p, q, k, v)
    qp, kp, vp = _packed(q, ids), _packed(k, ids), _packed(v, ids)
    o_pk = torch.full_like(q, float("nan"))
    wsa.attention(p, qp, kp, vp, out=o_pk, canonical=False)
    assert p.device_status() == 0
    assert torch.equal(o_pk, o_can[ids])
    qn, kn, vn = (t.float().cpu().numpy() for t in (q, k, v))
    on = o_pk.float().cpu().numpy()
    n = np.diff(op.offsets)
    rng = np.random.default_rng(7 + layout)
    for win in sorted({int(np.argmin(n)), int(np.argmax(n)), op.num_windows - 1}):
        h = int(rng.integers(w.heads))
        ref = oracle.window_attention_rows(qn, kn, vn, op, win, h, np.arange(n[win]))
        assert_bf16_close(on[op.offsets[win]:op.offsets[win + 1], h, :], ref, f"{name} packed win {win} head {h}")


def test_neighbour_rows_never_enter_a_tile(wsa):
    # Non-finite values in one window's packed rows leave every other window's
    # output finite and bit-identical: the partial last tile of the window
    # before it is zero-filled, not read past its end.
    w = MID
    g = _grid(w)
    p = wsa.Plan(*g, 1)
    op = oracle.make_plan(*g, 1)
    q, k, v = wsa_inputs.qkv(w, device="cuda")
    ids = torch.from_numpy(op.ids.astype(np.int64)).cuda()
    qp, kp, vp = _packed(q, ids), _packed(k, ids), _packed(v, ids)
    sizes = np.diff(op.offsets)
    # a window whose predecessor ends in a partial tile
    win = next(i for i in range(1, op.num_windows) if sizes[i - 1] % 128 != 0)
    lo, hi = int(op.offsets[win]), int(op.offsets[win + 1])
    o_ref = wsa.attention(p, qp, kp, vp, canonical=False)
    q2, k2, v2 = qp.clone(), kp.clone(), vp.clone()
    q2[lo:hi] = float("nan")
    k2[lo:hi] = float("inf")
    v2[lo:hi] = float("nan")
    o2 = wsa.attention(p, q2, k2, v2, canonical=False)
    assert p.device_status() == 0
    keep = torch.ones(w.num_tokens, dtype=torch.bool, device="cuda")
    keep[lo:hi] = False
    assert bool(torch.isfinite(o2[keep]).all())
    assert torch.equal(o2[keep], o_ref[keep])


@pytest.mark.parametrize("heads", [1, 5])
def test_packed_head_counts(wsa, heads):
    # The tile maps' row stride is heads x 256 bytes: one head (rows back to
    # back) and an odd count; whole-tile windows so that every tile is a TMA tile.
    w = wsa_inputs.custom(8, 44, 76, 1, 4, 4, heads=heads, head_dim=128, name=f"whole-tiles-{heads}h")
    g = _grid(w)
    p = wsa.Plan(*g, 0)
    op = oracle.make_plan(*g, 0)
    q, k, v = wsa_inputs.qkv(w, device="cuda")
    ids = torch.from_numpy(op.ids.astype(np.int64)).cuda()
    o_can = wsa.attention(p, q, k, v)
    o_pk = wsa.attention(p, _packed(q, ids), _packed(k, ids), _packed(v, ids), canonical=False)
    assert p.device_status() == 0
    assert torch.equal(o_pk, o_can[ids])
    qn, kn, vn = (t.float().cpu().numpy() for t in (q, k, v))
    on = o_pk.float().cpu().numpy()
    for win in (0, op.num_windows - 1):
        n = int(op.offsets[win + 1] - op.offsets[win])
        ref = oracle.window_attention_rows(qn, kn, vn, op, win, heads - 1, np.arange(n))
        assert_bf16_close(on[op.offsets[win]:op.offsets[win + 1], heads - 1, :], ref, f"{heads} heads win {win}")


def test_single_full_tile_window(wsa):
    # A grid whose one window is exactly one 128-row tile: Q, K and V all by TMA.
    w = wsa_inputs.custom(2, 8, 8, 1, 1, 1, heads=2, head_dim=128, name="one-tile")
    g = _grid(w)
    p = wsa.Plan(*g, 0)
    assert p.num_windows == 1 and p.num_tokens == 128
    op = oracle.make_plan(*g, 0)
    q, k, v = wsa_inputs.qkv(w, device="cuda")
    ids = torch.from_numpy(op.ids.astype(np.int64)).cuda()
    o_pk = wsa.attention(p, _packed(q, ids), _packed(k, ids), _packed(v, ids), canonical=False)
    assert p.device_status() == 0
    ref = oracle.window_attention(to64(q), to64(k), to64(v), op)[op.ids]
    assert_bf16_close(to64(o_pk), ref, "one full tile")
