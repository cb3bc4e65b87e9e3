"""GPU window attention over [video window, replicated text] segments against
the fp64 oracle ("Window-Aligned Sequence Parallelism (SeedVR2)", sections
"Text stream" and "SeedVR2 integration").  Tolerance: bf16 max-abs 2e-2 and
relative RMS 1e-2 on both the video rows and the window-averaged text rows."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import wsa_inputs
from tests import oracle_pool
from tests.helpers import BF16_MAX_ABS, BF16_REL_RMS, assert_bf16_close, to64
from wsa_inputs import WORKLOADS

pytestmark = pytest.mark.gpu

MID = wsa_inputs.custom(8, 24, 40, 2, 2, 2, heads=2, head_dim=128, name="mid")
TINY = wsa_inputs.custom(4, 9, 16, 2, 9, 16, heads=3, head_dim=128, name="tiny-bf16")


@pytest.fixture(scope="module")
def wsa():
    import shifted_window_attention_gb300 as m
    return m


def _grid(w):
    return (w.T, w.H, w.W, w.nt, w.nh, w.nw)


def _text(w, n_text, seed, device="cpu"):
    shape = (n_text, w.heads, w.head_dim)
    return tuple(wsa_inputs.randn(shape, seed + j, device).to(torch.bfloat16) for j in range(3))


@pytest.mark.parametrize("w", [TINY, MID], ids=lambda w: w.name)
@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("n_text", [1, 77, 300])
def test_text_segment_full_compare(wsa, w, layout, n_text):
    p = wsa.Plan(*_grid(w), layout)
    q, k, v = wsa_inputs.qkv(w)
    qt, kt, vt = _text(w, n_text, 500 + n_text)
    o, ot = wsa.attention_text(p, *(t.cuda() for t in (q, k, v, qt, kt, vt)))
    ref, ref_t = oracle.window_attention_text(to64(q), to64(k), to64(v), to64(qt), to64(kt), to64(vt),
                                              oracle.make_plan(*_grid(w), layout))
    assert_bf16_close(to64(o), ref, f"{w.name} L{layout} text {n_text} video rows")
    assert_bf16_close(to64(ot), ref_t, f"{w.name} L{layout} text {n_text} text rows")
    assert p.device_status() == 0


def test_packed_order_and_determinism(wsa):
    w, n_text = MID, 64
    p = wsa.Plan(*_grid(w), 1)
    q, k, v = wsa_inputs.qkv(w)
    qt, kt, vt = (t.cuda() for t in _text(w, n_text, 900))
    o, ot = wsa.attention_text(p, q.cuda(), k.cuda(), v.cuda(), qt, kt, vt)
    o2, ot2 = wsa.attention_text(p, q.cuda(), k.cuda(), v.cuda(), qt, kt, vt)
    assert torch.equal(o, o2) and torch.equal(ot, ot2)
    ids = torch.from_numpy(oracle.make_plan(*_grid(w), 1).ids.astype(np.int64))
    qp, kp, vp = (t[ids].contiguous().cuda() for t in (q, k, v))
    op, otp = wsa.attention_text(p, qp, kp, vp, qt, kt, vt, canonical=False)
    assert torch.equal(op.cpu(), o.cpu()[ids])
    assert torch.equal(otp, ot)


@pytest.mark.parametrize("layout", [0, 1])
def test_720p_text_every_window_and_head(wsa, layout):
    # Full-size grid with 256 text tokens: every video row of every window
    # and head, and every text row (the mean over all windows' text outputs)
    w = WORKLOADS["720p"]
    n_text = 256
    p = wsa.Plan(*_grid(w), layout)
    op = oracle.make_plan(*_grid(w), layout)
    q, k, v = wsa_inputs.qkv(w, layer=layout, device="cuda")
    qt, kt, vt = _text(w, n_text, 1300 + layout, device="cuda")
    o, ot = wsa.attention_text(p, q, k, v, qt, kt, vt)
    assert p.device_status() == 0
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(ot).all())
    (vmax, vrel, where), (tmax, trel) = oracle_pool.compare_text_layer(
        *(t.cpu() for t in (q, k, v, o, qt, kt, vt, ot)), op)
    print(f"720p text layout {layout}: video max-abs {vmax:.3e} at {where}, rel-RMS {vrel:.3e}; "
          f"text max-abs {tmax:.3e}, rel-RMS {trel:.3e}")
    assert vmax <= BF16_MAX_ABS and vrel <= BF16_REL_RMS, (vmax, vrel, where)
    assert tmax <= BF16_MAX_ABS and trel <= BF16_REL_RMS, (tmax, trel)


def test_text_errors(wsa):
    w = TINY
    p = wsa.Plan(*_grid(w), 0)
    q, k, v = (t.cuda() for t in wsa_inputs.qkv(w))
    qt, kt, vt = (t.cuda() for t in _text(w, 8, 70))
    need = wsa.attention_text_workspace_bytes(p, 8, w.heads)
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(wsa.WsaError) as e:
        wsa.attention_text(p, q, k, v, qt, kt, vt, workspace=ws)
    assert e.value.name == "WSA_ERR_INVALID_ARG"
    n = ctypes.c_size_t()
    assert wsa.lib.wsa_attention_text_workspace(p.handle, 8, w.heads, 128, 1, ctypes.byref(n)) == -2  # fp32
    assert wsa.lib.wsa_attention_text_workspace(p.handle, 0, w.heads, 128, 0, ctypes.byref(n)) == -1
    assert p.device_status() == 0
