"""Window-local 3D RoPE on the GPU (wsa_rope, wsa_rope_text) against the fp64
oracle ("Window-Aligned Sequence Parallelism (SeedVR2)", section "Reference
quirks reproduced on purpose"), then RoPE followed by window attention.

Tolerance of the rotation itself, from its arithmetic: the fp32 rotation is
rounded once to the output type.
- bf16: each element within 2^-8 |ref| + 1e-6 (one rounding is 2^-9 |ref|;
  the rest is margin for the fp32 sines and products).
- fp32: within 1e-5 (1 + |ref|).
Attention after RoPE uses the attention tolerances (bf16 max-abs 2e-2 and
rel-RMS 1e-2, fp32 max-abs 1e-4)."""

import numpy as np
import pytest
import torch

import oracle
import wsa_inputs
from oracle import rope as orope
from tests.helpers import assert_bf16_close, assert_fp32_close, to64
from wsa_inputs import WORKLOADS

pytestmark = pytest.mark.gpu

MID = wsa_inputs.custom(8, 24, 40, 2, 2, 2, heads=3, head_dim=128, name="mid")
TINY32 = wsa_inputs.custom(4, 9, 16, 2, 9, 16, heads=2, head_dim=64, dtype="fp32", name="tiny-fp32")


@pytest.fixture(scope="module")
def wsa():
    import shifted_window_attention_gb300 as m
    return m


def _grid(w):
    return (w.T, w.H, w.W, w.nt, w.nh, w.nw)


def _close_rot(got, ref, dtype, what):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    if dtype == torch.bfloat16:
        bound = 2.0 ** -8 * np.abs(ref) + 1e-6
    else:
        bound = 1e-5 * (1.0 + np.abs(ref))
    bad = np.abs(got - ref) > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} elements out of bound, worst {np.max(np.abs(got - ref)):.3e}"


@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("canonical", [True, False])
@pytest.mark.parametrize("text_len", [0, 77, 300])
def test_rope_bf16_mid(wsa, layout, canonical, text_len):
    w = MID
    p = wsa.Plan(*_grid(w), layout)
    op = oracle.make_plan(*_grid(w), layout)
    q, k, _ = wsa_inputs.qkv(w)
    if not canonical:
        ids = torch.from_numpy(op.ids.astype(np.int64))
        q, k = q[ids].contiguous(), k[ids].contiguous()
    qo, ko = wsa.rope(p, q.cuda(), k.cuda(), canonical=canonical, text_len=text_len)
    pos = orope.window_positions(op, text_len)
    if not canonical:
        pos = pos[op.ids]
    _close_rot(to64(qo), orope.apply_rope(to64(q), pos), torch.bfloat16, "q")
    _close_rot(to64(ko), orope.apply_rope(to64(k), pos), torch.bfloat16, "k")


@pytest.mark.parametrize("rope_dim", [60, 24])
def test_rope_fp32_head64(wsa, rope_dim):
    w = TINY32
    p = wsa.Plan(*_grid(w), 1)
    op = oracle.make_plan(*_grid(w), 1)
    q, k, _ = wsa_inputs.qkv(w)
    qo, ko = wsa.rope(p, q.cuda(), k.cuda(), text_len=5, rope_dim=rope_dim)
    pos = orope.window_positions(op, 5)
    _close_rot(to64(qo), orope.apply_rope(to64(q), pos, rope_dim=rope_dim), torch.float32, "q")
    _close_rot(to64(ko), orope.apply_rope(to64(k), pos, rope_dim=rope_dim), torch.float32, "k")
    assert torch.equal(qo[..., 3 * (rope_dim // 3):].cpu(), q[..., 3 * (rope_dim // 3):])


def test_rope_in_place_and_q_only(wsa):
    w = MID
    p = wsa.Plan(*_grid(w), 0)
    q, k, _ = (t.cuda() for t in wsa_inputs.qkv(w))
    ref_q, ref_k = wsa.rope(p, q, k, text_len=9)
    q2, k2 = q.clone(), k.clone()
    wsa.rope(p, q2, k2, q_out=q2, k_out=k2, text_len=9)
    assert torch.equal(q2, ref_q) and torch.equal(k2, ref_k)
    q_only, none = wsa.rope(p, q, text_len=9)
    assert none is None and torch.equal(q_only, ref_q)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_rope_text(wsa, dtype):
    n_text, heads = 300, 2
    qt = wsa_inputs.randn((n_text, heads, 128), 61, "cuda").to(dtype)
    kt = wsa_inputs.randn((n_text, heads, 128), 62, "cuda").to(dtype)
    qo, ko = wsa.rope_text(qt, kt)
    pos = orope.text_positions(n_text)
    _close_rot(to64(qo), orope.apply_rope(to64(qt), pos), dtype, "q_txt")
    _close_rot(to64(ko), orope.apply_rope(to64(kt), pos), dtype, "k_txt")


def test_rope_720p_sampled_rows(wsa):
    # full size, 24 heads, both layouts; rows sampled across every window
    w = WORKLOADS["720p"]
    q, k, _ = wsa_inputs.qkv(w, device="cuda")
    rng = np.random.default_rng(3)
    for layout in (0, 1):
        p = wsa.Plan(*_grid(w), layout)
        op = oracle.make_plan(*_grid(w), layout)
        qo, ko = wsa.rope(p, q, k, text_len=256)
        rows = np.unique(np.concatenate([op.ids[op.offsets[:-1]], op.ids[op.offsets[1:] - 1],
                                         rng.integers(0, w.num_tokens, 2000)]))
        pos = orope.window_positions(op, 256)[rows]
        idx = torch.from_numpy(rows).cuda()
        _close_rot(to64(qo[idx]), orope.apply_rope(to64(q[idx]), pos), torch.bfloat16, f"q L{layout}")
        _close_rot(to64(ko[idx]), orope.apply_rope(to64(k[idx]), pos), torch.bfloat16, f"k L{layout}")


@pytest.mark.parametrize("layout", [0, 1])
def test_rope_then_attention(wsa, layout):
    w = MID
    p = wsa.Plan(*_grid(w), layout)
    op = oracle.make_plan(*_grid(w), layout)
    q, k, v = (t.cuda() for t in wsa_inputs.qkv(w))
    qr, kr = wsa.rope(p, q, k, text_len=64)
    o = wsa.attention(p, qr, kr, v)
    pos = orope.window_positions(op, 64)
    ref = oracle.window_attention(orope.apply_rope(to64(q), pos), orope.apply_rope(to64(k), pos), to64(v), op)
    assert_bf16_close(to64(o), ref, f"rope + attention L{layout}")


def test_rope_then_text_attention(wsa):
    w, n_text = MID, 96
    p = wsa.Plan(*_grid(w), 1)
    op = oracle.make_plan(*_grid(w), 1)
    q, k, v = (t.cuda() for t in wsa_inputs.qkv(w))
    qt, kt, vt = (wsa_inputs.randn((n_text, w.heads, 128), 70 + j, "cuda").to(torch.bfloat16) for j in range(3))
    qr, kr = wsa.rope(p, q, k, text_len=n_text)
    qtr, ktr = wsa.rope_text(qt, kt)
    o, ot = wsa.attention_text(p, qr, kr, v, qtr, ktr, vt)
    pos, tpos = orope.window_positions(op, n_text), orope.text_positions(n_text)
    ref, ref_t = oracle.window_attention_text(orope.apply_rope(to64(q), pos), orope.apply_rope(to64(k), pos), to64(v),
                                              orope.apply_rope(to64(qt), tpos), orope.apply_rope(to64(kt), tpos),
                                              to64(vt), op)
    assert_bf16_close(to64(o), ref, "video rows")
    assert_bf16_close(to64(ot), ref_t, "text rows")


def test_rope_fp32_then_attention(wsa):
    w = TINY32
    p = wsa.Plan(*_grid(w), 0)
    op = oracle.make_plan(*_grid(w), 0)
    q, k, v = (t.cuda() for t in wsa_inputs.qkv(w))
    qr, kr = wsa.rope(p, q, k, rope_dim=60)
    o = wsa.attention(p, qr, kr, v)
    pos = orope.window_positions(op, 0)
    ref = oracle.window_attention(orope.apply_rope(to64(q), pos, rope_dim=60),
                                  orope.apply_rope(to64(k), pos, rope_dim=60), to64(v), op)
    assert_fp32_close(to64(o), ref, "fp32 rope + attention")


def test_rope_errors(wsa):
    w = TINY32
    p = wsa.Plan(*_grid(w), 0)
    q, k, _ = (t.cuda() for t in wsa_inputs.qkv(w))
    with pytest.raises(wsa.WsaError) as e:
        wsa.rope(p, q, k)  # head_dim 64 -> rope_dim 64 -> 21 channels per axis (odd)
    assert e.value.name == "WSA_ERR_UNSUPPORTED"
    with pytest.raises(wsa.WsaError) as e:
        wsa.rope(p, q, k, rope_dim=60, text_len=-1)
    assert e.value.name == "WSA_ERR_INVALID_ARG"
    big = torch.empty(2 * q.numel(), dtype=q.dtype, device="cuda")
    part = big[q.numel() // 2: q.numel() // 2 + q.numel()].view_as(q)  # overlaps q_out = big[:N]
    with pytest.raises(wsa.WsaError):
        wsa.rope(p, q, part, q_out=big[:q.numel()].view_as(q), k_out=part, rope_dim=60)
    assert wsa.lib.wsa_rope(p.handle, q.data_ptr(), k.data_ptr(), q.data_ptr(), None, 2, 64, 1, 1, 0, 60, 0.0,
                            None) == -1  # k without k_out
