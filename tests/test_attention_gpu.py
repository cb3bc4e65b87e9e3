"""GPU window attention against the fp64 oracle ("Window-Aligned Sequence
Parallelism (SeedVR2)", section "Motivation": attention only inside a window).

Tolerances: bf16 max-abs 2e-2 and relative RMS 1e-2; fp32 max-abs 1e-4."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import wsa_inputs
from tests import oracle_pool
from tests.helpers import BF16_MAX_ABS, BF16_REL_RMS, assert_bf16_close, assert_fp32_close, to64
from wsa_inputs import WORKLOADS

pytestmark = pytest.mark.gpu

MID = wsa_inputs.custom(8, 24, 40, 2, 2, 2, heads=2, head_dim=128, name="mid")          # windows up to 3588 tokens
SMALL_BF16 = wsa_inputs.custom(4, 9, 16, 2, 9, 16, heads=3, head_dim=128, name="tiny-bf16")  # 4..50-token windows
ONE_TOKEN = wsa_inputs.custom(2, 3, 4, 2, 52, 69, heads=2, head_dim=128, name="one-token")


@pytest.fixture(scope="module")
def wsa():
    import shifted_window_attention_gb300 as m
    return m


def _grid(w):
    return (w.T, w.H, w.W, w.nt, w.nh, w.nw)


def _run(wsa, w, layout, dtype=None, layer=0, canonical=True):
    p = wsa.Plan(*_grid(w), layout)
    q, k, v = wsa_inputs.qkv(w, layer=layer)
    if dtype is not None:
        q, k, v = (t.to(dtype) for t in (q, k, v))
    qg, kg, vg = (t.cuda() for t in (q, k, v))
    o = wsa.attention(p, qg, kg, vg, canonical=canonical)
    return p, (q, k, v), o


@pytest.mark.parametrize("layout", [0, 1])
def test_fp32_tiny_full(wsa, layout):
    w = WORKLOADS["tiny"]
    p, (q, k, v), o = _run(wsa, w, layout)
    ref = oracle.window_attention(to64(q), to64(k), to64(v), oracle.make_plan(*_grid(w), layout))
    assert_fp32_close(to64(o), ref, f"fp32 tiny layout {layout}")
    assert p.device_status() == 0


def test_fp32_head_dim_128(wsa):
    w = wsa_inputs.custom(5, 10, 12, 2, 4, 4, heads=2, head_dim=128, dtype="fp32", name="fp32-128")
    p, (q, k, v), o = _run(wsa, w, 1)
    ref = oracle.window_attention(to64(q), to64(k), to64(v), oracle.make_plan(*_grid(w), 1))
    assert_fp32_close(to64(o), ref, "fp32 d128")


@pytest.mark.parametrize("w", [SMALL_BF16, MID], ids=lambda w: w.name)
@pytest.mark.parametrize("layout", [0, 1])
def test_bf16_full_compare(wsa, w, layout):
    p, (q, k, v), o = _run(wsa, w, layout)
    ref = oracle.window_attention(to64(q), to64(k), to64(v), oracle.make_plan(*_grid(w), layout))
    assert_bf16_close(to64(o), ref, f"{w.name} layout {layout}")
    assert p.device_status() == 0


def test_packed_order_matches_canonical(wsa):
    w = MID
    p, (q, k, v), o = _run(wsa, w, 1)
    ids = torch.from_numpy(oracle.make_plan(*_grid(w), 1).ids.astype(np.int64))
    qp, kp, vp = (t[ids].contiguous().cuda() for t in (q, k, v))
    op = wsa.attention(p, qp, kp, vp, canonical=False)
    assert torch.equal(op.cpu(), o.cpu()[ids])


def test_output_16_byte_aligned_only(wsa):
    # an output that is 16- but not 32-byte aligned takes the 16-byte store
    # path; it must write exactly what the 32-byte path writes
    w = MID
    p = wsa.Plan(*_grid(w), 1)
    q, k, v = (t.cuda() for t in wsa_inputs.qkv(w, layer=5))
    expect = wsa.attention(p, q, k, v)
    buf = torch.full((q.numel() + 8,), float("nan"), dtype=q.dtype, device="cuda")
    out = buf[8:].view(q.shape)  # 16 bytes past a 256-byte aligned base
    assert out.data_ptr() % 32 == 16
    wsa.attention(p, q, k, v, out=out)
    torch.cuda.synchronize()
    assert torch.equal(out, expect)
    assert bool(torch.isnan(buf[:8]).all())


def test_repeat_calls_identical(wsa):
    w = MID
    p, (q, k, v), o = _run(wsa, w, 0)
    qg, kg, vg = (t.cuda() for t in (q, k, v))
    for _ in range(3):
        o2 = wsa.attention(p, qg, kg, vg)
        assert torch.equal(o2, o)
    assert p.device_status() == 0


def test_isolation(wsa):
    # Perturb one window's inputs: every other window's output stays bit-identical.
    w = MID
    p, (q, k, v), o = _run(wsa, w, 1)
    op = oracle.make_plan(*_grid(w), 1)
    win = op.num_windows // 2
    rows = torch.from_numpy(op.ids[op.offsets[win]:op.offsets[win + 1]].astype(np.int64))
    q2, k2, v2 = q.clone(), k.clone(), v.clone()
    q2[rows] = -q2[rows]
    k2[rows] = k2[rows] * 2
    v2[rows] = v2[rows] + 1
    o2 = wsa.attention(p, q2.cuda(), k2.cuda(), v2.cuda()).cpu()
    mask = torch.ones(w.num_tokens, dtype=torch.bool)
    mask[rows] = False
    assert torch.equal(o2[mask], o.cpu()[mask])
    assert not torch.equal(o2[rows], o.cpu()[rows])


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_one_token_windows_give_v(wsa, dtype):
    w = ONE_TOKEN
    p, (q, k, v), o = _run(wsa, w, 0, dtype=dtype)
    assert p.num_windows == w.num_tokens
    assert torch.equal(o.cpu(), v)


def test_constant_keys_mean_of_values(wsa):
    w = MID
    p = wsa.Plan(*_grid(w), 1)
    q, k, v = wsa_inputs.qkv(w)
    k = torch.full_like(k, 0.25)
    o = wsa.attention(p, q.cuda(), k.cuda(), v.cuda())
    ref = oracle.window_attention(to64(q), to64(k), to64(v), oracle.make_plan(*_grid(w), 1))
    assert_bf16_close(to64(o), ref, "constant keys")


def _sample_windows(op, count, seed):
    n = np.diff(op.offsets)
    rng = np.random.default_rng(seed)
    picks = {int(np.argmin(n)), int(np.argmax(n)), 0, op.num_windows - 1}
    picks |= set(int(x) for x in rng.choice(op.num_windows, size=min(count, op.num_windows), replace=False))
    return sorted(picks)


def _full_layer(wsa, w, layout, layer=0, windows=None, heads=None):
    """One layer on the GPU (canonical rows), compared with the fp64 oracle on
    every element of the given windows and heads (all by default).  Prints
    and returns (max_abs, rel_rms)."""
    g = _grid(w)
    p = wsa.Plan(*g, layout)
    q, k, v = wsa_inputs.qkv(w, layer=layer, device="cuda")
    o = torch.full_like(q, float("nan"))
    wsa.attention(p, q, k, v, out=o)
    assert p.device_status() == 0
    # every output row of every head was written and is finite
    assert bool(torch.isfinite(o).all())
    q, k, v, o = (t.cpu() for t in (q, k, v, o))
    op = oracle.make_plan(*g, layout)
    max_abs, rel_rms, where, count = oracle_pool.compare_layer(q, k, v, o, op, windows=windows, heads=heads)
    what = (f"{w.name} layer {layer} ({'shifted' if layout else 'regular'}), "
            f"{'all' if windows is None else len(windows)} windows x {'all' if heads is None else len(heads)} heads")
    print(f"{what}: {count} elements, max-abs {max_abs:.3e} (worst window, head {where}), rel-RMS {rel_rms:.3e}")
    assert max_abs <= BF16_MAX_ABS and rel_rms <= BF16_REL_RMS, (
        f"{what}: max_abs={max_abs:.3e} (<= {BF16_MAX_ABS}) at {where}, rel_rms={rel_rms:.3e} (<= {BF16_REL_RMS})")
    return max_abs, rel_rms


@pytest.mark.parametrize("name", ["720p", "1080p", "long"])
@pytest.mark.parametrize("layout", [0, 1])
def test_every_window_and_head(wsa, name, layout):
    # the two-layer workloads compared in full: every output element of both
    # layouts (every window, all 24 heads) against the fp64 oracle
    _full_layer(wsa, WORKLOADS[name], layout)


@pytest.mark.parametrize("layer", [0, 1])
def test_32layer_first_layers_every_window_and_head(wsa, layer):
    # the 302,400-token grid: layers 0 (regular) and 1 (shifted) in full
    w = WORKLOADS["32layer"]
    _full_layer(wsa, w, layer % 2, layer=layer)


@pytest.mark.parametrize("layer", [2, 13, 30, 31])
def test_32layer_later_layers_sampled(wsa, layer):
    # later layers of the alternating schedule (fresh Q/K/V per layer): a
    # seeded sample of 8 windows plus the smallest and largest, all heads
    w = WORKLOADS["32layer"]
    op = oracle.make_plan(*_grid(w), layer % 2)
    _full_layer(wsa, w, layer % 2, layer=layer, windows=_sample_windows(op, 8, 100 + layer))


def test_argument_errors(wsa):
    w = SMALL_BF16
    p = wsa.Plan(*_grid(w), 0)
    q = torch.zeros(w.num_tokens, 2, 64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(wsa.WsaError) as e:
        wsa.attention(p, q, q.clone(), q.clone())
    assert e.value.name == "WSA_ERR_UNSUPPORTED"
    q = torch.zeros(w.num_tokens * 2 * 128 + 8, device="cuda", dtype=torch.bfloat16)
    qv = q[1:1 + w.num_tokens * 2 * 128]
    st = wsa.lib.wsa_attention(p.handle, ctypes.c_void_p(qv.data_ptr()), ctypes.c_void_p(qv.data_ptr()),
                               ctypes.c_void_p(qv.data_ptr()), ctypes.c_void_p(q.data_ptr() + 64), 2, 128, 0, 1,
                               0.0, None)
    assert st == -1  # misaligned
    x = torch.zeros(w.num_tokens, 2, 128, device="cuda", dtype=torch.bfloat16)
    st = wsa.lib.wsa_attention(p.handle, ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(x.data_ptr()),
                               ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(x.data_ptr()), 2, 128, 0, 1, 0.0, None)
    assert st == -1  # output aliases input
    with pytest.raises(wsa.WsaError):
        wsa.attention(p, x[:-1].contiguous(), x[:-1].contiguous(), x[:-1].contiguous())
    assert p.device_status() == 0


@pytest.mark.parametrize("scale", [0.02, 0.3])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_explicit_softmax_scale(wsa, scale, dtype):
    # softmax_scale > 0 replaces 1/sqrt(d).  0.3 is about 3.4x the default for
    # d = 128: peaked rows whose running max jumps, so the lazy rescale of O runs.
    if dtype == "bf16":
        w = MID
    else:
        w = wsa_inputs.custom(5, 10, 12, 2, 4, 4, heads=2, head_dim=128, dtype="fp32", name="fp32-128")
    p = wsa.Plan(*_grid(w), 1)
    q, k, v = wsa_inputs.qkv(w)
    o = wsa.attention(p, q.cuda(), k.cuda(), v.cuda(), scale=scale)
    assert p.device_status() == 0
    ref = oracle.window_attention(to64(q), to64(k), to64(v), oracle.make_plan(*_grid(w), 1), scale=scale)
    if dtype == "bf16":
        assert_bf16_close(to64(o), ref, f"bf16 scale {scale}")
    else:
        assert_fp32_close(to64(o), ref, f"fp32 scale {scale}")


# The kernel's lazy-rescale threshold in log2 units: O is rescaled only when a
# row max grows by more than this; below it the probabilities reach 2^64.
LAZY_RESCALE_LOG2 = 64


@pytest.mark.parametrize("gain", [8, 20], ids=["large-p-no-rescale", "rescale"])
@pytest.mark.parametrize("canonical", [True, False], ids=["canonical", "packed"])
def test_lazy_rescale_path(wsa, canonical, gain):
    # Keys after the first 128 packed rows of every window are scaled by
    # `gain`, so the row maxima of later key tiles exceed the first tile's.
    # gain 8: most rows' max (log2 domain) grows by 24-64, under the
    # threshold, so probabilities up to about 2^60 enter P, the sums and O
    # unrescaled.  gain 20: most rows grow by more than 64 (up to about 156,
    # where the rescale factor flushes to zero) and rescale O in TMEM.
    w = MID
    g = _grid(w)
    p = wsa.Plan(*g, 0)
    op = oracle.make_plan(*g, 0)
    q, k, v = wsa_inputs.qkv(w)
    scale = torch.ones(w.num_tokens)
    for win in range(op.num_windows):
        rows = op.ids[op.offsets[win] + 128:op.offsets[win + 1]].astype(np.int64)
        scale[torch.from_numpy(rows)] = float(gain)
    k = (k.float() * scale[:, None, None]).to(k.dtype)
    c = np.log2(np.e) / np.sqrt(128.0)
    growth = []
    for win in range(op.num_windows):
        rows = op.ids[op.offsets[win]:op.offsets[win + 1]].astype(np.int64)
        s = to64(q[rows, 0]) @ to64(k[rows, 0]).T * c
        growth.append(s.max(axis=1) - s[:, :128].max(axis=1))
    growth = np.concatenate(growth)
    if gain == 8:
        assert np.mean((growth > 24) & (growth <= LAZY_RESCALE_LOG2)) > 0.9
    else:
        assert np.mean(growth > LAZY_RESCALE_LOG2) > 0.9
    ref = oracle.window_attention(to64(q), to64(k), to64(v), op)
    ids = torch.from_numpy(op.ids.astype(np.int64))
    if canonical:
        o = wsa.attention(p, q.cuda(), k.cuda(), v.cuda())
        got = to64(o)
    else:
        o = wsa.attention(p, q[ids].contiguous().cuda(), k[ids].contiguous().cuda(), v[ids].contiguous().cuda(),
                          canonical=False)
        got = to64(o)[np.argsort(op.ids)]
    assert p.device_status() == 0
    assert_bf16_close(got, ref, f"lazy rescale, gain {gain} ({'canonical' if canonical else 'packed'})")
