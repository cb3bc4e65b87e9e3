"""The allocation-free attention entry point, wsa_attention_noalloc.

It serves callers that cannot call cudaMalloc -- device memory owned by
another framework's pool, or serving loops that must not take the
device-wide synchronisation of cudaMalloc/cudaFree -- and therefore cannot
create a plan.  It runs the same kernels as the plan-based wsa_attention on
tables it builds in the library's fixed scratch array, so its output must be
bit-identical to wsa_attention's, on consecutive calls that reuse the array,
and within the bf16 tolerance of the fp64 oracle.

This file is collected last so that a run stopping at the first failure has
already run every other test."""

import ctypes

import numpy as np
import pytest
import torch

import oracle
import wsa_inputs
from tests.helpers import assert_bf16_close, to64
from wsa_inputs import WORKLOADS

pytestmark = pytest.mark.gpu

MID = wsa_inputs.custom(8, 24, 40, 2, 2, 2, heads=2, head_dim=128, name="mid")


def _grid(w):
    return (w.T, w.H, w.W, w.nt, w.nh, w.nw)


def _noalloc(wsa, w, layout, q, k, v, canonical=True, out=None):
    out = torch.full_like(q, float("nan")) if out is None else out
    st = wsa.lib.wsa_attention_noalloc(*_grid(w), layout, 30, ctypes.c_void_p(q.data_ptr()),
                                       ctypes.c_void_p(k.data_ptr()), ctypes.c_void_p(v.data_ptr()),
                                       ctypes.c_void_p(out.data_ptr()), q.shape[1], 1 if canonical else 0, 0.0,
                                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, wsa.lib.wsa_last_error().decode()
    return out


def test_noalloc_matches_plan_entry_point_on_consecutive_calls():
    import shifted_window_attention_gb300 as wsa

    cases = [(MID, 0), (MID, 1), (WORKLOADS["720p"], 1), (WORKLOADS["720p"], 0)]
    for w, layout in cases:
        q, k, v = wsa_inputs.qkv(w, layer=layout, device="cuda")
        plan = wsa.Plan(*_grid(w), layout)
        expect = wsa.attention(plan, q, k, v)
        # two calls in a row through the C ABI: the second finds the first
        # call's tables and scheduler words in the shared array.  The same
        # kernels on the same tables give the same bits.
        first = _noalloc(wsa, w, layout, q, k, v)
        second = _noalloc(wsa, w, layout, q, k, v)
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        assert wsa.noalloc_device_status() == 0
        assert torch.equal(first, expect), f"{w.name} layout {layout}, first call"
        assert torch.equal(second, expect), f"{w.name} layout {layout}, second call"


@pytest.mark.parametrize("layout", [0, 1])
def test_noalloc_against_the_oracle(layout):
    import shifted_window_attention_gb300 as wsa

    w = MID
    q, k, v = wsa_inputs.qkv(w, layer=7 + layout)
    got = _noalloc(wsa, w, layout, *(t.cuda() for t in (q, k, v)))
    torch.cuda.synchronize()
    ref = oracle.window_attention(to64(q), to64(k), to64(v), oracle.make_plan(*_grid(w), layout))
    assert_bf16_close(to64(got), ref, f"noalloc {w.name} layout {layout}")


def test_noalloc_allocates_nothing():
    # after a first call (which loads the kernels and looks up the array's
    # address), further calls leave the device's free memory unchanged
    import shifted_window_attention_gb300 as wsa

    w = WORKLOADS["720p"]
    q, k, v = wsa_inputs.qkv(w, layer=2, device="cuda")
    outs = [torch.empty_like(q) for _ in range(3)]
    _noalloc(wsa, w, 1, q, k, v, out=outs[0])
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    _noalloc(wsa, w, 1, q, k, v, out=outs[1])
    _noalloc(wsa, w, 0, q, k, v, out=outs[2])
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.equal(outs[0], outs[1])


def test_noalloc_packed_order():
    import shifted_window_attention_gb300 as wsa

    w = MID
    plan = wsa.Plan(*_grid(w), 1)
    ids = plan.tables()[2].long()
    q, k, v = (t[ids].contiguous() for t in wsa_inputs.qkv(w, layer=3, device="cuda"))
    expect = wsa.attention(plan, q, k, v, canonical=False)
    got = _noalloc(wsa, w, 1, q, k, v, canonical=False)
    torch.cuda.synchronize()
    assert torch.equal(got, expect)


def test_noalloc_rejects_sizes_beyond_its_limit():
    import shifted_window_attention_gb300 as wsa

    x = torch.zeros(16, 1, 128, device="cuda", dtype=torch.bfloat16)
    y = torch.zeros_like(x)
    # 21 x 180 x 160 = 604,800 tokens > 524,288
    st = wsa.lib.wsa_attention_noalloc(21, 180, 160, 4, 3, 3, 0, 30, ctypes.c_void_p(x.data_ptr()),
                                       ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(x.data_ptr()),
                                       ctypes.c_void_p(y.data_ptr()), 1, 1, 0.0, None)
    assert st == -2
    assert b"static scratch limit" in wsa.lib.wsa_last_error()


def test_noalloc_device_status_reports_a_wait_that_ran_out():
    # a launch that hands out no work unit: every role's first wait runs out
    # after about a second and records its code in the fixed array; the
    # status call reports and clears it, and the next call is correct again
    import shifted_window_attention_gb300 as wsa

    w = MID
    q, k, v = wsa_inputs.qkv(w, layer=4, device="cuda")
    out = torch.full_like(q, float("nan"))
    try:
        wsa.debug_withhold_units(1)
        _noalloc(wsa, w, 0, q, k, v, out=out)
        with pytest.raises(wsa.WsaError) as e:
            wsa.noalloc_device_status()
    finally:
        wsa.debug_withhold_units(0)
    assert e.value.name == "WSA_ERR_DEVICE_CHECK"
    code = int(str(e.value).rsplit(" ", 1)[-1])
    assert code in {0x102, 0x201, 0x301}, hex(code)
    assert bool(torch.isnan(out).all())
    assert wsa.noalloc_device_status() == 0
    plan = wsa.Plan(*_grid(w), 0)
    assert torch.equal(_noalloc(wsa, w, 0, q, k, v), wsa.attention(plan, q, k, v))
    assert wsa.noalloc_device_status() == 0
