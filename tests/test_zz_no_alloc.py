"""The allocation-free attention entry point, wsa_attention_noalloc.

It serves callers that cannot call cudaMalloc -- device memory owned by
another framework's pool, or serving loops that must not take the
device-wide synchronisation of cudaMalloc/cudaFree -- and therefore cannot
create a plan.  Its output must agree with the
plan-based wsa_attention within the bf16 tolerance the other tests use, on
consecutive calls that reuse the library's fixed scratch array.

This file is collected last so that a run stopping at the first failure has
already run every other test."""

import ctypes

import pytest
import torch

import wsa_inputs
from tests.helpers import assert_bf16_close_torch
from wsa_inputs import WORKLOADS

pytestmark = pytest.mark.gpu

MID = wsa_inputs.custom(8, 24, 40, 2, 2, 2, heads=2, head_dim=128, name="mid")


def _grid(w):
    return (w.T, w.H, w.W, w.nt, w.nh, w.nw)


def _noalloc(wsa, w, layout, q, k, v, canonical=True):
    out = torch.full_like(q, float("nan"))
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
        # call's tables and scheduler words in the shared array
        first = _noalloc(wsa, w, layout, q, k, v)
        second = _noalloc(wsa, w, layout, q, k, v)
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        assert_bf16_close_torch(first, expect, f"{w.name} layout {layout}, first call")
        assert_bf16_close_torch(second, expect, f"{w.name} layout {layout}, second call")


def test_noalloc_packed_order():
    import shifted_window_attention_gb300 as wsa

    w = MID
    plan = wsa.Plan(*_grid(w), 1)
    ids = plan.tables()[2].long()
    q, k, v = (t[ids].contiguous() for t in wsa_inputs.qkv(w, layer=3, device="cuda"))
    expect = wsa.attention(plan, q, k, v, canonical=False)
    got = _noalloc(wsa, w, 1, q, k, v, canonical=False)
    torch.cuda.synchronize()
    assert_bf16_close_torch(got, expect, "packed order")


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
