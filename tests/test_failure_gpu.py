"""Failure path of the tensor-core attention kernel on a GPU, without a fault.

Every wait in the kernel is bounded: a wait that runs out records its code in
the plan's error word and the kernel unwinds, so the host sees a typed status
(WSA_ERR_DEVICE_CHECK) and the context stays usable.  wsa_debug_withhold_units
makes one launch hand out no work unit, so every role's first wait runs out
(after about one second) with nothing in flight; the test then checks the
status, that no output was written, and that the next launch on the same plan
is correct again."""

import numpy as np
import pytest
import torch

import oracle
import wsa_inputs
from tests.helpers import assert_bf16_close, to64

pytestmark = pytest.mark.gpu

W = wsa_inputs.custom(4, 20, 36, 2, 2, 2, heads=2, head_dim=128, name="failure")
# codes of the first wait of each role (the unit slot): gather, MMA, softmax
UNIT_WAIT_CODES = {0x102, 0x201, 0x301}


@pytest.fixture(scope="module")
def wsa():
    import shifted_window_attention_gb300 as m
    return m


def _grid():
    return (W.T, W.H, W.W, W.nt, W.nh, W.nw)


@pytest.mark.parametrize("canonical", [True, False], ids=["canonical", "packed"])
def test_withheld_units_time_out_and_recover(wsa, canonical):
    p = wsa.Plan(*_grid(), 1)
    op = oracle.make_plan(*_grid(), 1)
    q, k, v = wsa_inputs.qkv(W)
    ids = torch.from_numpy(op.ids.astype(np.int64))
    if not canonical:
        q, k, v = (t[ids].contiguous() for t in (q, k, v))
    qg, kg, vg = (t.cuda() for t in (q, k, v))
    out = torch.full_like(qg, float("nan"))
    try:
        wsa.debug_withhold_units(1)
        wsa.attention(p, qg, kg, vg, out=out, canonical=canonical)
        with pytest.raises(wsa.WsaError) as e:
            p.device_status()
    finally:
        wsa.debug_withhold_units(0)
    assert e.value.name == "WSA_ERR_DEVICE_CHECK"
    code = int(str(e.value).rsplit(" ", 1)[-1])
    assert code in UNIT_WAIT_CODES, hex(code)
    assert bool(torch.isnan(out).all()), "a launch that handed out no unit wrote output"
    # the error word was read and cleared; the context and the plan still work
    assert p.device_status() == 0
    wsa.attention(p, qg, kg, vg, out=out, canonical=canonical)
    assert p.device_status() == 0
    ref = oracle.window_attention(to64(q if canonical else q[torch.argsort(ids)]),
                                  to64(k if canonical else k[torch.argsort(ids)]),
                                  to64(v if canonical else v[torch.argsort(ids)]), op)
    if not canonical:
        ref = ref[op.ids]
    assert_bf16_close(to64(out), ref, f"after recovery ({'canonical' if canonical else 'packed'})")
