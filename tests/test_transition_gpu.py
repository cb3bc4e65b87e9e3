"""GPU layout transition against the oracle, bit for bit ("Window-Aligned
Sequence Parallelism (SeedVR2)", sections "Motivation" and "Plan A
redistribution": with one rank a layout change is a local permutation)."""

import numpy as np
import pytest
import torch

import oracle
import wsa_inputs
from wsa_inputs import WORKLOADS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def wsa():
    import shifted_window_attention_gb300 as m
    return m


def _plans(wsa, w):
    g = (w.T, w.H, w.W, w.nt, w.nh, w.nw)
    return wsa.Plan(*g, 0), wsa.Plan(*g, 1), oracle.make_plan(*g, 0), oracle.make_plan(*g, 1)


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_bit_exact_both_directions(wsa, name):
    w = WORKLOADS[name]
    reg, sft, oreg, osft = _plans(wsa, w)
    x = wsa_inputs.activation(w, device="cuda")  # rows in regular packed order
    y = wsa.transition(reg, sft, x)
    xc = x.cpu()
    g = torch.from_numpy(oracle.gather_table(oreg, osft))
    assert torch.equal(y.cpu(), xc[g])  # oracle: x_dst[p] = x_src[pos_src[ids_dst[p]]]
    back = wsa.transition(sft, reg, y)
    assert torch.equal(back, x)
    assert reg.device_status() == 0


@pytest.mark.parametrize("channels,dtype", [(3072, torch.bfloat16), (24, torch.float32), (7, torch.bfloat16),
                                            (5, torch.float32), (1, torch.bfloat16), (4096, torch.float32)])
def test_row_widths_and_dtypes(wsa, channels, dtype):
    w = WORKLOADS["tiny"]
    reg, sft, oreg, osft = _plans(wsa, w)
    x = (torch.randn(w.num_tokens, channels, generator=torch.Generator().manual_seed(channels))).to(dtype).cuda()
    y = wsa.transition(reg, sft, x)
    g = torch.from_numpy(oracle.gather_table(oreg, osft))
    assert torch.equal(y.cpu(), x.cpu()[g])


def test_labels_and_identity(wsa):
    w = WORKLOADS["720p"]
    reg, sft, oreg, osft = _plans(wsa, w)
    lab = torch.from_numpy(oreg.ids.astype(np.float32)).view(-1, 1).repeat(1, 4).cuda()
    out = wsa.transition(reg, sft, lab)
    assert np.array_equal(out[:, 0].cpu().numpy().astype(np.int64), osft.ids)
    same = wsa.transition(reg, reg, lab)
    assert torch.equal(same, lab)


def test_errors(wsa):
    w = WORKLOADS["tiny"]
    reg, sft, _, _ = _plans(wsa, w)
    other = wsa.Plan(4, 9, 17, 2, 9, 16, 1)
    x = torch.zeros(w.num_tokens, 8, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(wsa.WsaError) as e:
        wsa.transition(reg, other, x)
    assert e.value.name in ("WSA_ERR_MISMATCH", "WSA_ERR_INVALID_ARG")
    import ctypes
    st = wsa.lib.wsa_transition(reg.handle, other.handle, ctypes.c_void_p(x.data_ptr()),
                                ctypes.c_void_p(torch.empty_like(x).data_ptr()), 8, 0, None)
    assert st == -5
    # overlapping buffers
    big = torch.zeros(2 * w.num_tokens, 8, device="cuda", dtype=torch.bfloat16)
    st = wsa.lib.wsa_transition(reg.handle, sft.handle, ctypes.c_void_p(big.data_ptr()),
                                ctypes.c_void_p(big[10:].data_ptr()), 8, 0, None)
    assert st == -1
