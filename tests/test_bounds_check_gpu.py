"""The bounds-checked build (libwsa_checked.so) and the allocation-failure hook.

The library ships a second build of the same sources, a stand-in for a
memory checker, in which every row index read from a plan table is
range-checked on the device before it addresses memory.  These tests call it
through the C ABI and check that:

* on valid tables its results are bit-identical to the product build's, with
  a clean device status;
* with out-of-range entries planted in a plan's ids and pos tables, the
  attention kernels and the transition skip exactly the accesses those
  entries would make, leave every other output row as the product build
  writes it, and report WSA_ERR_DEVICE_CHECK (code 0x401) through
  wsa_plan_device_status; the same plan is clean again once its tables are
  restored.

Only the checked build is ever given a corrupted table.  The last test forces
a plan allocation failure through wsa_debug_fail_allocations and checks the
WSA_ERR_OOM path of the product build.
"""

import ctypes

import pytest
import torch

import wsa_inputs

pytestmark = pytest.mark.gpu

E_BOUNDS = 0x401
DEVICE_CHECK = -6


@pytest.fixture(scope="module")
def wsa():
    import __graft_entry__
    __graft_entry__.build()
    import shifted_window_attention_gb300 as m
    torch.cuda.set_device(0)
    return m


class CheckedPlan:
    """A plan of the checked build, driven through its C ABI."""

    def __init__(self, wsa, grid, layout):
        self.lib = wsa.checked_library()
        self.wsa = wsa
        h = ctypes.c_void_p()
        st = self.lib.wsa_plan_create(*grid, layout, 30, None, ctypes.byref(h))
        assert st == 0, self.lib.wsa_last_error()
        self.h = h
        vals = [ctypes.c_int() for _ in range(7)]
        assert self.lib.wsa_plan_info(h, *[ctypes.byref(v) for v in vals]) == 0
        self.num_windows, self.num_tokens = vals[0].value, vals[1].value

    def tables(self):
        ptrs = [ctypes.c_void_p() for _ in range(4)]
        assert self.lib.wsa_plan_tables(self.h, *[ctypes.byref(x) for x in ptrs]) == 0
        sizes = [self.num_windows + 1, 6 * self.num_windows, self.num_tokens, self.num_tokens]
        return tuple(torch.as_tensor(self.wsa._DeviceArray(x.value, n, self), device="cuda")
                     for x, n in zip(ptrs, sizes))

    def status(self):
        code = ctypes.c_int()
        st = self.lib.wsa_plan_device_status(self.h, ctypes.byref(code))
        return st, code.value

    def attention(self, q, k, v, o, canonical=True):
        dt = 0 if q.dtype == torch.bfloat16 else 1
        st = self.lib.wsa_attention(self.h, q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), q.shape[1],
                                    q.shape[2], dt, 1 if canonical else 0, 0.0, None)
        assert st == 0, self.lib.wsa_last_error()

    def transition_to(self, dst, x, y):
        dt = 0 if x.dtype == torch.bfloat16 else 1
        st = self.lib.wsa_transition(self.h, dst.h, x.data_ptr(), y.data_ptr(), x.shape[1], dt, None)
        assert st == 0, self.lib.wsa_last_error()

    def __del__(self):
        try:
            self.lib.wsa_plan_destroy(self.h)
        except Exception:
            pass


def _grid(w):
    return (w.T, w.H, w.W, w.nt, w.nh, w.nw)


MID = wsa_inputs.custom(6, 40, 64, 2, 2, 2, heads=3, head_dim=128, name="bounds-mid")


def test_checked_build_matches_product_on_valid_tables(wsa):
    w = MID
    q, k, v = wsa_inputs.qkv(w, layer=2, device="cuda")
    x = wsa_inputs.activation(w, device="cuda")
    plans = [wsa.Plan(*_grid(w), lay) for lay in (0, 1)]
    cplans = [CheckedPlan(wsa, _grid(w), lay) for lay in (0, 1)]
    for lay in (0, 1):
        for t_prod, t_chk in zip(plans[lay].tables(), cplans[lay].tables()):
            assert torch.equal(t_prod, t_chk)
        expect = wsa.attention(plans[lay], q, k, v)
        got = torch.empty_like(q)
        cplans[lay].attention(q, k, v, got)
        torch.cuda.synchronize()
        assert torch.equal(got, expect)
        # packed rows (full tiles by TMA)
        ids = plans[lay].tables()[2].long()
        qp, kp, vp = (t[ids].contiguous() for t in (q, k, v))
        expect_p = wsa.attention(plans[lay], qp, kp, vp, canonical=False)
        got_p = torch.empty_like(qp)
        cplans[lay].attention(qp, kp, vp, got_p, canonical=False)
        torch.cuda.synchronize()
        assert torch.equal(got_p, expect_p)
        assert cplans[lay].status() == (0, 0)
    y_expect = wsa.transition(plans[0], plans[1], x)
    y = torch.empty_like(x)
    cplans[0].transition_to(cplans[1], x, y)
    torch.cuda.synchronize()
    assert torch.equal(y, y_expect)
    assert cplans[1].status() == (0, 0)


def _windows_of(offsets, positions):
    import bisect
    return {bisect.bisect_right(offsets, p) - 1 for p in positions}


def test_out_of_range_ids_are_skipped_and_reported(wsa):
    w = MID
    g = _grid(w)
    q, k, v = wsa_inputs.qkv(w, layer=4, device="cuda")
    plan = wsa.Plan(*g, 1)
    expect = wsa.attention(plan, q, k, v)
    cp = CheckedPlan(wsa, g, 1)
    offsets, _, ids, _ = cp.tables()
    saved = ids.clone()
    n = cp.num_tokens
    bad_pos = [3, n // 2, n - 1]
    for p, val in zip(bad_pos, [n + 7, -3, 2 ** 30]):
        ids[p] = val
    torch.cuda.synchronize()
    o = torch.full_like(q, float("nan"))
    cp.attention(q, k, v, o)
    st, code = cp.status()
    assert st == DEVICE_CHECK and code == E_BOUNDS
    assert b"out of range" in cp.lib.wsa_last_error()
    # every window without a planted entry is exactly the product result
    off = offsets.cpu().tolist()
    hit = _windows_of(off, bad_pos)
    rows = saved.long().cpu()
    for win in range(cp.num_windows):
        if win in hit:
            continue
        r = rows[off[win]:off[win + 1]].cuda()
        assert torch.equal(o[r], expect[r]), f"window {win}"
    # restored tables: clean status and the product result everywhere
    ids.copy_(saved)
    torch.cuda.synchronize()
    cp.attention(q, k, v, o)
    assert cp.status() == (0, 0)
    assert torch.equal(o, expect)


def test_out_of_range_ids_fp32_kernel(wsa):
    w = wsa_inputs.WORKLOADS["tiny"]
    g = _grid(w)
    q, k, v = wsa_inputs.qkv(w, device="cuda")
    plan = wsa.Plan(*g, 0)
    expect = wsa.attention(plan, q, k, v)
    cp = CheckedPlan(wsa, g, 0)
    offsets, _, ids, _ = cp.tables()
    saved = ids.clone()
    bad_pos = [5, 200]
    ids[5] = cp.num_tokens
    ids[200] = -1
    torch.cuda.synchronize()
    o = torch.zeros_like(q)
    cp.attention(q, k, v, o)
    st, code = cp.status()
    assert st == DEVICE_CHECK and code == E_BOUNDS
    off = offsets.cpu().tolist()
    hit = _windows_of(off, bad_pos)
    rows = saved.long().cpu()
    for win in range(cp.num_windows):
        if win not in hit:
            r = rows[off[win]:off[win + 1]].cuda()
            assert torch.equal(o[r], expect[r]), f"window {win}"
    ids.copy_(saved)
    torch.cuda.synchronize()
    cp.attention(q, k, v, o)
    assert cp.status() == (0, 0)
    assert torch.equal(o, expect)


def test_out_of_range_transition_tables(wsa):
    w = MID
    g = _grid(w)
    x = wsa_inputs.activation(w, device="cuda")
    y_expect = wsa.transition(wsa.Plan(*g, 0), wsa.Plan(*g, 1), x)
    src, dst = CheckedPlan(wsa, g, 0), CheckedPlan(wsa, g, 1)
    _, _, ids_dst, _ = dst.tables()
    _, _, _, pos_src = src.tables()
    ids_saved, pos_saved = ids_dst.clone(), pos_src.clone()
    n = src.num_tokens
    ids_dst[10] = n + 100          # first level out of range
    tok = int(ids_saved[20])
    pos_src[tok] = -5               # second level out of range for destination row 20
    torch.cuda.synchronize()
    sentinel = torch.full_like(x, 7.0)
    y = sentinel.clone()
    src.transition_to(dst, x, y)
    st, code = dst.status()
    assert st == DEVICE_CHECK and code == E_BOUNDS
    keep = torch.ones(n, dtype=torch.bool, device="cuda")
    keep[10] = False
    keep[20] = False
    assert torch.equal(y[keep], y_expect[keep])
    assert torch.equal(y[~keep], sentinel[~keep])  # skipped rows are left unwritten
    ids_dst.copy_(ids_saved)
    pos_src.copy_(pos_saved)
    torch.cuda.synchronize()
    src.transition_to(dst, x, y)
    assert dst.status() == (0, 0)
    assert torch.equal(y, y_expect)


def test_forced_allocation_failure(wsa):
    w = MID
    assert wsa.lib.wsa_debug_fail_allocations(1) == 0
    with pytest.raises(wsa.WsaError) as ei:
        wsa.Plan(*_grid(w), 0)
    assert ei.value.name == "WSA_ERR_OOM"
    assert "wsa_debug_fail_allocations" in str(ei.value)
    p = wsa.Plan(*_grid(w), 0)  # the hook fired once; the next plan is created
    assert p.num_tokens == w.T * w.H * w.W
    assert wsa.lib.wsa_debug_fail_allocations(0) == 0
