"""Host-side checks of the C ABI (no GPU): the library loads, exports every
symbol include/wsa.h declares, and its host geometry matches the oracle."""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from wsa_inputs import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wsa.h")


@pytest.fixture(scope="module")
def wsa():
    import __graft_entry__
    __graft_entry__.build()
    import shifted_window_attention_gb300 as m
    return m


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(wsa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ("wsa_plan_create", "wsa_attention", "wsa_transition", "wsa_last_error"):
        assert name in syms


@pytest.mark.parametrize("which", ["product", "checked"])
def test_library_exports_every_declared_symbol(wsa, which):
    lib = ctypes.CDLL(wsa._LIB_PATH if which == "product" else wsa._CHECKED_LIB_PATH)
    missing = [s for s in declared_symbols() if not hasattr(lib, s)]
    assert missing == []


def test_bounds_checked_flag(wsa):
    # the product build runs no device range checks; the checked build does
    assert wsa.lib.wsa_bounds_checked() == 0
    assert wsa.checked_library().wsa_bounds_checked() == 1


def test_version(wsa):
    assert wsa.version() == 100


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_host_geometry_matches_oracle(wsa, name):
    w = WORKLOADS[name]
    g = (w.T, w.H, w.W, w.nt, w.nh, w.nw)
    assert wsa.window_size(*g) == oracle.window_size(*g)
    for layout in (0, 1):
        p = oracle.make_plan(*g, layout)
        assert wsa.layout_windows(*g, layout) == [tuple(b) for b in p.boxes]


def test_host_geometry_random_grids(wsa):
    rng = np.random.default_rng(21)
    checked = 0
    for _ in range(300):
        T, H, W = (int(x) for x in rng.integers(1, 200, size=3))
        nt, nh, nw = (int(x) for x in rng.integers(1, 20, size=3))
        mt = int(rng.integers(1, 40))
        try:
            expect = oracle.window_size(T, H, W, nt, nh, nw, mt)
        except ValueError:
            with pytest.raises(wsa.WsaError):
                wsa.window_size(T, H, W, nt, nh, nw, mt)
            continue
        assert wsa.window_size(T, H, W, nt, nh, nw, mt) == expect
        for layout in (0, 1):
            assert wsa.layout_windows(T, H, W, nt, nh, nw, layout, mt) == [
                tuple(b) for b in oracle.windows(T, H, W, *expect, layout == 1)]
        checked += 1
    assert checked > 100


def test_round_half_even_on_host(wsa):
    # H*scale = 22.5 exactly: half-to-even gives 22 (C's round() would give 23)
    assert wsa.window_size(1, 45, 320, 1, 1, 1) == (1, 22, 160)
    assert wsa.window_size(1, 225, 64, 1, 1, 1) == (1, 112, 32)


@pytest.mark.parametrize("bad", [
    (0, 9, 16, 2, 9, 16, 30), (4, 9, 16, 0, 9, 16, 30), (4, 9, 16, 2, 9, 16, 0),
    (1, 1, 100000, 1, 1, 1, 30),
])
def test_invalid_geometry_is_an_error(wsa, bad):
    with pytest.raises(wsa.WsaError) as e:
        wsa.window_size(*bad)
    assert e.value.name == "WSA_ERR_INVALID_ARG"


def test_layout_capacity_and_null_checks(wsa):
    lib = wsa.lib
    n = ctypes.c_int()
    assert lib.wsa_layout_windows(4, 9, 16, 2, 9, 16, 1, 30, None, 0, ctypes.byref(n)) == 0
    assert n.value == 36
    small = (ctypes.c_int * 6)()
    assert lib.wsa_layout_windows(4, 9, 16, 2, 9, 16, 1, 30, small, 1, ctypes.byref(n)) == -1
    assert b"capacity" in lib.wsa_last_error()
    assert lib.wsa_layout_windows(4, 9, 16, 2, 9, 16, 7, 30, None, 0, ctypes.byref(n)) == -1
    assert lib.wsa_window_size(4, 9, 16, 2, 9, 16, 30, None, None, None) == -1
    assert lib.wsa_plan_destroy(None) == -1
    assert lib.wsa_plan_info(None, *([None] * 7)) == -1
    assert lib.wsa_attention(None, None, None, None, None, 1, 128, 0, 1, 0.0, None) == -1
    assert lib.wsa_transition(None, None, None, None, 8, 0, None) == -1


def test_ensure_layout_and_noalloc_status_null_checks(wsa):
    lib = wsa.lib
    moved = ctypes.c_int(7)
    assert lib.wsa_ensure_layout(None, None, None, None, 8, 0, None, ctypes.byref(moved)) == -1
    assert lib.wsa_ensure_layout(None, None, None, None, 8, 0, None, None) == -1
    assert lib.wsa_noalloc_device_status(None) == -1
