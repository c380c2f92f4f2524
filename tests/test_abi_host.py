"""C ABI checks that need no GPU: the library loads, exports every entry point
include/nys.h declares, lays the state out as documented and rejects bad
arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

nys = pytest.importorskip("streaming_nystr_landmark_gb300.nys")


def _declared():
    text = open(os.path.join(ROOT, "include", "nys.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"\b(nys_[a-z0-9_]+)\s*\(", text))


def test_every_declared_symbol_is_exported():
    declared = _declared()
    assert declared == set(nys.EXPORTED)
    lib = ctypes.CDLL(nys._LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name


def _align(x):
    return (x + 255) // 256 * 256


@pytest.mark.parametrize("geo", [(32, 128, 4, 2, 128, 128, 14336, 0),
                                 (8, 16, 4, 1, 64, 64, 1, 0),
                                 (64, 128, 4, 8, 128, 128, 512, 0),
                                 (5, 3, 0, 3, 12, 20, 7, 0),
                                 (8, 16, 4, 2, 32, 32, 9, 100)])
def test_memory_bytes_matches_documented_layout(geo):
    m, w, sink, H, d, dv, G, cap = geo
    cfg = nys.make_config(m, w, sink, H, d, dv, exact_cap=cap)
    sizes = [G * w * d, G * w * dv, G * sink * d, G * sink * dv, G * m * d,
             G * H * m * d, G * H * m * m, G * H * m * dv, G * H * m, G * H * m,
             G * H * m * dv / 2, G * H * m, G * H, G * 8,   # t_lo is bf16
             G * cap * d, G * cap * dv]
    want = sum(_align(int(4 * s)) for s in sizes)
    assert nys.nys_memory_bytes(cfg, G) == want


def test_memory_line_shares_window_across_heads():
    """The shared/private split: window, sinks and K~ are stored once per
    group, so doubling the heads of a group adds only per-head bytes."""
    one = nys.nys_memory_bytes(nys.make_config(32, 128, 4, 1, 128, 128), 1)
    two = nys.nys_memory_bytes(nys.make_config(32, 128, 4, 2, 128, 128), 1)
    per_head = 4 * (32 * 128 + 32 * 32 + 32 * 128 + 2 * 32 + 1) + 2 * 32 * 128 + 4 * 32
    assert abs((two - one) - per_head) <= 256 * 8
    assert two < 2 * one


@pytest.mark.parametrize("bad,code", [
    ((3, 128, 4, 2, 128, 128), nys.NYS_E_INVAL),     # m < 4
    ((32, 0, 4, 2, 128, 128), nys.NYS_E_INVAL),      # w < 1
    ((32, 128, -1, 2, 128, 128), nys.NYS_E_INVAL),   # sink < 0
    ((32, 128, 4, 0, 128, 128), nys.NYS_E_INVAL),    # no heads
    ((32, 128, 4, 2, 126, 128), nys.NYS_E_INVAL),    # d not a multiple of 4
    ((32, 128, 4, 2, 128, 0), nys.NYS_E_INVAL),      # dv = 0
    ((65, 128, 4, 2, 128, 128), nys.NYS_E_UNSUPPORTED),
    ((32, 128, 4, 2, 260, 128), nys.NYS_E_UNSUPPORTED),
    ((32, 128, 4, 65, 128, 128), nys.NYS_E_UNSUPPORTED),
    ((32, 2045, 4, 2, 128, 128), nys.NYS_E_UNSUPPORTED),
    ((32, 128, 4, 2, 128, 128, 0, -1), nys.NYS_E_INVAL),      # negative exact_cap
    ((32, 128, 4, 2, 128, 128, 0, 4097), nys.NYS_E_UNSUPPORTED),
])
def test_bad_geometry_rejected(bad, code):
    with pytest.raises(nys.NysError) as ei:
        nys.nys_memory_bytes(nys.make_config(*bad), 4)
    assert ei.value.code == code


def test_bad_rect_and_null_handle():
    with pytest.raises(nys.NysError) as ei:
        nys.nys_memory_bytes(nys.make_config(32, 128, 4, 2, 128, 128, rect=7), 1)
    assert ei.value.code == nys.NYS_E_INVAL
    lib = nys._lib
    assert lib.nys_seal(None, 0, 1, 256, None, None, None, None) == nys.NYS_E_INVAL
    assert lib.nys_step_batch(None, 0, 1, None, None, None, None, None) == nys.NYS_E_INVAL
    assert lib.nys_mark_sealed(None, 0, 1) == nys.NYS_E_INVAL
    assert lib.nys_debug_stall_once(None, 0) == nys.NYS_E_INVAL
    assert lib.nys_debug_stall_replay_once(None) == nys.NYS_E_INVAL
    assert lib.nys_free_states(None) == nys.NYS_OK
    assert lib.nys_memory_bytes(None, 1, None) == nys.NYS_E_INVAL


def test_strerror_total():
    for code in range(-12, 2):
        assert nys.nys_strerror(code)
