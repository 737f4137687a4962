"""Host-side checks of the C ABI that need no GPU: the library loads, exports every
function include/mmq.h declares, and refuses invalid arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

mmq = pytest.importorskip("block_quantized_int8_mmq_gb300")


def declared_functions():
    src = open(os.path.join(ROOT, "include", "mmq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mmq_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_function():
    names = declared_functions()
    assert len(names) >= 11
    lib = ctypes.CDLL(mmq.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(mmq.EXPORTED) == names


def test_sizes():
    assert mmq.mmq_q8_1_bytes(512, 3584) == 512 * 112 * 36
    assert mmq.mmq_q8_1_bytes(1, 33) == 0
    assert mmq.mmq_weight_row_bytes("q8_0", 3584) == 112 * 34
    assert mmq.mmq_weight_row_bytes("q4_k", 3584) == 14 * 144
    assert mmq.mmq_weight_row_bytes("q4_k", 3584 + 32) == 0


def test_status_strings():
    assert mmq.mmq_status_string(0) == "MMQ_OK"
    for s in range(-10, 0):
        assert mmq.mmq_status_string(s).startswith("MMQ_ERR_")
    assert mmq.mmq_status_string(-1000) == "MMQ_ERR_UNKNOWN"


def test_path_selection_round_trip():
    prev = mmq.mmq_set_path(mmq.PATH_SMALL)
    assert mmq.mmq_set_path(mmq.PATH_TC) == mmq.PATH_SMALL
    assert mmq.mmq_set_path(mmq.PATH_EXPAND) == mmq.PATH_TC
    assert mmq.mmq_set_path(prev) == mmq.PATH_EXPAND
    assert mmq.lib().mmq_set_path(7) == -9


def test_small_route_round_trip():
    prev = mmq.mmq_debug_small_route(mmq.SMALL_ROUTE_DP4A)
    assert mmq.mmq_debug_small_route(mmq.SMALL_ROUTE_MMA) == mmq.SMALL_ROUTE_DP4A
    assert mmq.mmq_debug_small_route(prev) == mmq.SMALL_ROUTE_MMA
    assert mmq.lib().mmq_debug_small_route(3) == -9
    assert mmq.lib().mmq_debug_small_route(-1) == -9
    assert mmq.mmq_debug_small_route(prev) == prev


L = mmq.lib()
V = ctypes.c_void_p


@pytest.mark.parametrize("fn", ["mmq_gemm_q8_0", "mmq_gemm_q4_k", "mmq_debug_block_dots_q8_0",
                                "mmq_debug_block_dots_q4_k"])
def test_contraction_refusals_launch_nothing(fn, capfd):
    f = getattr(L, fn)
    good = V(0x10000)
    kmul = 256 if fn.endswith("q4_k") else 32
    assert f(good, good, 0, 8, kmul, good, None) == -1            # M < 1
    assert f(good, good, 8, 0, kmul, good, None) == -1            # N < 1
    assert f(good, good, 8, 8, kmul + 16, good, None) == -2       # K multiple
    if kmul == 256:
        assert f(good, good, 8, 8, 288, good, None) == -2         # K % 32 == 0 but not % 256
    assert f(None, good, 8, 8, kmul, good, None) == -3            # NULL
    assert f(good, good, 8, 8, kmul, None, None) == -3
    assert f(V(0x10008), good, 8, 8, kmul, good, None) == -4      # misaligned xq
    assert f(good, V(0x10004), 8, 8, kmul, good, None) == -4      # misaligned wq
    assert f(good, good, 8, 8, kmul, V(0x10001), None) == -4      # misaligned output
    assert f(good, good, 1 << 30, 1 << 30, kmul, good, None) == -1  # too large
    err = capfd.readouterr().err
    assert err.count("refused") == 9 + (kmul == 256)


def test_quantize_refusals(capfd):
    f = L.mmq_quantize_q8_1
    good = V(0x10000)
    assert f(good, 0, 32, good, None) == -1
    assert f(good, 4, 48, good, None) == -2
    assert f(None, 4, 32, good, None) == -3
    assert f(V(0x10004), 4, 32, good, None) == -4   # x must be 16-byte aligned
    assert f(good, 4, 32, V(0x10002), None) == -4   # xq must be 4-byte aligned
    assert capfd.readouterr().err.count("refused") == 5
