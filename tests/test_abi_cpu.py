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


def test_small_ksplit_switch_arguments():
    mmq.mmq_debug_small_ksplit(8, 4)
    mmq.mmq_debug_small_ksplit(0, 0)
    for bad in ((9, 0), (-1, 0), (2, 5), (2, -1)):
        assert mmq.lib().mmq_debug_small_ksplit(*bad) == -9


def test_small_stream_grid_rule():
    """The small-M tensor-core streams' grids under capture (host-only query; with no device
    it assumes 152 SMs, the count of the GPU the rule was measured on)."""
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("checked against the device's own SM count in the GPU tests")
    except ImportError:
        pass
    g = mmq.mmq_debug_small_grid
    # 224 one-box CTAs of 74 super-blocks on 304 slots: 3 boxes x 4 splits on 300 CTAs
    assert g("q4_k", 8, 3584, 18944) == (3, 4)
    assert g("q8_0", 8, 3584, 18944) == (3, 4)
    assert g("q5_k", 1, 3584, 18944) == (3, 4)
    # two passes: 448 CTAs in two waves -> 3 x 2 on 300; three and four passes: 3 boxes, unsplit
    assert g("q4_k", 16, 3584, 18944) == (3, 2)
    assert g("q4_k", 24, 3584, 18944) == (3, 1)
    assert g("q4_k", 32, 3584, 18944) == (3, 1)
    # few boxes: 32 of them x 4 splits; 128 x 2
    assert g("q4_k", 8, 512, 18944) == (1, 4)
    assert g("q4_k", 8, 2048, 18944) == (1, 2)
    # 4096 x 14336 through sixteen rows: 512 CTAs in two waves -> 2 boxes, one wave
    assert g("q4_k", 16, 4096, 14336) == (2, 1)
    # kept: short K (14 super-blocks), a grid already in one even wave, several passes of a short K
    assert g("q4_k", 8, 3584, 3584) == (1, 1)
    assert g("q4_k", 8, 18944, 3584) == (2, 1)      # 592 32-row boxes, two per CTA
    assert g("q8_0", 8, 18944, 3584) == (4, 1)      # 1184 16-row boxes, four per CTA
    assert g("q4_k", 16, 18944, 3584) == (2, 1)
    assert g("q4_k", 8, 4096, 14336) == (1, 1)
    # the test switch: forced splits and boxes, then back to the rule
    mmq.mmq_debug_small_ksplit(5, 2)
    try:
        assert g("q4_k", 8, 3584, 3584) == (2, 5)
        mmq.mmq_debug_small_ksplit(1, 0)
        assert g("q4_k", 8, 3584, 18944) == (1, 1)
    finally:
        mmq.mmq_debug_small_ksplit(0, 0)
    assert g("q4_k", 8, 3584, 18944) == (3, 4)
    assert mmq.lib().mmq_debug_small_grid(3, 8, 3584, 18944, None, None) == -9  # Q6_K: not this stream


def test_expand_tiling_rule():
    """The expanded path's tile width and K splits (host-only query; with no device it
    assumes 152 SMs, the count of the GPU the rule was measured on)."""
    try:
        import torch
        if torch.cuda.is_available():
            pytest.skip("checked against the device's own SM count in the GPU tests")
    except ImportError:
        pass
    t = mmq.mmq_debug_expand_tiling
    # 4 x 28 = 112 tiles 128 wide on 152 SMs; 4 x 38 = 152 tiles 96 wide
    assert t("q8_0", 512, 3584, 3584) == (96, 1)
    assert t("q4_k", 1024, 3584, 3584) == (96, 1)      # 2 waves either way: 2 x 96 < 0.9 x 2 x 128
    assert t("q4_k", 300, 3301, 512) == (96, 1)        # 3 x 26 = 78 > 76 tiles, 105 in 96-wide ones
    assert t("q4_k", 2048, 18944, 3584) == (128, 1)    # 16 x 148 tiles: 16 waves against 21 x 96 / 128
    assert t("q6_k", 2048, 3584, 18944) == (128, 1)    # 448 tiles, 3 waves; 608 narrow ones take 4
    # at most half as many tiles as SMs: 128 wide and K split to fill the SMs
    assert t("q4_k", 128, 3584, 3584) == (128, 5)      # 28 tiles, 152 // 28 = 5 splits of 14 groups
    assert t("q8_0", 256, 3584, 18944) == (128, 2)
    assert t("q8_0", 64, 256, 512) == (128, 1)         # two groups: no split below two groups each
    assert t("q5_k", 9, 33, 4096) == (128, 8)          # one tile: at most 8 splits
    for M, N, K in [(1, 1, 256), (777, 5000, 2048), (4096, 3584, 3584), (640, 1000, 1024)]:
        bn, sp = t("q4_k", M, N, K)
        assert bn in (96, 128) and 1 <= sp <= 8
        assert sp == 1 or bn == 128
        assert sp * 2 <= K // 256 or sp == 1
    with pytest.raises(mmq.MMQError):
        t("q4_k", 8, 8, 100)
    with pytest.raises(mmq.MMQError):
        t(4, 8, 8, 256)
    assert mmq.lib().mmq_debug_expand_tiling(1, 8, 8, 256, None, None) == -3  # MMQ_ERR_NULL


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
