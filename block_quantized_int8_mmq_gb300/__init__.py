"""Python binding of libmmq, the GB300 (sm_103a) block-quantized int8 matrix multiply.

Each function has the name of the C entry point it calls (include/mmq.h) and only
marshals arguments: torch tensors supply device memory and the current CUDA stream,
every computation runs in the library's CUDA kernels.  There is no CPU fallback: if
libmmq.so is not built, importing this package raises ImportError.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmmq.so")

QK, QK_K = 32, 256
Q8_1_BYTES, Q8_0_BYTES, Q4_K_BYTES, Q5_K_BYTES, Q6_K_BYTES = 36, 34, 144, 176, 210
FMT = {"q8_0": 0, "q4_k": 1, "q5_k": 2, "q6_k": 3}
PATH_AUTO, PATH_SMALL, PATH_TC, PATH_EXPAND = 0, 1, 2, 3

EXPORTED = (
    "mmq_status_string", "mmq_q8_1_bytes", "mmq_weight_row_bytes", "mmq_quantize_q8_1",
    "mmq_gemm_q8_0", "mmq_gemm_q4_k", "mmq_debug_block_dots_q8_0", "mmq_debug_block_dots_q4_k",
    "mmq_set_path", "mmq_last_path", "mmq_get_device_error", "mmq_profile_enable", "mmq_profile_read",
    "mmq_gemm_noalloc", "mmq_linear_q8_0", "mmq_linear_q4_k", "mmq_gemm_grouped_q8_0", "mmq_gemm_grouped_q4_k",
    "mmq_gemm_q5_k", "mmq_linear_q5_k", "mmq_debug_block_dots_q5_k",
    "mmq_gemm_q6_k", "mmq_linear_q6_k", "mmq_debug_block_dots_q6_k", "mmq_gemm_grouped_q5_k",
    "mmq_debug_product_dots", "mmq_debug_refuse_smem", "mmq_debug_set_wait_limit",
    "mmq_debug_small_route", "mmq_debug_expand_tiling", "mmq_gemm_grouped_q6_k", "mmq_debug_small_ksplit",
    "mmq_debug_small_grid",
)


class KernelTime(ctypes.Structure):
    """mmq_kernel_time: per-kernel launch count and total device time."""
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int64), ("total_ms", ctypes.c_double)]


class MMQError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn}: {_lib.mmq_status_string(status).decode()} ({status})")
        self.status = status


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built: run `python block_quantized_int8_mmq_gb300/_build.py`")
    L = ctypes.CDLL(LIB_PATH)
    P, I64, I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    L.mmq_status_string.argtypes = [I]
    L.mmq_status_string.restype = ctypes.c_char_p
    L.mmq_q8_1_bytes.argtypes = [I64, I64]
    L.mmq_q8_1_bytes.restype = ctypes.c_size_t
    L.mmq_weight_row_bytes.argtypes = [I, I64]
    L.mmq_weight_row_bytes.restype = ctypes.c_size_t
    L.mmq_quantize_q8_1.argtypes = [P, I64, I64, P, P]
    for f in ("mmq_gemm_q8_0", "mmq_gemm_q4_k", "mmq_gemm_q5_k", "mmq_gemm_q6_k", "mmq_debug_block_dots_q8_0",
              "mmq_debug_block_dots_q4_k", "mmq_debug_block_dots_q5_k", "mmq_debug_block_dots_q6_k"):
        getattr(L, f).argtypes = [P, P, I64, I64, I64, P, P]
    L.mmq_set_path.argtypes = [I]
    L.mmq_get_device_error.argtypes = [P]
    L.mmq_gemm_noalloc.argtypes = [I, P, P, I64, I64, I64, P, P]
    for f in ("mmq_linear_q8_0", "mmq_linear_q4_k", "mmq_linear_q5_k", "mmq_linear_q6_k"):
        getattr(L, f).argtypes = [P, I64, I64, P, I64, P, P, P]
    for f in ("mmq_gemm_grouped_q8_0", "mmq_gemm_grouped_q4_k", "mmq_gemm_grouped_q5_k", "mmq_gemm_grouped_q6_k"):
        getattr(L, f).argtypes = [P, P, I64, P, I64, I64, I64, P, P]
    L.mmq_debug_product_dots.argtypes = [I, P, P, I64, I64, I64, P, P]
    L.mmq_debug_refuse_smem.argtypes = [I]
    L.mmq_debug_small_route.argtypes = [I]
    L.mmq_debug_small_ksplit.argtypes = [I, I]
    L.mmq_debug_small_grid.argtypes = [I, I64, I64, I64, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]
    L.mmq_debug_expand_tiling.argtypes = [I, I64, I64, I64, ctypes.POINTER(ctypes.c_int32),
                                          ctypes.POINTER(ctypes.c_int32)]
    L.mmq_debug_set_wait_limit.argtypes = [I64]
    L.mmq_profile_enable.argtypes = [I]
    L.mmq_profile_read.argtypes = [ctypes.POINTER(KernelTime), I, I]
    return L


_lib = _load()


def lib():
    return _lib


def _stream(stream):
    import torch
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(fn, st):
    if st != 0:
        raise MMQError(fn, st)


def _ptr(t):
    """Device address of a contiguous CUDA tensor (the library takes raw device pointers)."""
    if not t.is_cuda:
        raise ValueError("libmmq takes CUDA tensors (device memory); got a tensor on " + str(t.device))
    if not t.is_contiguous():
        raise ValueError("libmmq takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def mmq_profile_enable(on: bool) -> bool:
    """Turn per-kernel event timing on or off; returns the previous state."""
    return bool(_lib.mmq_profile_enable(1 if on else 0))


def mmq_profile_read(reset: bool = False) -> dict:
    """{kernel name: (launches, total device ms)} of the launches timed so far."""
    n = _lib.mmq_profile_read(None, 0, 0)
    if n < 0:
        raise MMQError("mmq_profile_read", n)
    buf = (KernelTime * max(n, 1))()
    n = _lib.mmq_profile_read(buf, n, 1 if reset else 0)
    if n < 0:
        raise MMQError("mmq_profile_read", n)
    return {buf[i].name.decode(): (int(buf[i].launches), float(buf[i].total_ms)) for i in range(n)}


def mmq_status_string(status: int) -> str:
    return _lib.mmq_status_string(int(status)).decode()


def mmq_q8_1_bytes(M: int, K: int) -> int:
    return int(_lib.mmq_q8_1_bytes(M, K))


def mmq_weight_row_bytes(fmt: str, K: int) -> int:
    return int(_lib.mmq_weight_row_bytes(FMT[fmt], K))


def mmq_quantize_q8_1(x, xq=None, stream=None):
    """x: f32 [M, K] CUDA tensor -> uint8 [M, K/32*36] q8_1 blocks."""
    import torch
    M, K = x.shape
    if xq is None:
        xq = torch.empty((M, K // QK * Q8_1_BYTES), dtype=torch.uint8, device=x.device)
    _check("mmq_quantize_q8_1", _lib.mmq_quantize_q8_1(_ptr(x), M, K, _ptr(xq), _stream(stream)))
    return xq


def _gemm(fn, xq, wq, M, N, K, out, stream):
    import torch
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=xq.device)
    _check(fn, getattr(_lib, fn)(_ptr(xq), _ptr(wq), M, N, K, _ptr(out), _stream(stream)))
    return out


def mmq_gemm_q8_0(xq, wq, M, N, K, out=None, stream=None):
    """q8_1 [M, K/32*36] x Q8_0 [N, K/32*34] -> f32 [M, N]."""
    return _gemm("mmq_gemm_q8_0", xq, wq, M, N, K, out, stream)


def mmq_gemm_q4_k(xq, wq, M, N, K, out=None, stream=None):
    """q8_1 [M, K/32*36] x Q4_K [N, K/256*144] -> f32 [M, N]."""
    return _gemm("mmq_gemm_q4_k", xq, wq, M, N, K, out, stream)


def mmq_gemm_noalloc(fmt, xq, wq, M, N, K, out=None, stream=None):
    """The contraction on the expanded tensor-core path with the library's fixed 64 MiB
    device scratch: no device allocation.  fmt: "q8_0", "q4_k", "q5_k", "q6_k" or 0 .. 3."""
    import torch
    f = FMT[fmt] if isinstance(fmt, str) else int(fmt)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=xq.device)
    _check("mmq_gemm_noalloc", _lib.mmq_gemm_noalloc(f, _ptr(xq), _ptr(wq), M, N, K, _ptr(out), _stream(stream)))
    return out


def _dots(fn, xq, wq, M, N, K, dots, stream):
    import torch
    if dots is None:
        dots = torch.empty((M, N, K // QK), dtype=torch.int32, device=xq.device)
    _check(fn, getattr(_lib, fn)(_ptr(xq), _ptr(wq), M, N, K, _ptr(dots), _stream(stream)))
    return dots


def mmq_debug_block_dots_q8_0(xq, wq, M, N, K, dots=None, stream=None):
    return _dots("mmq_debug_block_dots_q8_0", xq, wq, M, N, K, dots, stream)


def mmq_debug_block_dots_q4_k(xq, wq, M, N, K, dots=None, stream=None):
    return _dots("mmq_debug_block_dots_q4_k", xq, wq, M, N, K, dots, stream)


def mmq_debug_product_dots(fmt, xq, wq, M, N, K, dots=None, stream=None):
    """The integer block dots of the expanded-path contraction as it forms them (K-quants:
    the sub-scale folded into the weight codes): int32 [M, N, K/32]."""
    import torch
    if dots is None:
        dots = torch.empty((M, N, K // QK), dtype=torch.int32, device=xq.device)
    f = FMT[fmt] if isinstance(fmt, str) else int(fmt)
    _check("mmq_debug_product_dots",
           _lib.mmq_debug_product_dots(f, _ptr(xq), _ptr(wq), M, N, K, _ptr(dots), _stream(stream)))
    return dots


def mmq_debug_refuse_smem(on: bool) -> bool:
    """Test switch: treat every shared-memory limit request as refused; returns the previous state."""
    return bool(_lib.mmq_debug_refuse_smem(1 if on else 0))


def mmq_debug_set_wait_limit(ns: int) -> None:
    """Test switch: the bound of the expanded-path contraction's waits for its operand copies, in
    ns (0: give up at the first such wait whose copy has not landed; < 0: the 2 s default)."""
    _check("mmq_debug_set_wait_limit", _lib.mmq_debug_set_wait_limit(int(ns)))


SMALL_ROUTE_AUTO, SMALL_ROUTE_DP4A, SMALL_ROUTE_MMA = 0, 1, 2


def mmq_debug_small_route(route: int) -> int:
    """Which small-M kernel takes K % 256 == 0 shapes (0 measured choice, 1 dp4a stream up to four
    rows, 2 tensor-core stream); returns the previous setting."""
    prev = _lib.mmq_debug_small_route(int(route))
    if prev < 0:
        raise MMQError("mmq_debug_small_route", prev)
    return prev


def mmq_debug_small_ksplit(splits: int, boxes: int = 0) -> None:
    """K splits of the Q8_0 / Q4_K / Q5_K tensor-core streams (0 the measured rule, n > 0 n
    splits, 1 never) and, with forced splits, boxes per CTA (0 the unsplit grid's)."""
    _check("mmq_debug_small_ksplit", _lib.mmq_debug_small_ksplit(int(splits), int(boxes)))


def mmq_debug_small_grid(fmt, M: int, N: int, K: int) -> tuple:
    """(boxes per CTA, K splits) of the Q8_0 / Q4_K / Q5_K tensor-core stream for this shape
    under stream capture (host-only query)."""
    b, z = ctypes.c_int32(0), ctypes.c_int32(0)
    f = FMT[fmt] if isinstance(fmt, str) else int(fmt)
    _check("mmq_debug_small_grid", _lib.mmq_debug_small_grid(f, int(M), int(N), int(K), ctypes.byref(b),
                                                              ctypes.byref(z)))
    return b.value, z.value


def mmq_debug_expand_tiling(fmt, M: int, N: int, K: int) -> tuple:
    """(tile_n, splits): the weight rows per output tile and the K splits per tile the
    expanded tensor-core path takes for this shape on the current device (host-only query)."""
    tn, sp = ctypes.c_int32(0), ctypes.c_int32(0)
    f = FMT[fmt] if isinstance(fmt, str) else int(fmt)
    _check("mmq_debug_expand_tiling", _lib.mmq_debug_expand_tiling(f, int(M), int(N), int(K), ctypes.byref(tn),
                                                                    ctypes.byref(sp)))
    return tn.value, sp.value


def mmq_set_path(path: int) -> int:
    prev = _lib.mmq_set_path(int(path))
    if prev < 0:
        raise MMQError("mmq_set_path", prev)
    return prev


def mmq_last_path() -> int:
    return int(_lib.mmq_last_path())


def mmq_get_device_error(stream=None) -> int:
    return int(_lib.mmq_get_device_error(_stream(stream)))


def mmq_gemm_q5_k(xq, wq, M, N, K, out=None, stream=None):
    """q8_1 [M, K/32*36] x Q5_K [N, K/256*176] -> f32 [M, N]."""
    return _gemm("mmq_gemm_q5_k", xq, wq, M, N, K, out, stream)


def mmq_debug_block_dots_q5_k(xq, wq, M, N, K, dots=None, stream=None):
    return _dots("mmq_debug_block_dots_q5_k", xq, wq, M, N, K, dots, stream)


def mmq_gemm_q6_k(xq, wq, M, N, K, out=None, stream=None):
    """q8_1 [M, K/32*36] x Q6_K [N, K/256*210] -> f32 [M, N]."""
    return _gemm("mmq_gemm_q6_k", xq, wq, M, N, K, out, stream)


def mmq_debug_block_dots_q6_k(xq, wq, M, N, K, dots=None, stream=None):
    return _dots("mmq_debug_block_dots_q6_k", xq, wq, M, N, K, dots, stream)


def gemm(fmt: str, xq, wq, M, N, K, out=None, stream=None):
    f = {"q8_0": mmq_gemm_q8_0, "q4_k": mmq_gemm_q4_k, "q5_k": mmq_gemm_q5_k, "q6_k": mmq_gemm_q6_k}[fmt]
    return f(xq, wq, M, N, K, out, stream)


def block_dots(fmt: str, xq, wq, M, N, K, dots=None, stream=None):
    f = {"q8_0": mmq_debug_block_dots_q8_0, "q4_k": mmq_debug_block_dots_q4_k,
         "q5_k": mmq_debug_block_dots_q5_k, "q6_k": mmq_debug_block_dots_q6_k}[fmt]
    return f(xq, wq, M, N, K, dots, stream)


def mmq_gemm_grouped(fmt: str, xq, row_expert, wq, E: int, N: int, K: int, out=None, stream=None):
    """Expert-grouped contraction: row r of xq (q8_1 [R, K/32*36]) with expert
    row_expert[r] (int32 [R]) of wq (E matrices stacked, [E*N, ...] blocks): f32 [R, N]."""
    import torch
    R = xq.shape[0]
    if out is None:
        out = torch.empty((R, N), dtype=torch.float32, device=xq.device)
    fn = "mmq_gemm_grouped_" + fmt
    _check(fn, getattr(_lib, fn)(_ptr(xq), _ptr(row_expert), R, _ptr(wq), E, N, K, _ptr(out), _stream(stream)))
    return out


def mmq_linear(x, wq, fmt: str, N: int, xq=None, out=None, stream=None):
    """Quantize x (f32 [M, K]) to q8_1 (into xq) and contract it with weights wq in one
    call (mmq_linear_<fmt>): f32 [M, N]."""
    import torch
    M, K = x.shape
    if xq is None:
        xq = torch.empty((M, K // QK * Q8_1_BYTES), dtype=torch.uint8, device=x.device)
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    fn = "mmq_linear_" + fmt
    _check(fn, getattr(_lib, fn)(_ptr(x), M, K, _ptr(wq), N, _ptr(xq), _ptr(out), _stream(stream)))
    return out
