"""CPU oracle for block-quantized int8 MMQ (ctypes wrapper around mmq_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this package.  The product library never loads it and
it never loads the product library: the two share no code.

All results are plain numpy arrays: quantized blocks as uint8, block dots as int32,
contraction results and their error norms as float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mmq_oracle.c")
_LIB = os.path.join(_HERE, "libmmq_oracle.so")

QK, QK_K = 32, 256
Q8_1_BYTES, Q8_0_BYTES, Q4_K_BYTES, Q5_K_BYTES, Q6_K_BYTES = 36, 34, 144, 176, 210


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no FMA contraction, OpenMP over rows)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared",
             _SRC, "-o", tmp, "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P, I64 = ctypes.c_void_p, ctypes.c_int64
        L.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        L.oracle_f16_to_f64.restype = ctypes.c_double
        L.oracle_f64_to_f16.argtypes = [ctypes.c_double]
        L.oracle_f64_to_f16.restype = ctypes.c_uint16
        L.oracle_quantize_q8_1.argtypes = [P, I64, I64, P]
        L.oracle_q4_k_scale_min.argtypes = [P, ctypes.c_int, P, P]
        for f in ("oracle_block_dots_q8_0", "oracle_block_dots_q4_k", "oracle_block_dots_q5_k",
                  "oracle_block_dots_q6_k"):
            getattr(L, f).argtypes = [P, P, I64, I64, I64, P]
        for f in ("oracle_gemm_q8_0", "oracle_gemm_q4_k", "oracle_gemm_q5_k", "oracle_gemm_q6_k"):
            getattr(L, f).argtypes = [P, P, I64, I64, I64, P, P]
        for f in ("oracle_gemm_q8_0_at", "oracle_gemm_q4_k_at", "oracle_gemm_q5_k_at",
                  "oracle_gemm_q6_k_at"):
            getattr(L, f).argtypes = [P, P, I64, I64, I64, P, P, I64, P, P]
        L.oracle_num_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def f16_to_f64(h: int) -> float:
    return lib().oracle_f16_to_f64(int(h))


def f64_to_f16(v: float) -> int:
    return int(lib().oracle_f64_to_f16(float(v)))


def quantize_q8_1(x: np.ndarray) -> np.ndarray:
    """x f32 [M, K] -> uint8 [M, K/32*36] q8_1 blocks."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    M, K = x.shape
    assert K % QK == 0
    out = np.empty((M, K // QK * Q8_1_BYTES), dtype=np.uint8)
    lib().oracle_quantize_q8_1(_ptr(x), M, K, _ptr(out))
    return out


def q4_k_scale_min(p12: np.ndarray, j: int) -> tuple[int, int]:
    p12 = np.ascontiguousarray(p12, dtype=np.uint8)
    assert p12.size == 12
    sc, m = ctypes.c_int(), ctypes.c_int()
    lib().oracle_q4_k_scale_min(_ptr(p12), int(j), ctypes.byref(sc), ctypes.byref(m))
    return sc.value, m.value


def _check(fmt, xq, wq, M, N, K):
    assert fmt in ("q8_0", "q4_k", "q5_k", "q6_k")
    assert xq.dtype == np.uint8 and wq.dtype == np.uint8
    assert xq.size == M * (K // QK) * Q8_1_BYTES
    rb = {"q8_0": K // QK * Q8_0_BYTES, "q4_k": K // QK_K * Q4_K_BYTES, "q5_k": K // QK_K * Q5_K_BYTES,
          "q6_k": K // QK_K * Q6_K_BYTES}[fmt]
    assert wq.size == N * rb


def block_dots(fmt: str, xq: np.ndarray, wq: np.ndarray, M: int, N: int, K: int) -> np.ndarray:
    """int32 [M, N, K/32]: per-32-block integer dot products (Q6_K: with the 16-element
    sub-scales and the centring inside)."""
    xq, wq = np.ascontiguousarray(xq), np.ascontiguousarray(wq)
    _check(fmt, xq, wq, M, N, K)
    out = np.empty((M, N, K // QK), dtype=np.int32)
    getattr(lib(), f"oracle_block_dots_{fmt}")(_ptr(xq), _ptr(wq), M, N, K, _ptr(out))
    return out


def gemm(fmt: str, xq: np.ndarray, wq: np.ndarray, M: int, N: int, K: int):
    """(out, norm) float64 [M, N]: the contraction and sum of |terms| per entry."""
    xq, wq = np.ascontiguousarray(xq), np.ascontiguousarray(wq)
    _check(fmt, xq, wq, M, N, K)
    out = np.empty((M, N), dtype=np.float64)
    norm = np.empty((M, N), dtype=np.float64)
    getattr(lib(), f"oracle_gemm_{fmt}")(_ptr(xq), _ptr(wq), M, N, K, _ptr(out), _ptr(norm))
    return out, norm


def gemm_at(fmt: str, xq: np.ndarray, wq: np.ndarray, M: int, N: int, K: int, im, inn):
    """(out, norm) float64 [cnt] at the sampled entries (im[i], inn[i])."""
    xq, wq = np.ascontiguousarray(xq), np.ascontiguousarray(wq)
    _check(fmt, xq, wq, M, N, K)
    im = np.ascontiguousarray(im, dtype=np.int64)
    inn = np.ascontiguousarray(inn, dtype=np.int64)
    assert im.shape == inn.shape and im.ndim == 1
    assert (im >= 0).all() and (im < M).all() and (inn >= 0).all() and (inn < N).all()
    out = np.empty(im.size, dtype=np.float64)
    norm = np.empty(im.size, dtype=np.float64)
    getattr(lib(), f"oracle_gemm_{fmt}_at")(_ptr(xq), _ptr(wq), M, N, K, _ptr(im), _ptr(inn), im.size,
                                           _ptr(out), _ptr(norm))
    return out, norm


def num_threads() -> int:
    return int(lib().oracle_num_threads())
