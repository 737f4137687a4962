"""The no-allocation entry point (fixed device scratch) against the allocating one.

Collected last (file name), and independent of the order: it passes alone and after
the other GPU tests.  Two consecutive calls of different shapes and formats reuse the
same fixed scratch; each result must equal, bit for bit, the allocating entry point on
the same expanded-code path, and both must be within the parity tolerance of the oracle.
"""
import ctypes
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 1e-4


@pytest.fixture(scope="module")
def mmq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_quantized_int8_mmq_gb300 as m
    yield m
    m.mmq_set_path(m.PATH_AUTO)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


CASES = [("q4_k", 300, 520, 1024, 71), ("q8_0", 512, 3584, 3584, 72), ("q5_k", 130, 300, 512, 73),
         ("q6_k", 200, 260, 768, 74)]


def test_two_consecutive_calls_match_the_allocating_path(mmq):
    results = []
    for fmt, M, N, K, seed in CASES:
        x = synth.activations(seed, M, K, True)
        w = synth.weights(fmt, seed + 100, N, K)
        xq = mmq.mmq_quantize_q8_1(dev(x))
        wd = dev(w)
        out = torch.full((M, N), float("nan"), device="cuda")
        mmq.mmq_gemm_noalloc(fmt, xq, wd, M, N, K, out=out)
        results.append((fmt, M, N, K, x, w, xq, wd, out))
    torch.cuda.synchronize()
    assert mmq.mmq_get_device_error() == 0
    mmq.mmq_set_path(mmq.PATH_EXPAND)
    try:
        for fmt, M, N, K, x, w, xq, wd, out in results:
            ref_gpu = mmq.gemm(fmt, xq, wd, M, N, K)
            o = out.cpu().numpy()
            assert not np.isnan(o).any()
            assert np.array_equal(o, ref_gpu.cpu().numpy()), f"{fmt} {M}x{N}x{K}: differs from mmq_gemm"
            rows = np.arange(0, M, 37)
            ref, norm = oracle.gemm(fmt, oracle.quantize_q8_1(x[rows]), w, len(rows), N, K)
            assert np.all(np.abs(o[rows] - ref) <= TOL * norm)
    finally:
        mmq.mmq_set_path(mmq.PATH_AUTO)


def test_refuses_shapes_beyond_the_fixed_scratch(mmq):
    M, N, K = 2048, 18944, 3584          # ~155 MiB of scratch
    xq = torch.zeros((M, K // 32 * 36), dtype=torch.uint8, device="cuda")
    wq = torch.zeros((N, K // 32 * 34), dtype=torch.uint8, device="cuda")
    out = torch.full((M, N), float("nan"), device="cuda")
    lib = mmq.lib()
    st = lib.mmq_gemm_noalloc(0, ctypes.c_void_p(xq.data_ptr()), ctypes.c_void_p(wq.data_ptr()), M, N, K,
                              ctypes.c_void_p(out.data_ptr()), None)
    assert st == -1
    st = lib.mmq_gemm_noalloc(0, ctypes.c_void_p(xq.data_ptr()), ctypes.c_void_p(wq.data_ptr()), 64, 64, 3584 + 32,
                              ctypes.c_void_p(out.data_ptr()), None)
    assert st == -2
    st = lib.mmq_gemm_noalloc(4, ctypes.c_void_p(xq.data_ptr()), ctypes.c_void_p(wq.data_ptr()), 64, 64, 256,
                              ctypes.c_void_p(out.data_ptr()), None)
    assert st == -9
    torch.cuda.synchronize()
    assert torch.isnan(out).all()


# Run in a fresh process so that nothing earlier has grown a memory pool: with the CUDA
# modules loaded eagerly (the fixed scratch array is part of the library's module image),
# every tensor created first, free device memory is read before the first no-allocation
# call and after two rounds of calls over every case, the split-K shape (q4_k 300 x 520 x
# 1024, K split in two) included.  A call that allocated device memory, from the library's
# pool or any other, would leave less free memory behind.
CHILD = r"""
import json, sys
import numpy as np
import torch
sys.path.insert(0, ROOT)
import block_quantized_int8_mmq_gb300 as mmq
import synth
cases = CASES
ops = []
for fmt, M, N, K, seed in cases:
    x = torch.from_numpy(synth.activations(seed, M, K, True)).cuda()
    w = torch.from_numpy(synth.weights(fmt, seed + 100, N, K)).cuda()
    ops.append((fmt, M, N, K, mmq.mmq_quantize_q8_1(x), w, torch.empty((M, N), device="cuda")))
torch.cuda.synchronize()
free0 = torch.cuda.mem_get_info()[0]
for _ in range(2):
    for fmt, M, N, K, xq, w, out in ops:
        mmq.mmq_gemm_noalloc(fmt, xq, w, M, N, K, out=out)
torch.cuda.synchronize()
free1 = torch.cuda.mem_get_info()[0]
print(json.dumps({"free0": free0, "free1": free1, "err": mmq.mmq_get_device_error(),
                  "finite": bool(all(torch.isfinite(o[6]).all().item() for o in ops))}))
"""


def test_calls_allocate_no_device_memory():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = CHILD.replace("ROOT", repr(root)).replace("CASES", repr(CASES))
    env = dict(os.environ, CUDA_MODULE_LOADING="EAGER")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["err"] == 0 and res["finite"]
    assert res["free1"] >= res["free0"], f"free device memory fell by {res['free0'] - res['free1']} bytes"
