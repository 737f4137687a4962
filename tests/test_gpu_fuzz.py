"""Seeded random parity: shapes, formats and forced paths drawn at random (a fixed seed, so
every run draws the same cases), each call compared with the oracle on the same operands.

The hand-picked shapes of test_gpu_parity.py cover the known edges (tile tails, K splits,
narrow tiles, few-row passes); these cases add combinations nobody picked: any M from one
row to several tiles, any N, K from one group to sixteen, every format on every path that
takes it, the fused quantize + contraction, and expert-grouped calls with random routing.
Acceptance as everywhere: |gpu - oracle| <= 1e-4 * norm per entry, q8_1 bytes bit-exact.
"""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 1e-4
FMTS = ["q8_0", "q4_k", "q5_k", "q6_k"]
MAX_WORK = 1.5e9  # M * N * K of one case (oracle time)


@pytest.fixture(scope="module")
def mmq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_quantized_int8_mmq_gb300 as m
    yield m
    m.mmq_set_path(m.PATH_AUTO)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def check_close(out, ref, norm, what):
    err = np.abs(np.asarray(out, dtype=np.float64) - ref)
    bad = err > TOL * norm
    assert not bad.any(), f"{what}: {int(bad.sum())} entries over tolerance, worst {float(np.max(err - TOL * norm))}"


def log_uniform(rng, lo, hi):
    return int(round(float(np.exp(rng.uniform(np.log(lo), np.log(hi))))))


def draw_dense(i):
    """Case i: (fmt, path, M, N, K, linear, seed)."""
    rng = np.random.default_rng(9000 + i)
    fmt = FMTS[rng.integers(len(FMTS))]
    paths = ["auto", "small", "expand"] + ([] if fmt == "q6_k" else ["tc"])
    path = paths[rng.integers(len(paths))]
    band = rng.integers(3)
    M = [log_uniform(rng, 1, 8), log_uniform(rng, 9, 96), log_uniform(rng, 97, 700)][band]
    N = log_uniform(rng, 1, 6000)
    kmul = 32 if (fmt == "q8_0" and path in ("auto", "small")) else 256
    K = kmul * log_uniform(rng, 1, 4096 // kmul)
    while M * N * K > MAX_WORK:
        N = max(1, N // 2)
    linear = bool(rng.integers(4) == 0) and K % 256 == 0 and path in ("auto", "expand")
    return fmt, path, M, N, K, linear, 9100 + i


DENSE = [draw_dense(i) for i in range(128)]


@pytest.mark.parametrize("case", range(len(DENSE)), ids=[f"{c[0]}-{c[1]}-{c[2]}x{c[3]}x{c[4]}{'-lin' if c[5] else ''}"
                                                          for c in DENSE])
def test_random_dense_parity(mmq, case):
    fmt, path, M, N, K, linear, seed = DENSE[case]
    x = synth.activations(seed, M, K, True)
    w = synth.weights(fmt, seed + 1, N, K)
    xq_ref = oracle.quantize_q8_1(x)
    ids = {"auto": mmq.PATH_AUTO, "small": mmq.PATH_SMALL, "tc": mmq.PATH_TC, "expand": mmq.PATH_EXPAND}
    mmq.mmq_set_path(ids[path])
    try:
        out = torch.full((M, N), float("nan"), device="cuda")
        if linear:
            xq = torch.empty((M, K // 32 * 36), dtype=torch.uint8, device="cuda")
            mmq.mmq_linear(dev(x), dev(w), fmt, N, xq=xq, out=out)
        else:
            xq = mmq.mmq_quantize_q8_1(dev(x))
            mmq.gemm(fmt, xq, dev(w), M, N, K, out=out)
        if path != "auto":
            assert mmq.mmq_last_path() == ids[path]
    finally:
        mmq.mmq_set_path(mmq.PATH_AUTO)
    assert np.array_equal(xq.cpu().numpy().reshape(-1), xq_ref.reshape(-1)), "q8_1 bytes differ"
    o = out.cpu().numpy()
    assert not np.isnan(o).any(), "output not fully written"
    ref, norm = oracle.gemm(fmt, xq_ref, w, M, N, K)
    check_close(o, ref, norm, f"{fmt} {path} {M}x{N}x{K}")
    assert mmq.mmq_get_device_error() == 0


def draw_grouped(i):
    """Case i: (fmt, path, R, E, N, K, invalid fraction, seed)."""
    rng = np.random.default_rng(9500 + i)
    fmt = FMTS[rng.integers(len(FMTS))]
    path = ["expand", "small", "tc"][rng.integers(3)]
    if path == "tc" and fmt == "q6_k":
        path = "expand"
    R = log_uniform(rng, 1, 3000)
    E = log_uniform(rng, 1, 64)
    N = log_uniform(rng, 1, 600)
    K = 256 * log_uniform(rng, 1, 8)
    while R * N * K > MAX_WORK:
        N = max(1, N // 2)
    bad = [0.0, 0.0, 0.1][rng.integers(3)]
    return fmt, path, R, E, N, K, bad, 9600 + i


GROUPED = [draw_grouped(i) for i in range(32)]


@pytest.mark.parametrize("case", range(len(GROUPED)), ids=[f"{c[0]}-{c[1]}-R{c[2]}-E{c[3]}-{c[4]}x{c[5]}"
                                                            for c in GROUPED])
def test_random_grouped_parity(mmq, case):
    fmt, path, R, E, N, K, bad, seed = GROUPED[case]
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, E, R).astype(np.int32)
    if bad:
        sel = rng.random(R) < bad
        ids[sel] = np.where(rng.random(int(sel.sum())) < 0.5, -1, E).astype(np.int32)
    x = synth.activations(seed, R, K, True)
    w = synth.weights(fmt, seed + 1, E * N, K)
    xq_ref = oracle.quantize_q8_1(x)
    xq = mmq.mmq_quantize_q8_1(dev(x))
    out = torch.full((R, N), float("nan"), device="cuda")
    pid = {"tc": mmq.PATH_TC, "small": mmq.PATH_SMALL, "expand": mmq.PATH_EXPAND}[path]
    mmq.mmq_set_path(pid)
    try:
        mmq.mmq_gemm_grouped(fmt, xq, dev(ids), dev(w), E, N, K, out=out)
        assert mmq.mmq_last_path() == pid
    finally:
        mmq.mmq_set_path(mmq.PATH_AUTO)
    o = out.cpu().numpy()
    assert not np.isnan(o).any(), "output not fully written"
    ref = np.zeros((R, N))
    norm = np.zeros((R, N))
    rows_w = w.reshape(E, N, -1)
    for e in range(E):
        rows = np.nonzero(ids == e)[0]
        if len(rows):
            r_e, n_e = oracle.gemm(fmt, np.ascontiguousarray(xq_ref[rows]), np.ascontiguousarray(rows_w[e]), len(rows),
                                   N, K)
            ref[rows], norm[rows] = r_e, n_e
    check_close(o, ref, norm, f"grouped {fmt} {path} R={R} E={E} {N}x{K}")
    assert mmq.mmq_get_device_error() == 0
