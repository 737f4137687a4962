"""GPU checks through the C ABI's test hooks.

- The expanded-code contraction's own integer block dots (mmq_debug_product_dots): for the
  K-quants it folds the sub-scale into the weight codes, so its dots are the oracle's raw
  block dots times sc_j, bit for bit ("When the Product Won't Collapse", sec. "The
  obstruction": each constant-scale block is one exact integer sum).
- The two failure statuses a correct call never produces ("13 . r7-r8 raw-byte MMQ
  kernel", sec. 3.3: a launch that did nothing must never pass for a result): a refused
  shared-memory request (MMQ_ERR_SMEM, nothing launched, nothing written) and a pipeline
  wait that runs out (MMQ_ERR_TIMEOUT from the device error word), after which the next
  call is correct again.
- The 7B k/v projection at 2K-token prefill (M = 2048, N = 512, K = 3584) on the automatic
  path, sampled against the oracle.
"""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 1e-4
MMQ_ERR_SMEM, MMQ_ERR_TIMEOUT = -5, -7


@pytest.fixture(scope="module")
def mmq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_quantized_int8_mmq_gb300 as m
    yield m
    m.mmq_set_path(m.PATH_AUTO)
    m.mmq_debug_refuse_smem(False)
    m.mmq_debug_set_wait_limit(-1)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def check_close(out, ref, norm, what):
    err = np.abs(np.asarray(out, dtype=np.float64) - ref)
    bad = err > TOL * norm
    assert not bad.any(), f"{what}: {bad.sum()} entries over tolerance"


def sub_scales(fmt, w, N, K):
    """sc_j of every (row, 32-block), decoded by the oracle from each super-block's 12 scale bytes."""
    sb = 144 if fmt == "q4_k" else 176
    ng = K // 256
    rows = w.reshape(N, ng, sb)
    sc = np.zeros((N, K // 32), dtype=np.int64)
    for n in range(N):
        for g in range(ng):
            p = np.ascontiguousarray(rows[n, g, 4:16])
            for j in range(8):
                sc[n, 8 * g + j] = oracle.q4_k_scale_min(p, j)[0]
    return sc


# several tiles of either width plus ragged tails; 300 x 520 x 1024 splits K in two
PRODUCT_SHAPES = [(5, 9, 256), (70, 150, 512), (129, 257, 1024), (300, 520, 1024)]


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k", "q5_k", "q6_k"])
def test_product_dots_bit_exact(mmq, fmt):
    for (M, N, K) in PRODUCT_SHAPES:
        x = synth.activations(M * 3 + 31, M, K, True)
        w = synth.weights(fmt, N * 5 + 17, N, K)
        xq = mmq.mmq_quantize_q8_1(dev(x))
        dots = mmq.mmq_debug_product_dots(fmt, xq, dev(w), M, N, K).cpu().numpy().astype(np.int64)
        assert mmq.mmq_last_path() == mmq.PATH_EXPAND
        ref = oracle.block_dots(fmt, oracle.quantize_q8_1(x), w, M, N, K).astype(np.int64)
        if fmt in ("q4_k", "q5_k"):
            ref = ref * sub_scales(fmt, w, N, K)[None, :, :]
        assert np.array_equal(dots, ref), f"{fmt} {M}x{N}x{K}: product dots differ"
    assert mmq.mmq_get_device_error() == 0


def test_product_dots_extreme_q5_k(mmq):
    # the largest folded dot: activation codes +-127, Q5_K codes 31, every sub-scale 63:
    # |D| = 32 * 127 * 31 * 63 = 7936992
    M, N, K = 130, 100, 512
    xs = np.where(np.arange(M)[:, None] % 2 == 0, 1.0, -1.0) * np.ones((M, K))
    xs = xs.astype(np.float32)       # every block all +127 or all -127
    w = synth.weights("q5_k", 5, N, K).reshape(N, K // 256, 176).copy()
    w[:, :, 4:16] = 0xFF            # sc_j = m_j = 63 for every j
    w[:, :, 16:] = 0xFF             # every code 31
    w = w.reshape(N, -1)
    xq = mmq.mmq_quantize_q8_1(dev(xs))
    dots = mmq.mmq_debug_product_dots("q5_k", xq, dev(w), M, N, K).cpu().numpy().astype(np.int64)
    ref = oracle.block_dots("q5_k", oracle.quantize_q8_1(xs), w, M, N, K).astype(np.int64) * 63
    assert np.abs(ref).min() == np.abs(ref).max() == 7936992
    assert np.array_equal(dots, ref)


def test_refused_shared_memory_launches_and_writes_nothing(mmq):
    M, N, K = 256, 384, 512
    x = synth.activations(91, M, K, True)
    w = synth.weights("q4_k", 92, N, K)
    xq = mmq.mmq_quantize_q8_1(dev(x))
    wd = dev(w)
    torch.cuda.synchronize()
    out = torch.full((M, N), float("nan"), device="cuda")
    mmq.mmq_profile_read(reset=True)
    prev_prof = mmq.mmq_profile_enable(True)
    mmq.mmq_debug_refuse_smem(True)
    try:
        for path in (mmq.PATH_EXPAND, mmq.PATH_TC):
            mmq.mmq_set_path(path)
            with pytest.raises(mmq.MMQError) as e:
                mmq.mmq_gemm_q4_k(xq, wd, M, N, K, out=out)
            assert e.value.status == MMQ_ERR_SMEM
        with pytest.raises(mmq.MMQError) as e:
            mmq.mmq_gemm_noalloc("q4_k", xq, wd, M, N, K, out=out)
        assert e.value.status == MMQ_ERR_SMEM
    finally:
        mmq.mmq_debug_refuse_smem(False)
        mmq.mmq_set_path(mmq.PATH_AUTO)
    torch.cuda.synchronize()
    assert mmq.mmq_profile_read(reset=True) == {}, "a refused call launched a kernel"
    mmq.mmq_profile_enable(prev_prof)
    assert torch.isnan(out).all(), "a refused call wrote the output"
    # and the same call goes through once the switch is off
    mmq.mmq_set_path(mmq.PATH_EXPAND)
    try:
        mmq.mmq_gemm_q4_k(xq, wd, M, N, K, out=out)
    finally:
        mmq.mmq_set_path(mmq.PATH_AUTO)
    ref, norm = oracle.gemm("q4_k", oracle.quantize_q8_1(x), w, M, N, K)
    check_close(out.cpu().numpy(), ref, norm, "after the refusal")


def test_wait_timeout_is_reported_and_the_next_call_is_correct(mmq):
    M, N, K = 512, 3584, 3584
    x = synth.activations(93, M, K, True)
    w = synth.weights("q8_0", 94, N, K)
    xq = mmq.mmq_quantize_q8_1(dev(x))
    wd = dev(w)
    out = torch.full((M, N), float("nan"), device="cuda")
    torch.cuda.synchronize()
    assert mmq.mmq_get_device_error() == 0
    mmq.mmq_set_path(mmq.PATH_EXPAND)
    try:
        # a bound of 0: the first wait whose phase is not already complete gives up (the
        # MMA issuers' first wait on a copy just started, at the latest)
        mmq.mmq_debug_set_wait_limit(0)
        mmq.mmq_gemm_q8_0(xq, wd, M, N, K, out=out)
        assert mmq.mmq_get_device_error() == MMQ_ERR_TIMEOUT
        assert mmq.mmq_get_device_error() == 0, "the error word is read and cleared"
    finally:
        mmq.mmq_debug_set_wait_limit(-1)
    try:
        out.fill_(float("nan"))
        mmq.mmq_gemm_q8_0(xq, wd, M, N, K, out=out)
        assert mmq.mmq_get_device_error() == 0
    finally:
        mmq.mmq_set_path(mmq.PATH_AUTO)
    o = out.cpu().numpy()
    assert not np.isnan(o).any()
    rng = np.random.default_rng(3)
    im, inn = rng.integers(0, M, 500), rng.integers(0, N, 500)
    ref, norm = oracle.gemm_at("q8_0", oracle.quantize_q8_1(x), w, M, N, K, im, inn)
    check_close(o[im, inn], ref, norm, "after the timeout")


def test_kv_projection_at_prefill_sampled_parity(mmq):
    M, N, K = 2048, 512, 3584
    x = synth.layer_activations(0, M, K, 0)
    w = synth.layer_weights(0, "k", N, K)
    mmq.mmq_set_path(mmq.PATH_AUTO)
    xq = mmq.mmq_quantize_q8_1(dev(x))
    out = torch.full((M, N), float("nan"), device="cuda")
    mmq.mmq_gemm_q4_k(xq, dev(w), M, N, K, out=out)
    assert mmq.mmq_last_path() == mmq.PATH_EXPAND
    o = out.cpu().numpy()
    assert not np.isnan(o).any()
    xq_ref = oracle.quantize_q8_1(x)
    assert np.array_equal(xq.cpu().numpy(), xq_ref)
    rng = np.random.default_rng(4)
    im = np.concatenate([rng.integers(0, M, 3000), [0, M - 1, 127, 128, M - 1]])
    inn = np.concatenate([rng.integers(0, N, 3000), [0, N - 1, 95, 96, 0]])
    ref, norm = oracle.gemm_at("q4_k", xq_ref, w, M, N, K, im, inn)
    check_close(o[im, inn], ref, norm, "k/v projection 2048x512x3584")
    assert mmq.mmq_get_device_error() == 0
