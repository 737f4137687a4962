"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the same
seeded operands.

Acceptance (the method's own bar):
  - q8_1 quantization: bit-exact bytes (codes, f16 d, f16 s);
  - per-block int32 dots from the debug hook: bit-exact;
  - f32 outputs: |gpu - oracle| <= TOL * sum_b |terms| per entry, TOL = 1e-4, where the
    oracle is the fp64 contraction on the same quantized operands.
Shapes: small ones the oracle computes in full (spanning several tiles plus ragged
tails), and the full workload sizes checked on sampled entries.
"""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL = 1e-4
PATHS = ["small", "tc", "expand"]
PATH_IDS = {"small": 1, "tc": 2, "expand": 3}


@pytest.fixture(scope="module")
def mmq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import block_quantized_int8_mmq_gb300 as m
    yield m
    m.mmq_set_path(m.PATH_AUTO)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def set_path(mmq, path):
    mmq.mmq_set_path({"auto": mmq.PATH_AUTO, "small": mmq.PATH_SMALL, "tc": mmq.PATH_TC,
                      "expand": mmq.PATH_EXPAND}[path])


def check_close(out, ref, norm, what=""):
    out = np.asarray(out, dtype=np.float64)
    err = np.abs(out - ref)
    bad = err > TOL * norm
    if bad.any():
        i = np.argmax(np.where(norm > 0, err / np.maximum(norm, 1e-300), np.inf))
        raise AssertionError(f"{what}: {bad.sum()} entries over tolerance; worst at flat index {i}: "
                             f"gpu {out.flat[i]!r} oracle {ref.flat[i]!r} norm {norm.flat[i]!r}")


# ------------------------------------------------------------------ quantize

def tricky_activations(M=16, K=256):
    rng = np.random.default_rng(5)
    x = rng.normal(size=(M, K))
    x[0] = 0.0                                                  # all-zero row
    x[1, :32] = 3.25                                            # all-equal block
    x[1, 32:64] = (np.arange(32) - 16) * 0.5                    # half-integer ties
    x[2] *= 1e-3                                                # f16-subnormal scales
    x[3] *= 1e-30                                               # tiny values
    x[4] *= 3e3                                                 # large values
    x[5, :32] = [127, 62.5, 2.5, 1.5, 0.5, -0.5, -1.5, -2.5] + [0] * 24
    x[6, :32] = np.arange(32) - 16
    x[7, ::7] = -0.0
    x[8] = np.where(np.arange(K) % 32 == 3, 5.0, 0.0)           # one nonzero per block
    return x.astype(np.float32)


@pytest.mark.parametrize("M,K", [(1, 32), (3, 96), (17, 512), (64, 512), (512, 3584), (2048, 18944)])
def test_quantize_bit_exact(mmq, M, K):
    x = synth.activations(1000 + M, M, K, True)
    xq = mmq.mmq_quantize_q8_1(dev(x))
    assert np.array_equal(xq.cpu().numpy(), oracle.quantize_q8_1(x))


def test_quantize_edge_blocks_bit_exact(mmq):
    x = tricky_activations()
    xq = mmq.mmq_quantize_q8_1(dev(x))
    assert np.array_equal(xq.cpu().numpy(), oracle.quantize_q8_1(x))


def test_quantize_true_division_example(mmq):
    # a block where x/d and x*(1/d) round to different codes (hand example E5)
    from conftest import as_floats, read_golden
    g = read_golden("hand_examples.txt")
    x = np.array(as_floats(g["e5_x"]), dtype=np.float32)[None, :]
    xq = mmq.mmq_quantize_q8_1(dev(x))
    assert np.array_equal(xq.cpu().numpy(), oracle.quantize_q8_1(x))


# ------------------------------------------------------------------ contractions, full compare

SMALL_SHAPES = {
    "q8_0": [(1, 1, 32), (3, 7, 64), (9, 33, 512), (64, 256, 512), (130, 200, 1024), (257, 129, 2304),
             (8, 300, 3584)],
    "q4_k": [(1, 1, 256), (3, 7, 256), (9, 33, 512), (64, 256, 512), (130, 200, 1024), (257, 129, 2304),
             (8, 300, 3584)],
}
SMALL_SHAPES["q5_k"] = SMALL_SHAPES["q6_k"] = SMALL_SHAPES["q4_k"]
FMTS = ["q8_0", "q4_k", "q5_k", "q6_k"]
NO_TC = ("q6_k",)  # formats the converter kernel refuses


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("fmt", FMTS)
def test_gemm_parity_full(mmq, fmt, path):
    if fmt in NO_TC and path == "tc":
        pytest.skip("the converter kernel takes Q8_0 and Q4_K (refusal tested below)")
    set_path(mmq, path)
    for (M, N, K) in SMALL_SHAPES[fmt]:
        if path != "small" and K % 256:
            continue  # the tensor-core paths stage 256-value groups (refusal tested below)
        x = synth.activations(M * 7 + N, M, K, True)
        w = synth.weights(fmt, M + N * 3, N, K)
        xq = mmq.mmq_quantize_q8_1(dev(x))
        out = mmq.gemm(fmt, xq, dev(w), M, N, K)
        assert mmq.mmq_last_path() == PATH_IDS[path]
        ref, norm = oracle.gemm(fmt, oracle.quantize_q8_1(x), w, M, N, K)
        check_close(out.cpu().numpy(), ref, norm, f"{fmt} {path} {M}x{N}x{K}")
    assert mmq.mmq_get_device_error() == 0


@pytest.mark.parametrize("path", ["tc", "expand"])
def test_tc_paths_refuse_partial_k_groups_and_auto_routes_them(mmq, path):
    M, N, K = 80, 40, 96
    x = synth.activations(21, M, K, True)
    w = synth.q8_0_weights(22, N, K)
    xq = mmq.mmq_quantize_q8_1(dev(x))
    set_path(mmq, path)
    with pytest.raises(mmq.MMQError) as e:
        mmq.mmq_gemm_q8_0(xq, dev(w), M, N, K)
    assert e.value.status == -2
    set_path(mmq, "auto")
    out = mmq.mmq_gemm_q8_0(xq, dev(w), M, N, K)
    assert mmq.mmq_last_path() == mmq.PATH_SMALL
    ref, norm = oracle.gemm("q8_0", oracle.quantize_q8_1(x), w, M, N, K)
    check_close(out.cpu().numpy(), ref, norm, "auto K % 256 != 0")


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("fmt", FMTS)
def test_block_dots_bit_exact(mmq, fmt, path):
    if fmt in NO_TC and path == "tc":
        pytest.skip("the converter kernel takes Q8_0 and Q4_K")
    set_path(mmq, path)
    for (M, N, K) in [(5, 9, 256), (70, 150, 512), (129, 257, 1024)]:
        x = synth.activations(M + 11, M, K, True)
        w = synth.weights(fmt, N + 13, N, K)
        xq = mmq.mmq_quantize_q8_1(dev(x))
        dots = mmq.block_dots(fmt, xq, dev(w), M, N, K)
        ref = oracle.block_dots(fmt, oracle.quantize_q8_1(x), w, M, N, K)
        assert np.array_equal(dots.cpu().numpy(), ref), f"{fmt} {path} {M}x{N}x{K}"


# Outputs with fewer 128 x 128 tiles than SMs: the expanded path splits K across up to 8
# CTAs per tile (each at least two 256-value groups) and sums their partial tiles in a fixed
# order; M * N not a multiple of 4 takes the summing kernel's scalar tail.
SPLIT_SHAPES = [(7, 33, 2304), (130, 131, 4096), (1, 1, 1024), (128, 128, 512), (200, 300, 18944)]


@pytest.mark.parametrize("fmt", FMTS)
def test_split_k_parity_dots_and_determinism(mmq, fmt):
    set_path(mmq, "expand")
    for (M, N, K) in SPLIT_SHAPES:
        x = synth.activations(M * 5 + K, M, K, True)
        w = synth.weights(fmt, N * 7 + K, N, K)
        xq = mmq.mmq_quantize_q8_1(dev(x))
        wd = dev(w)
        out = mmq.gemm(fmt, xq, wd, M, N, K)
        again = mmq.gemm(fmt, xq, wd, M, N, K)
        assert torch.equal(out, again), f"{fmt} {M}x{N}x{K}: not deterministic"
        ref, norm = oracle.gemm(fmt, oracle.quantize_q8_1(x), w, M, N, K)
        check_close(out.cpu().numpy(), ref, norm, f"{fmt} split {M}x{N}x{K}")
        if M * N * K <= 130 * 131 * 4096:
            dots = mmq.block_dots(fmt, xq, wd, M, N, K)
            assert np.array_equal(dots.cpu().numpy(), oracle.block_dots(fmt, oracle.quantize_q8_1(x), w, M, N, K))
    assert mmq.mmq_get_device_error() == 0


# 96-wide weight tiles (taken where the 128-wide ones would leave SMs idle): the last tile
# cut inside an epilogue warp's 24 columns, N odd or not a multiple of 4 (scalar stores)
NARROW_SHAPES = [(300, 3300, 512), (300, 3301, 512), (257, 3850, 768)]


@pytest.mark.parametrize("fmt", FMTS)
def test_narrow_tile_parity_and_determinism(mmq, fmt):
    set_path(mmq, "expand")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for (M, N, K) in NARROW_SHAPES:
        bn, splits = mmq.mmq_debug_expand_tiling(fmt, M, N, K)
        if sms == 152:
            assert (bn, splits) == (96, 1), f"{M}x{N}x{K}: tiling {bn}, {splits}"
        x = synth.activations(M * 3 + N, M, K, True)
        w = synth.weights(fmt, N * 5 + K, N, K)
        xq = mmq.mmq_quantize_q8_1(dev(x))
        wd = dev(w)
        out = torch.full((M, N), float("nan"), device="cuda")
        mmq.gemm(fmt, xq, wd, M, N, K, out=out)
        again = mmq.gemm(fmt, xq, wd, M, N, K)
        assert torch.equal(out, again), f"{fmt} {M}x{N}x{K}: not deterministic"
        o = out.cpu().numpy()
        assert not np.isnan(o).any(), "output not fully written"
        ref, norm = oracle.gemm(fmt, oracle.quantize_q8_1(x), w, M, N, K)
        check_close(o, ref, norm, f"{fmt} narrow tiles {M}x{N}x{K}")
    assert mmq.mmq_get_device_error() == 0


# one to eight activation rows on the small path: weight rows dealt out to warps (several
# rows per warp when N exceeds the resident warps), rows of 1 to 10 pieces with a partial
# last piece, N = 1, and token counts that leave part of a 4- or 8-row pass empty
STREAM_SHAPES = [(1, 1, 256), (2, 7, 2304), (1, 300, 3584), (2, 77, 18944), (1, 40000, 256), (2, 9000, 512),
                 (3, 77, 2304), (4, 300, 3584), (5, 9000, 512), (8, 513, 3584), (7, 40, 7168)]


@pytest.mark.parametrize("route", ["auto", "mma"])
@pytest.mark.parametrize("fmt", FMTS)
def test_few_row_stream_parity_and_dots(mmq, fmt, route):
    set_path(mmq, "small")
    mmq.mmq_debug_small_route(mmq.SMALL_ROUTE_MMA if route == "mma" else mmq.SMALL_ROUTE_AUTO)
    try:
        few_row_cases(mmq, fmt)
    finally:
        mmq.mmq_debug_small_route(mmq.SMALL_ROUTE_AUTO)


def few_row_cases(mmq, fmt):
    for (M, N, K) in STREAM_SHAPES:
        x = synth.activations(M * 5 + N, M, K, True)
        w = synth.weights(fmt, N * 7 + K, N, K)
        xq = mmq.mmq_quantize_q8_1(dev(x))
        xq_ref = oracle.quantize_q8_1(x)
        out = mmq.gemm(fmt, xq, dev(w), M, N, K)
        ref, norm = oracle.gemm(fmt, xq_ref, w, M, N, K)
        check_close(out.cpu().numpy(), ref, norm, f"{fmt} stream {M}x{N}x{K}")
        if N * K <= 300 * 18944:
            dots = mmq.block_dots(fmt, xq, dev(w), M, N, K)
            assert np.array_equal(dots.cpu().numpy(), oracle.block_dots(fmt, xq_ref, w, M, N, K)), \
                f"{fmt} stream dots {M}x{N}x{K}"
    assert mmq.mmq_get_device_error() == 0


# the Q6_K tensor-core stream (K % 512 == 0, N % 8 == 0): 128-row boxes with rows past N
# (8, 136, 1000, 4104 rows), one to eight rows and passes with rows past M, K split over
# clusters of 1, 2, 4 and 8 CTAs (the split is chosen from the boxes and the K chunks:
# S = 1 for 8 x 512, 2 for 136 x 1024, 4 for 1000 x 2048 and 3584 x 3584, 8 for 128 x 7168),
# several passes (17 and 13 rows), and the one-row case the tensor-core route forces
Q6S_SHAPES = [(1, 8, 512), (2, 136, 1024), (3, 1000, 2048), (8, 128, 7168), (5, 3584, 3584), (8, 4104, 4096),
              (13, 264, 1536), (17, 64, 1024), (8, 18944, 512), (6, 2048, 18944)]


@pytest.mark.parametrize("route", ["auto", "mma"])
def test_q6_k_tensor_core_stream_parity_and_dots(mmq, route):
    set_path(mmq, "small")
    mmq.mmq_debug_small_route(mmq.SMALL_ROUTE_MMA if route == "mma" else mmq.SMALL_ROUTE_AUTO)
    try:
        for (M, N, K) in Q6S_SHAPES:
            x = synth.activations(M * 13 + N, M, K, True)
            w = synth.weights("q6_k", N * 3 + K, N, K)
            xq = mmq.mmq_quantize_q8_1(dev(x))
            xq_ref = oracle.quantize_q8_1(x)
            wd = dev(w)
            out = torch.full((M, N), float("nan"), device="cuda")
            mmq.gemm("q6_k", xq, wd, M, N, K, out=out)
            again = mmq.gemm("q6_k", xq, wd, M, N, K)
            assert torch.equal(out, again), f"{M}x{N}x{K}: not deterministic"
            o = out.cpu().numpy()
            assert not np.isnan(o).any(), f"{M}x{N}x{K}: output not fully written"
            if M * N * K <= 2e9:
                ref, norm = oracle.gemm("q6_k", xq_ref, w, M, N, K)
                check_close(o, ref, norm, f"q6_k tensor-core stream {M}x{N}x{K}")
            else:
                im, inn = sample_entries(M, N, 1500, M + N)
                ref, norm = oracle.gemm_at("q6_k", xq_ref, w, M, N, K, im, inn)
                check_close(o[im, inn], ref, norm, f"q6_k tensor-core stream {M}x{N}x{K}")
            if N * K <= 4200 * 4096:
                dots = mmq.block_dots("q6_k", xq, wd, M, N, K)
                assert np.array_equal(dots.cpu().numpy(), oracle.block_dots("q6_k", xq_ref, w, M, N, K)), \
                    f"q6_k tensor-core stream dots {M}x{N}x{K}"
    finally:
        mmq.mmq_debug_small_route(mmq.SMALL_ROUTE_AUTO)
    assert mmq.mmq_get_device_error() == 0


# AUTO above eight Q6_K rows follows the Q6_K stream's cost model (waves of CTAs x chunks
# per CTA) against the expanded path's; these are the measured sides of its crossovers on
# GB300 (small / expanded, us): 16 x 18944 x 3584 31 / 106, 64 x 18944 x 3584 118 / 107,
# 32 x 3584^2 15.1 / 23.7, 48 x 3584^2 29.0 / 24.4, 128 x 512 x 3584 11.1 / 15.3
Q6_AUTO = [((16, 18944, 3584), "small"), ((64, 18944, 3584), "expand"), ((32, 3584, 3584), "small"),
           ((48, 3584, 3584), "expand"), ((128, 512, 3584), "small")]


def test_q6_k_auto_path_follows_the_stream_cost_model(mmq):
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the crossovers are those of a 152-SM GB300")
    set_path(mmq, "auto")
    for (M, N, K), want in Q6_AUTO:
        x = synth.activations(M + N + K, M, K, True)
        w = synth.weights("q6_k", N + 2 * K, N, K)
        xq_ref = oracle.quantize_q8_1(x)
        out = mmq.gemm("q6_k", mmq.mmq_quantize_q8_1(dev(x)), dev(w), M, N, K)
        assert mmq.mmq_last_path() == PATH_IDS[want], f"{M}x{N}x{K}: path {mmq.mmq_last_path()}, expected {want}"
        im, inn = sample_entries(M, N, 1000, M * 7 + N)
        ref, norm = oracle.gemm_at("q6_k", xq_ref, w, M, N, K, im, inn)
        check_close(out.cpu().numpy()[im, inn], ref, norm, f"q6_k auto {M}x{N}x{K}")
    assert mmq.mmq_get_device_error() == 0


# three to a hundred rows on the small path (the int8 tensor-core stream, 8 rows per pass):
# passes with rows past M, weight tiles with rows past N, one to hundreds of tiles
# (3, 5000, 512) and (4, 18944, 768): three or four rows of a wide weight, which the K-quants
# take on the int8 stream (one partly empty pass) rather than the dp4a stream
TCS_SHAPES = [(3, 1, 256), (16, 129, 768), (17, 300, 2304), (32, 128, 512), (33, 3584, 256), (64, 200, 3584),
              (100, 1000, 1024), (5, 18944, 512), (3, 5000, 512), (4, 18944, 768)]


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k", "q5_k"])
def test_tens_of_rows_small_path_parity_and_dots(mmq, fmt):
    set_path(mmq, "small")
    for (M, N, K) in TCS_SHAPES:
        x = synth.activations(M * 11 + N, M, K, True)
        w = synth.weights(fmt, N * 5 + K, N, K)
        xq = mmq.mmq_quantize_q8_1(dev(x))
        xq_ref = oracle.quantize_q8_1(x)
        out = torch.full((M, N), float("nan"), device="cuda")
        mmq.gemm(fmt, xq, dev(w), M, N, K, out=out)
        o = out.cpu().numpy()
        assert not np.isnan(o).any(), f"{fmt} {M}x{N}x{K}: output not fully written"
        ref, norm = oracle.gemm(fmt, xq_ref, w, M, N, K)
        check_close(o, ref, norm, f"{fmt} small {M}x{N}x{K}")
        again = mmq.gemm(fmt, xq, dev(w), M, N, K)
        assert torch.equal(again, out), f"{fmt} {M}x{N}x{K}: repeat differs"
        if M * N * K <= 64 * 1000 * 3584:
            dots = mmq.block_dots(fmt, xq, dev(w), M, N, K)
            assert np.array_equal(dots.cpu().numpy(), oracle.block_dots(fmt, xq_ref, w, M, N, K)), \
                f"{fmt} small dots {M}x{N}x{K}"
    assert mmq.mmq_get_device_error() == 0


# K splits of the Q8_0 / Q4_K / Q5_K tensor-core streams, forced to 2, 3, 5 and 8 splits
# with 1 to 4 boxes per CTA: super-blocks dealt unevenly among the splits (K = 2048 under 8
# splits: one each), passes with rows past M, boxes with rows past N, CTAs with fewer boxes
# than the others.  Within the tolerance, the same bits on a
# second call, and the summing kernel launched once per call.
KSPLIT_SHAPES = [(1, 40, 2048), (3, 77, 4096), (8, 264, 4608), (13, 520, 2816), (9, 33, 7168)]


@pytest.mark.parametrize("fmt", ["q8_0", "q4_k", "q5_k"])
def test_stream_k_split_parity_and_determinism(mmq, fmt):
    set_path(mmq, "small")
    route = mmq.mmq_debug_small_route(mmq.SMALL_ROUTE_MMA)
    try:
        for (M, N, K) in KSPLIT_SHAPES:
            x = synth.activations(M * 13 + N, M, K, True)
            w = synth.weights(fmt, N * 3 + K, N, K)
            xq = mmq.mmq_quantize_q8_1(dev(x))
            wd = dev(w)
            ref, norm = oracle.gemm(fmt, oracle.quantize_q8_1(x), w, M, N, K)
            mmq.mmq_debug_small_ksplit(1)
            whole = mmq.gemm(fmt, xq, wd, M, N, K)
            check_close(whole.cpu().numpy(), ref, norm, f"{fmt} {M}x{N}x{K} unsplit")
            for z, boxes in ((2, 0), (3, 2), (5, 4), (8, 3)):
                mmq.mmq_debug_small_ksplit(z, boxes)
                torch.cuda.synchronize()
                mmq.mmq_profile_read(reset=True)
                was = mmq.mmq_profile_enable(True)
                try:
                    out = torch.full((M, N), float("nan"), device="cuda")
                    mmq.gemm(fmt, xq, wd, M, N, K, out=out)
                    torch.cuda.synchronize()
                    prof = mmq.mmq_profile_read(reset=True)
                finally:
                    mmq.mmq_profile_enable(was)
                assert prof.get("k_stream_ksum", (0, 0))[0] == 1, (fmt, M, N, K, z, prof)
                o = out.cpu().numpy()
                assert not np.isnan(o).any(), f"{fmt} {M}x{N}x{K} z={z}: output not fully written"
                check_close(o, ref, norm, f"{fmt} {M}x{N}x{K} z={z}")
                again = mmq.gemm(fmt, xq, wd, M, N, K)
                assert torch.equal(again, out), f"{fmt} {M}x{N}x{K} z={z}: repeat differs"
    finally:
        mmq.mmq_debug_small_ksplit(0)
        mmq.mmq_debug_small_route(route)
    assert mmq.mmq_get_device_error() == 0


# the Q6_K tensor-core stream split over independent CTAs (forced 2, 3 and 5 splits: chunks
# dealt unevenly, several passes, boxes with rows past N) against the oracle, the same bits
# on a second call, and the summing kernel launched once
@pytest.mark.parametrize("M,N,K", [(8, 128, 7168), (13, 264, 1536), (5, 1000, 5120), (3, 3584, 3584)])
def test_q6_k_stream_split_parity(mmq, M, N, K):
    set_path(mmq, "small")
    route = mmq.mmq_debug_small_route(mmq.SMALL_ROUTE_MMA)
    try:
        x = synth.activations(M * 17 + N, M, K, True)
        w = synth.weights("q6_k", N * 11 + K, N, K)
        xq, wd = mmq.mmq_quantize_q8_1(dev(x)), dev(w)
        ref, norm = oracle.gemm("q6_k", oracle.quantize_q8_1(x), w, M, N, K)
        for z in (2, 3, 5):
            mmq.mmq_debug_small_ksplit(z, 0)
            torch.cuda.synchronize()
            mmq.mmq_profile_read(reset=True)
            was = mmq.mmq_profile_enable(True)
            try:
                out = torch.full((M, N), float("nan"), device="cuda")
                mmq.gemm("q6_k", xq, wd, M, N, K, out=out)
                torch.cuda.synchronize()
                prof = mmq.mmq_profile_read(reset=True)
            finally:
                mmq.mmq_profile_enable(was)
            assert prof.get("k_mmq_q6_stream", (0, 0))[0] == 1, prof
            assert prof.get("k_stream_ksum", (0, 0))[0] == 1, (M, N, K, z, prof)
            o = out.cpu().numpy()
            assert not np.isnan(o).any(), f"q6_k {M}x{N}x{K} z={z}: output not fully written"
            check_close(o, ref, norm, f"q6_k {M}x{N}x{K} z={z}")
            assert torch.equal(mmq.gemm("q6_k", xq, wd, M, N, K), out), f"q6_k {M}x{N}x{K} z={z}: repeat differs"
    finally:
        mmq.mmq_debug_small_ksplit(0)
        mmq.mmq_debug_small_route(route)
    assert mmq.mmq_get_device_error() == 0


# the measured rule: 3 boxes per CTA x 4 splits for 3584 x 18944 through eight rows (against
# 224 one-box CTAs of 74 super-blocks on 152 SMs) and 3 x 2 through sixteen, none for
# 18944 x 3584 at eight or sixteen rows; the split call in a
# captured graph (its scratch a graph allocation outside the chain of kernels) replays to
# the eager call's bits, next to an unsplit call captured after it
@pytest.mark.parametrize("fmt", ["q8_0", "q4_k", "q5_k"])
def test_stream_k_split_rule_and_graph_capture(mmq, fmt):
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the grids are those of a 152-SM GB300")
    set_path(mmq, "auto")
    route = mmq.mmq_debug_small_route(mmq.SMALL_ROUTE_AUTO)
    mmq.mmq_debug_small_ksplit(0)
    try:
        def launches(M, N, K, xq, wd):
            torch.cuda.synchronize()
            mmq.mmq_profile_read(reset=True)
            was = mmq.mmq_profile_enable(True)
            try:
                out = mmq.gemm(fmt, xq, wd, M, N, K)
                torch.cuda.synchronize()
                return out, mmq.mmq_profile_read(reset=True)
            finally:
                mmq.mmq_profile_enable(was)

        M, N, K = 8, 3584, 18944
        x = synth.activations(77, M, K, True)
        w = synth.weights(fmt, 78, N, K)
        xq, wd = mmq.mmq_quantize_q8_1(dev(x)), dev(w)
        eager, prof = launches(M, N, K, xq, wd)
        assert prof.get("k_stream_ksum", (0, 0))[0] == 1, prof
        im, inn = sample_entries(M, N, 400, 5)
        ref, norm = oracle.gemm_at(fmt, oracle.quantize_q8_1(x), w, M, N, K, im, inn)
        check_close(eager.cpu().numpy()[im, inn], ref, norm, f"{fmt} {M}x{N}x{K} split")
        for (m2, n2, k2) in [(8, 18944, 3584), (16, 18944, 3584)]:
            x2 = synth.activations(m2 + n2, m2, k2, True)
            w2 = synth.weights(fmt, n2 + k2, n2, k2)
            _, p2 = launches(m2, n2, k2, mmq.mmq_quantize_q8_1(dev(x2)), dev(w2))
            assert "k_stream_ksum" not in p2, (m2, n2, k2, p2)
        # two passes through the long K: 3 boxes x 2 splits in one wave
        x3 = synth.activations(81, 16, K, True)
        out3, p3 = launches(16, N, K, mmq.mmq_quantize_q8_1(dev(x3)), wd)
        assert p3.get("k_stream_ksum", (0, 0))[0] == 1, p3
        im, inn = sample_entries(16, N, 400, 6)
        ref, norm = oracle.gemm_at(fmt, oracle.quantize_q8_1(x3), w, 16, N, K, im, inn)
        check_close(out3.cpu().numpy()[im, inn], ref, norm, f"{fmt} 16x{N}x{K} split")

        x2 = synth.activations(79, 4, 3584, True)
        w2 = synth.weights(fmt, 80, 512, 3584)
        xq2, wd2 = mmq.mmq_quantize_q8_1(dev(x2)), dev(w2)
        eager2 = mmq.gemm(fmt, xq2, wd2, 4, 512, 3584)
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        out = torch.full((M, N), float("nan"), device="cuda")
        out2 = torch.full((4, 512), float("nan"), device="cuda")
        with torch.cuda.graph(g, stream=s):
            mmq.gemm(fmt, xq, wd, M, N, K, out=out, stream=s)
            mmq.gemm(fmt, xq2, wd2, 4, 512, 3584, out=out2, stream=s)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, eager), f"{fmt}: captured split call differs from the eager one"
        assert torch.equal(out2, eager2), f"{fmt}: captured call after the split differs"
        del g
    finally:
        mmq.mmq_debug_small_ksplit(0)
        mmq.mmq_debug_small_route(route)
    assert mmq.mmq_get_device_error() == 0


# quantize + contraction in one call: on the expanded path the quantize is fused into the
# activation expansion.  xq must hold the q8_1 bytes of x and out must equal the separate
# quantize + gemm calls on the same path bit for bit (same kernels downstream of the
# expanded operands), and the oracle within tolerance.
@pytest.mark.parametrize("path", ["auto", "expand", "small", "tc"])
@pytest.mark.parametrize("fmt", FMTS)
def test_linear_matches_separate_calls(mmq, fmt, path):
    if fmt in NO_TC and path == "tc":
        pytest.skip("the converter kernel takes Q8_0 and Q4_K")
    set_path(mmq, path)
    # (100, 600, 512): five weight tiles per activation tile, so the fused quantize is
    # spread over one CTA per 32-block
    for (M, N, K) in [(300, 200, 1024), (129, 257, 2304), (4, 130, 512), (513, 64, 256), (100, 600, 512)]:
        x = synth.activations(M + 3 * N + K, M, K, True)
        w = synth.weights(fmt, 2 * M + N, N, K)
        xd, wd = dev(x), dev(w)
        xq = torch.full((M, K // 32 * 36), 0xAB, dtype=torch.uint8, device="cuda")
        out = mmq.mmq_linear(xd, wd, fmt, N, xq=xq)
        taken = mmq.mmq_last_path()
        xq_ref = oracle.quantize_q8_1(x)
        assert np.array_equal(xq.cpu().numpy(), xq_ref), f"{fmt} {path} {M}x{N}x{K}: q8_1 bytes"
        sep = mmq.gemm(fmt, mmq.mmq_quantize_q8_1(xd), wd, M, N, K)
        assert mmq.mmq_last_path() == taken
        assert torch.equal(out, sep), f"{fmt} {path} {M}x{N}x{K}: fused != separate"
        ref, norm = oracle.gemm(fmt, xq_ref, w, M, N, K)
        check_close(out.cpu().numpy(), ref, norm, f"{fmt} linear {path} {M}x{N}x{K}")
    assert mmq.mmq_get_device_error() == 0


# 6 tiles: K = 512 (two groups) is not split, K = 1024 is split in two and summed
@pytest.mark.parametrize("K,kernels", [(512, {"k_expand", "k_mmq_tcx"}),
                                       (1024, {"k_expand", "k_mmq_tcx", "k_splitk_sum"})])
def test_linear_graph_capture(mmq, K, kernels):
    set_path(mmq, "expand")
    M, N = 256, 384
    x = synth.activations(91, M, K, True)
    w = synth.q4_k_weights(92, N, K)
    xd, wd = dev(x), dev(w)
    xq = torch.empty((M, K // 32 * 36), dtype=torch.uint8, device="cuda")
    out = torch.full((M, N), float("nan"), device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    prev = mmq.mmq_profile_enable(True)
    try:
        with torch.cuda.graph(g, stream=s):
            mmq.mmq_linear(xd, wd, "q4_k", N, xq=xq, out=out, stream=s)
        g.replay()
        torch.cuda.synchronize()
        prof = mmq.mmq_profile_read(reset=True)
    finally:
        mmq.mmq_profile_enable(prev)
    assert set(prof) == kernels and all(n == 1 for n, _ in prof.values()), prof
    xq_ref = oracle.quantize_q8_1(x)
    assert np.array_equal(xq.cpu().numpy(), xq_ref)
    ref, norm = oracle.gemm("q4_k", xq_ref, w, M, N, K)
    check_close(out.cpu().numpy(), ref, norm, "captured linear")
    assert mmq.mmq_get_device_error() == 0


@pytest.mark.parametrize("path", PATHS)
def test_extreme_codes_block_dots(mmq, path):
    # |D| reaches 32*127*128 with all codes at the ends of their ranges
    set_path(mmq, path)
    M, N, K = 16, 16, 256
    x = np.where(np.arange(M * K).reshape(M, K) % 3 == 0, -1.0, 1.0).astype(np.float32)
    x[::2] = -1.0
    w = np.zeros((N, K // 32, 34), dtype=np.uint8)
    w[:, :, 0:2] = np.array([0.5], dtype=np.float16).view(np.uint8)
    codes = np.where(np.arange(N * K).reshape(N, K // 32, 32) % 2 == 0, -128, 127).astype(np.int8)
    codes[::3] = -128
    w[:, :, 2:] = codes.view(np.uint8)
    w = w.reshape(N, -1)
    xq = mmq.mmq_quantize_q8_1(dev(x))
    dots = mmq.mmq_debug_block_dots_q8_0(xq, dev(w), M, N, K)
    xq_ref = oracle.quantize_q8_1(x)
    ref = oracle.block_dots("q8_0", xq_ref, w, M, N, K)
    assert np.abs(ref).max() == 32 * 127 * 128
    assert np.array_equal(dots.cpu().numpy(), ref)
    out = mmq.mmq_gemm_q8_0(xq, dev(w), M, N, K)
    r, nrm = oracle.gemm("q8_0", xq_ref, w, M, N, K)
    check_close(out.cpu().numpy(), r, nrm, "extreme codes")


# Every K-quant code and 6-bit scale at its maximum, activation blocks all +127 or all -127:
# the int8 stream's integer product sc_j * D_j then reaches 63 * 32 * 127 * 15 (Q4_K, the
# largest value it converts exactly) and Q5_K's dot 32 * 127 * 31.  (8, 300, 1024) is one
# full pass with a ragged last tile; (3, 5000, 512) a partly empty pass on a wide weight.
@pytest.mark.parametrize("M,N,K", [(8, 300, 1024), (3, 5000, 512)])
@pytest.mark.parametrize("fmt", ["q4_k", "q5_k"])
def test_k_quant_extreme_scales_int8_stream(mmq, fmt, M, N, K):
    set_path(mmq, "small")
    sb = 144 if fmt == "q4_k" else 176
    sign = np.where((np.arange(M)[:, None] + np.arange(K // 32)[None, :]) % 2 == 0, 1.0, -1.0)
    x = np.repeat(sign, 32, axis=1).astype(np.float32)
    w = synth.weights(fmt, 11, N, K).reshape(N, K // 256, sb).copy()
    w[:, :, 4:] = 0xFF  # scales and mins 63, every code 15 (Q4_K) / 31 (Q5_K)
    w = w.reshape(N, -1)
    xq = mmq.mmq_quantize_q8_1(dev(x))
    xq_ref = oracle.quantize_q8_1(x)
    dots = mmq.block_dots(fmt, xq, dev(w), M, N, K).cpu().numpy()
    ref_dots = oracle.block_dots(fmt, xq_ref, w, M, N, K)
    assert np.abs(ref_dots).min() == np.abs(ref_dots).max() == 32 * 127 * (15 if fmt == "q4_k" else 31)
    assert np.array_equal(dots, ref_dots)
    out = mmq.gemm(fmt, xq, dev(w), M, N, K)
    ref, norm = oracle.gemm(fmt, xq_ref, w, M, N, K)
    check_close(out.cpu().numpy(), ref, norm, f"{fmt} extreme scales {M}x{N}x{K}")
    assert mmq.mmq_get_device_error() == 0


@pytest.mark.parametrize("fmt", NO_TC)
def test_refused_by_converter_kernel_auto_takes_it(mmq, fmt):
    M, N, K = 600, 64, 512
    x = synth.activations(31, M, K, True)
    w = synth.weights(fmt, 32, N, K)
    xq = mmq.mmq_quantize_q8_1(dev(x))
    set_path(mmq, "tc")
    with pytest.raises(mmq.MMQError) as e:
        mmq.gemm(fmt, xq, dev(w), M, N, K)
    assert e.value.status == -9  # MMQ_ERR_ARG
    set_path(mmq, "auto")
    out = mmq.gemm(fmt, xq, dev(w), M, N, K)
    assert mmq.mmq_last_path() in (mmq.PATH_SMALL, mmq.PATH_EXPAND)
    ref, norm = oracle.gemm(fmt, oracle.quantize_q8_1(x), w, M, N, K)
    check_close(out.cpu().numpy(), ref, norm, f"{fmt} auto")
    assert mmq.mmq_get_device_error() == 0


def test_q5_k_extreme_codes_block_dots(mmq):
    M, N, K = 600, 64, 512
    x = synth.activations(31, M, K, True)
    xq = mmq.mmq_quantize_q8_1(dev(x))
    # Q5_K codes at the ends of 0..31 with the largest 6-bit scale: (q * sc) up to 31 * 63
    # and the min term at 63 * 63 on every sub-block
    w2 = synth.q5_k_weights(33, N, K).reshape(N, K // 256, 176).copy()
    w2[:, :, 4:16] = 0xFF
    w2[:, :, 16:] = np.where(np.arange(160) % 3 == 0, 0xFF, 0x00).astype(np.uint8)
    w2 = w2.reshape(N, -1)
    for path in ("expand", "small", "tc"):
        set_path(mmq, path)
        dots = mmq.mmq_debug_block_dots_q5_k(xq, dev(w2), M, N, K)
        assert np.array_equal(dots.cpu().numpy(), oracle.block_dots("q5_k", oracle.quantize_q8_1(x), w2, M, N, K))
    assert mmq.mmq_get_device_error() == 0


# ------------------------------------------------------------------ full sizes, sampled

def sample_entries(M, N, count, seed):
    rng = np.random.default_rng(seed)
    im = rng.integers(0, M, count)
    inn = rng.integers(0, N, count)
    edges_m = np.array([0, M - 1, min(M - 1, 127), min(M - 1, 128), M // 2])
    edges_n = np.array([0, N - 1, min(N - 1, 255), min(N - 1, 256), N // 2])
    em, en = np.meshgrid(edges_m, edges_n)
    return np.concatenate([im, em.ravel()]), np.concatenate([inn, en.ravel()])


@pytest.fixture(scope="module")
def full_operands():
    cache = {}

    def get(index, M=None):
        key = (index, M)
        if key not in cache:
            x, w, spec = synth.config_operands(index, M)
            cache[key] = (x, w, spec, oracle.quantize_q8_1(x))
        return cache[key]
    return get


@pytest.mark.parametrize("index,path", [(0, "auto"), (1, "auto"), (2, "auto"), (3, "auto"), (1, "tc"),
                                        (3, "tc")])
def test_config_sampled_parity(mmq, full_operands, index, path):
    set_path(mmq, path)
    x, w, spec, xq_ref = full_operands(index)
    M, N, K, fmt = spec["M"], spec["N"], spec["K"], spec["fmt"]
    xq = mmq.mmq_quantize_q8_1(dev(x))
    assert np.array_equal(xq.cpu().numpy(), xq_ref)
    out = torch.full((M, N), float("nan"), device="cuda")
    mmq.gemm(fmt, xq, dev(w), M, N, K, out=out)
    o = out.cpu().numpy()
    assert not np.isnan(o).any(), "output not fully written"
    im, inn = sample_entries(M, N, 3000, index)
    ref, norm = oracle.gemm_at(fmt, xq_ref, w, M, N, K, im, inn)
    check_close(o[im, inn], ref, norm, f"config {index} {path}")
    assert mmq.mmq_get_device_error() == 0
    if path == "auto":  # the converter kernel is never the automatic choice
        assert mmq.mmq_last_path() == (mmq.PATH_EXPAND if M >= 512 else mmq.PATH_SMALL)


@pytest.mark.parametrize("index", [1, 2, 3])
def test_config_linear_sampled_parity(mmq, full_operands, index):
    """The fused quantize + contraction at the full workload sizes (the bench's step)."""
    set_path(mmq, "auto")
    x, w, spec, xq_ref = full_operands(index)
    M, N, K, fmt = spec["M"], spec["N"], spec["K"], spec["fmt"]
    xq = torch.empty((M, K // 32 * 36), dtype=torch.uint8, device="cuda")
    out = torch.full((M, N), float("nan"), device="cuda")
    mmq.mmq_linear(dev(x), dev(w), fmt, N, xq=xq, out=out)
    assert mmq.mmq_last_path() == mmq.PATH_EXPAND
    assert np.array_equal(xq.cpu().numpy(), xq_ref)
    o = out.cpu().numpy()
    assert not np.isnan(o).any(), "output not fully written"
    im, inn = sample_entries(M, N, 3000, index + 10)
    ref, norm = oracle.gemm_at(fmt, xq_ref, w, M, N, K, im, inn)
    check_close(o[im, inn], ref, norm, f"config {index} linear")
    assert mmq.mmq_get_device_error() == 0


@pytest.mark.parametrize("M", synth.M_SWEEP)
def test_m_sweep_sampled_parity(mmq, M):
    set_path(mmq, "auto")
    N = K = 3584
    x = synth.activations(synth.substream(synth.BASE_SEED + 4, 7000 + M), M, K, True)
    w = synth.layer_weights(0, "q", N, K)
    xq = mmq.mmq_quantize_q8_1(dev(x))
    out = mmq.mmq_gemm_q4_k(xq, dev(w), M, N, K).cpu().numpy()
    xq_ref = oracle.quantize_q8_1(x)
    im, inn = sample_entries(M, N, 1500, M)
    ref, norm = oracle.gemm_at("q4_k", xq_ref, w, M, N, K, im, inn)
    check_close(out[im, inn], ref, norm, f"M sweep {M}")


def test_q6_k_extreme_codes_block_dots(mmq):
    # |D| up to 32 * 127 * 32 * 128 = 16646144 (just under 2^24): activation codes +-127,
    # weight codes 0 or 63 (q - 32 = -32 or 31), sub-scales -128 or 127
    M, N, K = 130, 136, 512
    xs = np.where(np.arange(M * K).reshape(M, K) % 5 == 0, -1.0, 1.0).astype(np.float32)
    xs[::2] = -1.0
    w = synth.q6_k_weights(41, N, K).reshape(N, K // 256, 210).copy()
    w[:, :, :128] = np.where(np.arange(128) % 3 == 0, 0x00, 0xFF).astype(np.uint8)   # low nibbles 0 or 15
    w[:, :, 128:192] = np.where(np.arange(64) % 3 == 0, 0x00, 0xFF).astype(np.uint8)  # top bits 0 or 3
    w[:, :, 192:208] = np.where(np.arange(16) % 2 == 0, 0x80, 0x7F).astype(np.uint8)  # -128, 127
    w[:4, :, 128:192] = 0x00  # rows 0..3: every code 0 or 15 -> q - 32 <= -17
    w[4:8, :, :192] = 0x00    # rows 4..7: every code 0 -> D = -32 * sc * sum(u)
    w[4:8, :, 192:208] = 0x80
    w = w.reshape(N, -1)
    xq = mmq.mmq_quantize_q8_1(dev(xs))
    xq_ref = oracle.quantize_q8_1(xs)
    ref = oracle.block_dots("q6_k", xq_ref, w, M, N, K)
    assert np.abs(ref).max() == 32 * 127 * 32 * 128
    for path in ("expand", "small"):
        set_path(mmq, path)
        dots = mmq.mmq_debug_block_dots_q6_k(xq, dev(w), M, N, K)
        assert np.array_equal(dots.cpu().numpy(), ref), path
        out = mmq.mmq_gemm_q6_k(xq, dev(w), M, N, K)
        r, nrm = oracle.gemm("q6_k", xq_ref, w, M, N, K)
        check_close(out.cpu().numpy(), r, nrm, f"q6_k extreme codes {path}")
    assert mmq.mmq_get_device_error() == 0


@pytest.mark.parametrize("M,N,K", [(1, 18944, 3584), (1, 3584, 18944), (4, 18944, 3584), (8, 3584, 18944),
                                   (512, 3584, 3584), (2048, 18944, 3584)])
@pytest.mark.parametrize("fmt", ["q5_k", "q6_k"])
def test_k_quant_full_size_sampled_parity(mmq, fmt, M, N, K):
    """Q5_K and Q6_K at the 7B-class projection sizes: the small-M streams and the expanded path."""
    set_path(mmq, "auto")
    x = synth.activations(synth.substream(synth.BASE_SEED + 5, M + N), M, K, True)
    w = synth.weights(fmt, synth.substream(synth.BASE_SEED + 6, N + K), N, K)
    xq_ref = oracle.quantize_q8_1(x)
    xq = torch.empty((M, K // 32 * 36), dtype=torch.uint8, device="cuda")
    out = torch.full((M, N), float("nan"), device="cuda")
    mmq.mmq_linear(dev(x), dev(w), fmt, N, xq=xq, out=out)
    assert mmq.mmq_last_path() == (mmq.PATH_EXPAND if M >= 512 else mmq.PATH_SMALL)
    assert np.array_equal(xq.cpu().numpy(), xq_ref)
    o = out.cpu().numpy()
    assert not np.isnan(o).any(), "output not fully written"
    im, inn = sample_entries(M, N, 1500, M + 5)
    ref, norm = oracle.gemm_at(fmt, xq_ref, w, M, N, K, im, inn)
    check_close(o[im, inn], ref, norm, f"{fmt} {M}x{N}x{K}")
    assert mmq.mmq_get_device_error() == 0


# ------------------------------------------------------------------ protocol on the device

def test_refused_call_leaves_output_untouched(mmq):
    M, N, K = 8, 64, 256
    x = synth.activations(3, M, K, True)
    w = synth.q8_0_weights(4, N, K)
    xq = mmq.mmq_quantize_q8_1(dev(x))
    out = torch.full((M * N + 4,), float("nan"), device="cuda")
    wd = dev(w)
    lib = mmq.lib()
    import ctypes
    st = lib.mmq_gemm_q8_0(ctypes.c_void_p(xq.data_ptr()), ctypes.c_void_p(wd.data_ptr()), M, N, K,
                           ctypes.c_void_p(out.data_ptr() + 4), None)
    assert st == -4
    st = lib.mmq_gemm_q8_0(ctypes.c_void_p(xq.data_ptr()), ctypes.c_void_p(wd.data_ptr()), M, N, K + 16,
                           ctypes.c_void_p(out.data_ptr()), None)
    assert st == -2
    torch.cuda.synchronize()
    assert torch.isnan(out).all()
    with pytest.raises(mmq.MMQError):
        mmq.mmq_gemm_q4_k(xq, wd, M, N, K + 32)


def test_streams_and_device_error_word(mmq):
    s = torch.cuda.Stream()
    M, N, K = 33, 65, 512
    x = synth.activations(9, M, K, True)
    w = synth.q4_k_weights(10, N, K)
    with torch.cuda.stream(s):
        xd, wd = dev(x), dev(w)
        xq = mmq.mmq_quantize_q8_1(xd, stream=s)
        out = mmq.mmq_gemm_q4_k(xq, wd, M, N, K, stream=s)
    assert mmq.mmq_get_device_error(s) == 0
    ref, norm = oracle.gemm("q4_k", oracle.quantize_q8_1(x), w, M, N, K)
    check_close(out.cpu().numpy(), ref, norm, "side stream")


def test_graph_capture_and_replay_with_scratch(mmq):
    # under capture the expanded path's scratch becomes graph-owned memory; replaying the
    # graph twice gives the eager result, and the profiler's event nodes time the replay
    set_path(mmq, "expand")
    M, N, K = 192, 160, 512
    x = synth.activations(31, M, K, True)
    w = synth.q8_0_weights(32, N, K)
    xd, wd = dev(x), dev(w)
    xq = mmq.mmq_quantize_q8_1(xd)
    eager = mmq.mmq_gemm_q8_0(xq, wd, M, N, K)
    assert mmq.mmq_last_path() == mmq.PATH_EXPAND
    torch.cuda.synchronize()
    mmq.mmq_profile_read(reset=True)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    out = torch.full((M, N), float("nan"), device="cuda")
    prev = mmq.mmq_profile_enable(True)
    try:
        with torch.cuda.graph(g, stream=s):
            mmq.mmq_gemm_q8_0(xq, wd, M, N, K, out=out, stream=s)
        assert mmq.mmq_last_path() == mmq.PATH_EXPAND
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        prof = mmq.mmq_profile_read(reset=True)
    finally:
        mmq.mmq_profile_enable(prev)
    assert set(prof) == {"k_expand", "k_mmq_tcx"}, prof
    assert all(n == 1 and ms > 0 for n, ms in prof.values()), prof
    ref, norm = oracle.gemm("q8_0", oracle.quantize_q8_1(x), w, M, N, K)
    check_close(out.cpu().numpy(), ref, norm, "captured")
    check_close(eager.cpu().numpy(), ref, norm, "eager")
    assert mmq.mmq_get_device_error() == 0


def test_profile_counts_every_launch(mmq):
    set_path(mmq, "expand")
    torch.cuda.synchronize()
    mmq.mmq_profile_read(reset=True)
    prev = mmq.mmq_profile_enable(True)
    try:
        M, N, K = 100, 130, 512
        x = synth.activations(61, M, K, True)
        w = synth.q4_k_weights(62, N, K)
        xq = mmq.mmq_quantize_q8_1(dev(x))
        mmq.mmq_gemm_q4_k(xq, dev(w), M, N, K)          # expanded path: two kernels
        set_path(mmq, "auto")
        mmq.mmq_gemm_q4_k(xq[:4], dev(w), 4, N, K)      # M <= 8: one small-M kernel
        prof = mmq.mmq_profile_read(reset=True)
    finally:
        mmq.mmq_profile_enable(prev)
    assert prof["k_quantize_q8_1"][0] == 1
    assert prof["k_expand"][0] == prof["k_mmq_tcx"][0] == 1
    small = {k: n for k, (n, _) in prof.items()
             if k not in ("k_quantize_q8_1", "k_expand", "k_mmq_tcx")}
    assert sum(small.values()) == 1, prof  # one small-M kernel for the M = 4 call
    assert mmq.mmq_profile_read() == {}


def test_expand_path_concurrent_streams(mmq):
    # two streams in flight at once, each with its own stream-ordered scratch
    set_path(mmq, "expand")
    M, N, K = 256, 384, 1024
    ops = []
    for i in range(2):
        x = synth.activations(40 + i, M, K, True)
        w = synth.q4_k_weights(50 + i, N, K)
        ops.append((x, w))
    streams = [torch.cuda.Stream() for _ in ops]
    outs = []
    for (x, w), st in zip(ops, streams):
        with torch.cuda.stream(st):
            xq = mmq.mmq_quantize_q8_1(dev(x), stream=st)
            outs.append(mmq.mmq_gemm_q4_k(xq, dev(w), M, N, K, stream=st))
    torch.cuda.synchronize()
    for (x, w), o in zip(ops, outs):
        ref, norm = oracle.gemm("q4_k", oracle.quantize_q8_1(x), w, M, N, K)
        check_close(o.cpu().numpy(), ref, norm, "concurrent streams")
    assert mmq.mmq_get_device_error() == 0


# ------------------------------------------------------------------ expert-grouped contraction

def grouped_reference(fmt, xq_ref, ids, w, E, N, K):
    """out[r] = row r contracted with expert ids[r] (the oracle per expert); zeros for ids
    outside [0, E).  Returns (ref, norm)."""
    R = len(ids)
    ref = np.zeros((R, N))
    norm = np.zeros((R, N))
    rows_w = w.reshape(E, N, -1)
    for e in range(E):
        rows = np.nonzero(ids == e)[0]
        if len(rows) == 0:
            continue
        r_e, n_e = oracle.gemm(fmt, np.ascontiguousarray(xq_ref[rows]), np.ascontiguousarray(rows_w[e]), len(rows), N, K)
        ref[rows] = r_e
        norm[rows] = n_e
    return ref, norm


GROUPED_CASES = [  # (R, E, N, K, routing)
    (300, 5, 200, 512, "uniform"),
    (1000, 16, 130, 256, "uniform"),
    (64, 128, 64, 256, "uniform"),      # more experts than rows: most experts empty
    (700, 8, 96, 512, "hot"),           # every row to one expert: several full tiles
    (257, 6, 136, 256, "invalid"),      # some ids out of range: zero rows
    (2500, 40, 64, 256, "uniform"),     # several grouping CTAs (1024 rows each)
    (300, 9000, 32, 256, "invalid"),    # more experts than the shared-memory counters hold
    (70000, 24, 32, 256, "invalid"),    # more ids than the planning CTA counts itself
]


@pytest.mark.parametrize("path", ["expand", "small", "tc"])
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("case", range(len(GROUPED_CASES)))
def test_grouped_parity(mmq, fmt, case, path):
    """The three contractions over the device-built grouping, each forced: the expanded
    path (128-row tiles), the grouped dp4a weight stream (tiles of 2 or 4 rows; the
    automatic choice where experts hold few rows) and the converter kernel (MMQ_PATH_TC;
    not Q6_K, refused below)."""
    if fmt in NO_TC and path == "tc":
        pytest.skip("the converter kernel takes Q8_0, Q4_K and Q5_K")
    R, E, N, K, routing = GROUPED_CASES[case]
    rng = np.random.default_rng(100 + case)
    if routing == "hot":
        ids = np.full(R, 3 % E, dtype=np.int32)
    else:
        ids = rng.integers(0, E, R).astype(np.int32)
    if routing == "invalid":
        ids[::7] = -1
        ids[3::11] = E
    x = synth.activations(200 + case, R, K, True)
    w = synth.weights(fmt, 300 + case, E * N, K)
    xq = mmq.mmq_quantize_q8_1(dev(x))
    out = torch.full((R, N), float("nan"), device="cuda")
    set_path(mmq, path)
    try:
        mmq.mmq_gemm_grouped(fmt, xq, dev(ids), dev(w), E, N, K, out=out)
        assert mmq.mmq_last_path() == PATH_IDS[path]
        again = mmq.mmq_gemm_grouped(fmt, xq, dev(ids), dev(w), E, N, K)
    finally:
        set_path(mmq, "auto")
    assert mmq.mmq_get_device_error() == 0
    assert torch.equal(out, again), "grouped result depends on the run"
    ref, norm = grouped_reference(fmt, oracle.quantize_q8_1(x), ids, w, E, N, K)
    check_close(out.cpu().numpy(), ref, norm, f"grouped {fmt} {GROUPED_CASES[case]}")


@pytest.mark.parametrize("path", ["expand", "small", "tc"])
def test_grouped_graph_capture(mmq, path):
    R, E, N, K = 500, 12, 160, 512
    rng = np.random.default_rng(7)
    ids = rng.integers(0, E, R).astype(np.int32)
    x = synth.activations(401, R, K, True)
    w = synth.weights("q4_k", 402, E * N, K)
    xq = mmq.mmq_quantize_q8_1(dev(x))
    idd, wd = dev(ids), dev(w)
    out = torch.full((R, N), float("nan"), device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    set_path(mmq, path)
    try:
        with torch.cuda.graph(g, stream=s):
            mmq.mmq_gemm_grouped("q4_k", xq, idd, wd, E, N, K, out=out, stream=s)
    finally:
        set_path(mmq, "auto")
    g.replay()
    torch.cuda.synchronize()
    ref, norm = grouped_reference("q4_k", oracle.quantize_q8_1(x), ids, w, E, N, K)
    check_close(out.cpu().numpy(), ref, norm, "captured grouped")
    assert mmq.mmq_get_device_error() == 0


# MMQ_PATH_AUTO takes the grouped weight stream up to 10 rows per expert on average for
# Q4_K (Q8_0 14, Q5_K 9, Q6_K 7; every expert's weights read once per tile of 2 or 4 rows)
# and the expanded path above (every expert's weights expanded once, 128-row tiles)
@pytest.mark.parametrize("R,E,want", [(128, 128, "small"), (1280, 128, "small"), (1281, 128, "expand"),
                                      (4096, 64, "expand")])
def test_grouped_auto_follows_the_experts_fill(mmq, R, E, want):
    N, K = 64, 512
    rng = np.random.default_rng(R + E)
    ids = rng.integers(0, E, R).astype(np.int32)
    x = synth.activations(R + 11, R, K, True)
    w = synth.weights("q4_k", E + 12, E * N, K)
    xq = mmq.mmq_quantize_q8_1(dev(x))
    set_path(mmq, "auto")
    out = mmq.mmq_gemm_grouped("q4_k", xq, dev(ids), dev(w), E, N, K)
    assert mmq.mmq_last_path() == PATH_IDS[want]
    ref, norm = grouped_reference("q4_k", oracle.quantize_q8_1(x), ids, w, E, N, K)
    check_close(out.cpu().numpy(), ref, norm, f"grouped auto R={R} E={E}")
    assert mmq.mmq_get_device_error() == 0


def test_grouped_refusals(mmq):
    xq = torch.zeros((4, 8 * 36), dtype=torch.uint8, device="cuda")
    ids = torch.zeros(4, dtype=torch.int32, device="cuda")
    w = torch.zeros((2 * 8, 144), dtype=torch.uint8, device="cuda")
    with pytest.raises(mmq.MMQError) as e:  # K % 256
        mmq.mmq_gemm_grouped("q4_k", xq, ids, w, 2, 8, 128)
    assert e.value.status == -2
    with pytest.raises(mmq.MMQError) as e:  # E < 1
        mmq.mmq_gemm_grouped("q4_k", xq, ids, w, 0, 8, 256)
    assert e.value.status == -1
    out = torch.full((4, 8), float("nan"), device="cuda")
    wq6 = torch.zeros((2 * 8, 210), dtype=torch.uint8, device="cuda")
    set_path(mmq, "tc")
    try:
        with pytest.raises(mmq.MMQError) as e:  # Q6_K on the converter kernel
            mmq.mmq_gemm_grouped("q6_k", xq, ids, wq6, 2, 8, 256, out=out)
        assert e.value.status == -9
    finally:
        set_path(mmq, "auto")
    assert torch.isnan(out).all(), "a refused call writes nothing"
