"""Pins for the CPU oracle: each test checks it against something other than itself.

- binary16 conversion against numpy's IEEE float16 (an independent library);
- hand-worked examples whose values follow from the method's definitions
  (tests/golden/hand_examples.txt, derivations inline there);
- the quantizer against exact rational arithmetic with explicit f32 rounding steps;
- invariants of q8_1 (max |q| = 127, the half-step error bound, s = f16(d * S));
- Q4_K scale decoding against bytes built by an independent packer (tests/q4k_pack.py);
- block dots against numpy integer brute force;
- both contractions against dequantize-then-fp64-matmul (a different summation path:
  over elements instead of over scaled block dots);
- closed-form special cases (all-ones weights, zero sub-scales).
Methods: quantize and the Q8_0 contraction follow "When the Product Won't Collapse"
(sec. "The obstruction") and "13 . r7-r8 raw-byte MMQ kernel" (sec. 3.2); the Q4_K
contraction follows "When Does a Kernel Win Surface?" (sec. "Kept levers: Vulkan").
"""
import math
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from conftest import as_floats, as_ints
from q4k_pack import pack_nibbles, pack_scales, q5_k_super_block, q6_k_super_block, super_block

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ------------------------------------------------------------------ helpers

def fl32(v: Fraction) -> Fraction:
    """Round an exact rational to the nearest binary32 (ties to even); normal range only."""
    if v == 0:
        return Fraction(0)
    s = -1 if v < 0 else 1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)
    ulp = Fraction(2) ** (e - 23)
    q = a / ulp
    n = math.floor(q)
    r = q - n
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return s * n * ulp


def rne_int(v: Fraction) -> int:
    n = math.floor(v)
    r = v - n
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return n


def np_f16_bits(v) -> np.ndarray:
    return np.asarray(v, dtype=np.float32).astype(np.float16).view(np.uint16)


def split_q8_1(xq: np.ndarray):
    """(d f64 [M,nb], s f64 [M,nb], q int [M,nb,32]) decoded with numpy's float16."""
    M = xq.shape[0]
    b = xq.reshape(M, -1, 36)
    d = b[:, :, 0:2].copy().view(np.float16)[:, :, 0].astype(np.float64)
    s = b[:, :, 2:4].copy().view(np.float16)[:, :, 0].astype(np.float64)
    q = b[:, :, 4:].view(np.int8).astype(np.int64)
    return d, s, q


def split_q8_0(wq: np.ndarray):
    N = wq.shape[0]
    b = wq.reshape(N, -1, 34)
    d = b[:, :, 0:2].copy().view(np.float16)[:, :, 0].astype(np.float64)
    q = b[:, :, 2:].view(np.int8).astype(np.int64)
    return d, q


# ------------------------------------------------------------------ binary16

def test_f16_decode_all_patterns_match_numpy():
    pats = np.arange(65536, dtype=np.uint16)
    ref = pats.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_f64(int(h)) for h in pats])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_f16_encode_matches_numpy_rounding():
    rng = np.random.default_rng(7)
    # every f16 value, every midpoint between neighbours (ties) and nudges around them
    allh = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (allh[:-1] + allh[1:]) / 2
    vals = np.concatenate([allh[::7], mids[::5], np.nextafter(mids[::11], 0), np.nextafter(mids[::13], 1e9),
                           np.exp(rng.uniform(np.log(1e-9), np.log(7e4), 4000)), [65504.0, 65519.0, 65520.0, 1e6]])
    vals = np.concatenate([vals, -vals]).astype(np.float32)  # exact f32 values
    got = np.array([oracle.f64_to_f16(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, np_f16_bits(vals))


# ------------------------------------------------------------------ hand examples

def _quant_one(x):
    xq = oracle.quantize_q8_1(np.asarray(x, dtype=np.float32)[None, :])
    d_bits = int(xq[0, 0]) | int(xq[0, 1]) << 8
    s_bits = int(xq[0, 2]) | int(xq[0, 3]) << 8
    return xq, d_bits, s_bits, xq[0, 4:36].view(np.int8).astype(int).tolist()


def test_hand_example_ties(golden_hand):
    g = golden_hand
    xq, d, s, q = _quant_one(as_floats(g["e1_x"]))
    assert q == as_ints(g["e1_q"])
    assert d == as_ints(g["e1_d_f16"])[0] and s == as_ints(g["e1_s_f16"])[0]
    # Q8_0 contraction against all-ones codes, d = 0.5
    wblk = np.zeros(34, dtype=np.uint8)
    wblk[0:2] = np.array(as_ints(g["e1_q8_0_wd_f16"]), dtype=np.uint16).view(np.uint8)
    wblk[2:] = 1
    dots = oracle.block_dots("q8_0", xq, wblk[None, :], 1, 1, 32)
    assert int(dots[0, 0, 0]) == as_ints(g["e1_q8_0_dot"])[0]
    out, norm = oracle.gemm("q8_0", xq, wblk[None, :], 1, 1, 32)
    assert out[0, 0] == as_floats(g["e1_q8_0_out"])[0]
    assert norm[0, 0] == abs(out[0, 0])


def test_hand_example_nontrivial_scale(golden_hand):
    g = golden_hand
    _, d, s, q = _quant_one(as_floats(g["e2_x"]))
    assert q == as_ints(g["e2_q"])
    assert d == as_ints(g["e2_d_f16"])[0] and s == as_ints(g["e2_s_f16"])[0]


def test_hand_example_true_division(golden_hand):
    g = golden_hand
    _, d, s, q = _quant_one(as_floats(g["e5_x"]))
    assert q == as_ints(g["e5_q"])
    assert d == as_ints(g["e5_d_f16"])[0] and s == as_ints(g["e5_s_f16"])[0]


def test_hand_example_q4_k_super_block(golden_hand):
    g = golden_hand
    xq1, _, _, _ = _quant_one(as_floats(g["e1_x"]))
    xq = np.tile(xq1, (1, 8))  # eight identical blocks, K = 256
    sc, m = as_ints(g["e3_sc"]), as_ints(g["e3_m"])
    p = np.array(as_ints(g["e3_scale_bytes"]), dtype=np.uint8)
    assert np.array_equal(pack_scales(sc, m), p)
    for j in range(8):
        assert oracle.q4_k_scale_min(p, j) == (sc[j], m[j])
    blk = super_block(as_ints(g["e3_d_f16"])[0], as_ints(g["e3_dmin_f16"])[0], sc, m,
                      [as_ints(g["e3_nibble"])[0]] * 256)
    dots = oracle.block_dots("q4_k", xq, blk[None, :], 1, 1, 256)
    assert (dots == as_ints(g["e3_dot"])[0]).all()
    out, norm = oracle.gemm("q4_k", xq, blk[None, :], 1, 1, 256)
    assert out[0, 0] == as_floats(g["e3_out"])[0]
    assert norm[0, 0] == as_floats(g["e3_norm"])[0]


def test_hand_example_q5_k_super_block(golden_hand):
    g = golden_hand
    xq1, _, _, _ = _quant_one(as_floats(g["e1_x"]))
    xq = np.tile(xq1, (1, 8))
    sc, m = as_ints(g["e3_sc"]), as_ints(g["e3_m"])
    codes = np.repeat(as_ints(g["e6_codes"]), 32)
    blk = q5_k_super_block(as_ints(g["e3_d_f16"])[0], as_ints(g["e3_dmin_f16"])[0], sc, m, codes)
    assert (blk[16:48] == as_ints(g["e6_qh_byte"])[0]).all() and (blk[48:] == as_ints(g["e6_qs_byte"])[0]).all()
    assert np.array_equal(blk[4:16], np.array(as_ints(g["e3_scale_bytes"]), dtype=np.uint8))
    dots = oracle.block_dots("q5_k", xq, blk[None, :], 1, 1, 256)
    assert dots.reshape(8).tolist() == as_ints(g["e6_dots"])
    out, norm = oracle.gemm("q5_k", xq, blk[None, :], 1, 1, 256)
    assert out[0, 0] == as_floats(g["e6_out"])[0]
    assert norm[0, 0] == as_floats(g["e6_norm"])[0]


def test_hand_example_q6_k_super_block(golden_hand):
    g = golden_hand
    xq1, _, _, _ = _quant_one(as_floats(g["e2_x"]))
    xq = np.tile(xq1, (1, 8))
    codes = np.repeat(as_ints(g["e7_codes"]), 16)
    blk = q6_k_super_block(as_ints(g["e7_d_f16"])[0], as_ints(g["e7_sc"]), codes)
    assert blk[as_ints(g["e7_ql_at"])].tolist() == as_ints(g["e7_ql"])
    assert blk[128 + np.array(as_ints(g["e7_qh_at"]))].tolist() == as_ints(g["e7_qh"])
    dots = oracle.block_dots("q6_k", xq, blk[None, :], 1, 1, 256)
    assert dots.reshape(8).tolist() == as_ints(g["e7_dots"])
    out, norm = oracle.gemm("q6_k", xq, blk[None, :], 1, 1, 256)
    assert out[0, 0] == as_floats(g["e7_out"])[0]
    assert norm[0, 0] == sum(abs(v) for v in as_ints(g["e7_dots"])) * 129 / 2048


def test_hand_example_scale_top_bits(golden_hand):
    g = golden_hand
    p = np.array(as_ints(g["e4_scale_bytes"]), dtype=np.uint8)
    sc, m = as_ints(g["e4_sc"]), as_ints(g["e4_m"])
    assert np.array_equal(pack_scales(sc, m), p)
    assert [oracle.q4_k_scale_min(p, j) for j in range(8)] == list(zip(sc, m))


def test_format_facts(golden_facts):
    f = {k: v[0] for k, v in golden_facts.items()}
    assert int(f["block_elems"]) == oracle.QK == synth.QK
    assert int(f["q4_k_super_block_bytes"]) == oracle.Q4_K_BYTES == synth.Q4_K_BYTES
    assert int(f["q4_k_super_block_elems"]) == oracle.QK_K
    assert int(f["q4_k_blocks_per_super_block"]) * oracle.QK == oracle.QK_K
    assert int(f["act_codes_offset"]) == 4
    m, n, k = int(f["ladder_m"]), int(f["ladder_n"]), int(f["ladder_k"])
    assert round(2 * m * n * k / 1e9, 1) == float(f["ladder_gflop"])


# ------------------------------------------------------------------ quantizer

def _tricky_rows(rng):
    rows = []
    rows.append(np.zeros(32))                                     # all zero
    rows.append(np.full(32, 3.25))                                # all equal positive
    rows.append(np.where(np.arange(32) == 5, -2.0, 0.0))          # one nonzero
    rows.append((np.arange(32) - 16) * 0.5)                       # half-integer grid
    rows.append(np.arange(32) * 127.0 / 31.0)                     # ramp
    rows.append(rng.normal(size=32) * 1e-3)                       # f16-subnormal d
    rows.append(rng.normal(size=32) * 1e-30)                      # tiny values
    rows.append(rng.normal(size=32) * 3e3)                        # large values
    t = rng.integers(-127, 128, size=32).astype(np.float64)       # exact integer codes
    t[0] = 127.0
    rows.append(t * 0.75)
    return np.stack(rows).astype(np.float32)


def test_quantize_matches_exact_rational_definition():
    rng = np.random.default_rng(11)
    x = np.concatenate([_tricky_rows(rng), synth.activations(123, 6, 32, True)]).astype(np.float32)
    xq = oracle.quantize_q8_1(x)
    for r in range(x.shape[0]):
        blk = xq[r]
        vals = [Fraction(float(v)) for v in x[r]]
        amax = max(abs(v) for v in vals)
        d = fl32(amax / 127)
        if d == 0:
            q = [0] * 32
        else:
            q = [max(-127, min(127, rne_int(fl32(v / d)))) for v in vals]
        S = sum(q)
        assert blk[4:36].view(np.int8).astype(int).tolist() == q, r
        assert int(blk[0]) | int(blk[1]) << 8 == int(np_f16_bits(float(d))), r
        assert int(blk[2]) | int(blk[3]) << 8 == int(np_f16_bits(float(fl32(d * S)))), r


@pytest.mark.parametrize("outliers", [False, True])
def test_quantize_invariants(outliers):
    x = synth.activations(99 + outliers, 64, 1024, outliers)
    xq = oracle.quantize_q8_1(x)
    M, nb = 64, 1024 // 32
    xb = x.reshape(M, nb, 32).astype(np.float64)
    q = xq.reshape(M, nb, 36)[:, :, 4:].view(np.int8).astype(np.int64)
    amax = np.abs(xb).max(axis=2)
    d = (amax.astype(np.float32) / np.float32(127)).astype(np.float64)   # f32 division
    nz = amax > 0
    assert (np.abs(q).max(axis=2)[nz] == 127).all()
    assert (np.abs(q) <= 127).all()
    err = np.abs(xb - d[:, :, None] * q)
    assert (err <= d[:, :, None] / 2 * (1 + 2.0 ** -22)).all()
    # s is f16(f32(d) * S) and d is f16(f32 d)
    S = q.sum(axis=2)
    dbits = xq.reshape(M, nb, 36)[:, :, 0:2].copy().view(np.uint16)[:, :, 0]
    sbits = xq.reshape(M, nb, 36)[:, :, 2:4].copy().view(np.uint16)[:, :, 0]
    assert np.array_equal(dbits, np_f16_bits(d.astype(np.float32)))
    assert np.array_equal(sbits, np_f16_bits(d.astype(np.float32) * S.astype(np.float32)))


def test_quantize_amax_order_free():
    # amax is exact under any association; permuting a block permutes its codes
    x = synth.activations(5, 8, 32, True)
    perm = np.random.default_rng(3).permutation(32)
    a, b = oracle.quantize_q8_1(x), oracle.quantize_q8_1(x[:, perm])
    assert np.array_equal(a[:, :4], b[:, :4])
    assert np.array_equal(a[:, 4:][:, perm], b[:, 4:])


# ------------------------------------------------------------------ Q4_K scales

def test_q4_k_scale_round_trip_every_slot_value():
    rng = np.random.default_rng(17)
    for j in range(8):
        for v in range(64):
            sc = rng.integers(0, 64, 8)
            m = rng.integers(0, 64, 8)
            sc[j] = v
            m[(j + 3) % 8] = 63 - v
            p = pack_scales(sc, m)
            assert [oracle.q4_k_scale_min(p, i) for i in range(8)] == list(zip(sc.tolist(), m.tolist()))


def test_q4_k_scale_round_trip_random():
    rng = np.random.default_rng(19)
    for _ in range(3000):
        sc = rng.integers(0, 64, 8)
        m = rng.integers(0, 64, 8)
        p = pack_scales(sc, m)
        assert [oracle.q4_k_scale_min(p, i) for i in range(8)] == list(zip(sc.tolist(), m.tolist()))


def test_q4_k_scale_decode_is_a_bijection_of_the_96_bits():
    # flipping any single bit of the 12 bytes changes exactly one of the 16 decoded fields
    rng = np.random.default_rng(23)
    p = rng.integers(0, 256, 12).astype(np.uint8)
    base = [oracle.q4_k_scale_min(p, j) for j in range(8)]
    for byte in range(12):
        for bit in range(8):
            p2 = p.copy()
            p2[byte] ^= 1 << bit
            now = [oracle.q4_k_scale_min(p2, j) for j in range(8)]
            changed = sum((a[0] != b[0]) + (a[1] != b[1]) for a, b in zip(base, now))
            assert changed == 1


# ------------------------------------------------------------------ block dots

def test_block_dots_q8_0_brute_force():
    x = synth.activations(1, 5, 96, True)
    xq = oracle.quantize_q8_1(x)
    wq = synth.q8_0_weights(2, 7, 96)
    dots = oracle.block_dots("q8_0", xq, wq, 5, 7, 96)
    _, _, qa = split_q8_1(xq)
    _, qw = split_q8_0(wq)
    ref = np.einsum("mbk,nbk->mnb", qa, qw)
    assert np.array_equal(dots, ref)


def test_block_dots_q4_k_brute_force():
    x = synth.activations(3, 4, 512, True)
    xq = oracle.quantize_q8_1(x)
    wq = synth.q4_k_weights(4, 6, 512)
    dots = oracle.block_dots("q4_k", xq, wq, 4, 6, 512)
    _, _, qa = split_q8_1(xq)
    nib = wq.reshape(6, 2, 144)[:, :, 16:].reshape(6, 2, 4, 32)
    codes = np.stack([nib & 15, nib >> 4], axis=3).reshape(6, 2, 256).astype(np.int64)
    qw = codes.reshape(6, 16, 32)
    ref = np.einsum("mbk,nbk->mnb", qa, qw)
    assert np.array_equal(dots, ref)
    assert np.abs(dots).max() < 2 ** 31


def test_block_dot_extremes_fit_int32():
    x = np.full((1, 32), -5.0, dtype=np.float32)
    xq = oracle.quantize_q8_1(x)
    w = np.zeros((1, 34), dtype=np.uint8)
    w[0, 2:] = np.uint8(0x80)  # code -128
    assert int(oracle.block_dots("q8_0", xq, w, 1, 1, 32)[0, 0, 0]) == 32 * 127 * 128


# ------------------------------------------------------------------ contractions

@pytest.mark.parametrize("M,N,K", [(1, 1, 32), (2, 3, 64), (3, 2, 64), (7, 5, 512)])
def test_q8_0_equals_dequantized_fp64_matmul(M, N, K):
    x = synth.activations(10 + M, M, K, True)
    xq = oracle.quantize_q8_1(x)
    wq = synth.q8_0_weights(20 + N, N, K)
    out, norm = oracle.gemm("q8_0", xq, wq, M, N, K)
    da, _, qa = split_q8_1(xq)
    dw, qw = split_q8_0(wq)
    xh = (da[:, :, None] * qa).reshape(M, K)
    wh = (dw[:, :, None] * qw).reshape(N, K)
    ref = xh @ wh.T
    assert np.all(np.abs(out - ref) <= 1e-12 * np.abs(xh) @ np.abs(wh).T + 1e-300)
    assert np.all(norm >= np.abs(out) * (1 - 1e-15))


def _random_q4_k(rng, N, K):
    """Weights built from chosen fields, plus the fields themselves."""
    nsb = K // 256
    d = rng.uniform(1e-4, 2e-3, (N, nsb)).astype(np.float16)
    dmin = rng.uniform(1e-4, 2e-3, (N, nsb)).astype(np.float16)
    sc = rng.integers(0, 64, (N, nsb, 8))
    mn = rng.integers(0, 64, (N, nsb, 8))
    codes = rng.integers(0, 16, (N, nsb, 256))
    w = np.stack([super_block(int(d[n, s].view(np.uint16)), int(dmin[n, s].view(np.uint16)),
                              sc[n, s], mn[n, s], codes[n, s])
                  for n in range(N) for s in range(nsb)]).reshape(N, nsb * 144)
    return w, d.astype(np.float64), dmin.astype(np.float64), sc, mn, codes


@pytest.mark.parametrize("M,N,K", [(1, 1, 256), (2, 3, 256), (3, 2, 512), (5, 4, 768)])
def test_q4_k_equals_dequantized_fp64_matmul(M, N, K):
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    x = synth.activations(30 + M, M, K, True)
    xq = oracle.quantize_q8_1(x)
    w, d, dmin, sc, mn, codes = _random_q4_k(rng, N, K)
    out, norm = oracle.gemm("q4_k", xq, w, M, N, K)
    nsb = K // 256
    # dequantized weights from the chosen fields: w = d*sc*q - dmin*m
    wsub = (d[:, :, None] * sc)[:, :, :, None] * codes.reshape(N, nsb, 8, 32) \
        - (dmin[:, :, None] * mn)[:, :, :, None]
    wh = wsub.reshape(N, K)
    da, sa, qa = split_q8_1(xq)
    xh = (da[:, :, None] * qa).reshape(M, K)
    ref = xh @ wh.T
    # the contraction uses the stored block sum s where dequantization gives d*S
    S = qa.sum(axis=2)
    mterm = (dmin[:, :, None] * mn).reshape(N, nsb * 8)            # dmin*m per (n, block)
    ref += (da * S - sa) @ mterm.T
    scale = np.abs(xh) @ np.abs(wh).T + np.abs(sa) @ np.abs(mterm).T
    assert np.all(np.abs(out - ref) <= 1e-12 * scale)
    assert np.all(norm >= np.abs(out) * (1 - 1e-15))


def _random_q5_k(rng, N, K):
    nsb = K // 256
    d = rng.uniform(1e-4, 2e-3, (N, nsb)).astype(np.float16)
    dmin = rng.uniform(1e-4, 2e-3, (N, nsb)).astype(np.float16)
    sc = rng.integers(0, 64, (N, nsb, 8))
    mn = rng.integers(0, 64, (N, nsb, 8))
    codes = rng.integers(0, 32, (N, nsb, 256))
    w = np.stack([q5_k_super_block(int(d[n, s].view(np.uint16)), int(dmin[n, s].view(np.uint16)),
                                   sc[n, s], mn[n, s], codes[n, s])
                  for n in range(N) for s in range(nsb)]).reshape(N, nsb * 176)
    return w, d.astype(np.float64), dmin.astype(np.float64), sc, mn, codes


def test_block_dots_q5_k_brute_force_on_packed_codes():
    # every code of every element position: the fifth bit and the nibble of each element
    # land where the decoder looks for them
    rng = np.random.default_rng(51)
    M, N, K = 3, 5, 512
    x = synth.activations(51, M, K, True)
    xq = oracle.quantize_q8_1(x)
    w, d, dmin, sc, mn, codes = _random_q5_k(rng, N, K)
    dots = oracle.block_dots("q5_k", xq, w, M, N, K)
    _, _, qa = split_q8_1(xq)
    ref = np.einsum("mbk,nbk->mnb", qa, codes.reshape(N, K // 32, 32))
    assert np.array_equal(dots, ref)


@pytest.mark.parametrize("M,N,K", [(1, 1, 256), (2, 3, 512), (4, 2, 768)])
def test_q5_k_equals_dequantized_fp64_matmul(M, N, K):
    rng = np.random.default_rng(M * 100 + N * 10 + K + 5)
    x = synth.activations(60 + M, M, K, True)
    xq = oracle.quantize_q8_1(x)
    w, d, dmin, sc, mn, codes = _random_q5_k(rng, N, K)
    out, norm = oracle.gemm("q5_k", xq, w, M, N, K)
    nsb = K // 256
    wsub = (d[:, :, None] * sc)[:, :, :, None] * codes.reshape(N, nsb, 8, 32) \
        - (dmin[:, :, None] * mn)[:, :, :, None]
    wh = wsub.reshape(N, K)
    da, sa, qa = split_q8_1(xq)
    xh = (da[:, :, None] * qa).reshape(M, K)
    ref = xh @ wh.T
    S = qa.sum(axis=2)
    mterm = (dmin[:, :, None] * mn).reshape(N, nsb * 8)
    ref += (da * S - sa) @ mterm.T
    scale = np.abs(xh) @ np.abs(wh).T + np.abs(sa) @ np.abs(mterm).T
    assert np.all(np.abs(out - ref) <= 1e-12 * scale)
    assert np.all(norm >= np.abs(out) * (1 - 1e-15))


def test_q5_k_with_no_fifth_bits_equals_q4_k():
    # a Q5_K block whose high-bit bytes are zero is the Q4_K block with the same fields
    rng = np.random.default_rng(53)
    M, N, K = 2, 3, 512
    xq = oracle.quantize_q8_1(synth.activations(53, M, K, True))
    w4, d, dmin, sc, mn, codes = _random_q4_k(rng, N, K)
    w5 = np.stack([q5_k_super_block(int(np.float16(d[n, s]).view(np.uint16)),
                                    int(np.float16(dmin[n, s]).view(np.uint16)), sc[n, s], mn[n, s], codes[n, s])
                   for n in range(N) for s in range(K // 256)]).reshape(N, -1)
    o4, _ = oracle.gemm("q4_k", xq, w4, M, N, K)
    o5, _ = oracle.gemm("q5_k", xq, w5, M, N, K)
    assert np.array_equal(o4, o5)


def test_q4_k_zero_sub_scales_leave_only_the_min_term():
    rng = np.random.default_rng(41)
    M, N, K = 3, 2, 512
    x = synth.activations(41, M, K, True)
    xq = oracle.quantize_q8_1(x)
    w, d, dmin, sc, mn, codes = _random_q4_k(rng, N, K)
    w2 = w.reshape(N, 2, 144).copy()
    for n in range(N):
        for s in range(2):
            w2[n, s, 4:16] = pack_scales([0] * 8, mn[n, s])
    out, _ = oracle.gemm("q4_k", xq, w2.reshape(N, -1), M, N, K)
    _, sa, _ = split_q8_1(xq)
    mterm = (dmin[:, :, None] * mn).reshape(N, 16)
    assert np.allclose(out, -(sa @ mterm.T), rtol=1e-13, atol=0)


def test_q8_0_all_ones_weights_give_scaled_block_sums():
    M, N, K = 4, 3, 256
    x = synth.activations(43, M, K, True)
    xq = oracle.quantize_q8_1(x)
    w = np.zeros((N, K // 32, 34), dtype=np.uint8)
    wd = np.array([0.25, 0.5, 3.0], dtype=np.float16)
    w[:, :, 0:2] = wd.view(np.uint8).reshape(N, 1, 2)
    w[:, :, 2:] = 1
    out, _ = oracle.gemm("q8_0", xq, w.reshape(N, -1), M, N, K)
    da, _, qa = split_q8_1(xq)
    rowsum = (da * qa.sum(axis=2)).sum(axis=1)
    assert np.allclose(out, rowsum[:, None] * wd.astype(np.float64)[None, :], rtol=1e-13, atol=0)


def test_sampled_entries_match_full_contraction():
    for fmt, K in (("q8_0", 256), ("q4_k", 512)):
        M, N = 9, 11
        x = synth.activations(50, M, K, True)
        xq = oracle.quantize_q8_1(x)
        wq = synth.weights(fmt, 51, N, K)
        out, norm = oracle.gemm(fmt, xq, wq, M, N, K)
        rng = np.random.default_rng(1)
        im, inn = rng.integers(0, M, 40), rng.integers(0, N, 40)
        o2, n2 = oracle.gemm_at(fmt, xq, wq, M, N, K, im, inn)
        assert np.array_equal(o2, out[im, inn]) and np.array_equal(n2, norm[im, inn])


def _random_q6_k(rng, N, K):
    nsb = K // 256
    d = (rng.uniform(1e-5, 1e-4, (N, nsb)) * rng.choice([-1.0, 1.0], (N, nsb))).astype(np.float16)
    sc = rng.integers(-128, 128, (N, nsb, 16))
    codes = rng.integers(0, 64, (N, nsb, 256))
    w = np.stack([q6_k_super_block(int(d[n, s].view(np.uint16)), sc[n, s], codes[n, s])
                  for n in range(N) for s in range(nsb)]).reshape(N, nsb * 210)
    return w, d.astype(np.float64), sc, codes


def test_block_dots_q6_k_brute_force_on_packed_codes():
    # every element's six bits and its group's sub-scale land where the decoder looks
    rng = np.random.default_rng(61)
    M, N, K = 3, 5, 512
    xq = oracle.quantize_q8_1(synth.activations(61, M, K, True))
    w, d, sc, codes = _random_q6_k(rng, N, K)
    dots = oracle.block_dots("q6_k", xq, w, M, N, K)
    _, _, qa = split_q8_1(xq)
    wv = (codes - 32) * np.repeat(sc, 16, axis=2)                   # (q - 32) * sc per element
    ref = np.einsum("mbk,nbk->mnb", qa, wv.reshape(N, K // 32, 32))
    assert np.array_equal(dots, ref)
    assert np.abs(ref).max() > 2 ** 17  # the sub-scales reach the dots (not only the codes)


@pytest.mark.parametrize("M,N,K", [(1, 1, 256), (2, 3, 512), (4, 2, 768)])
def test_q6_k_equals_dequantized_fp64_matmul(M, N, K):
    rng = np.random.default_rng(M * 100 + N * 10 + K + 6)
    xq = oracle.quantize_q8_1(synth.activations(70 + M, M, K, True))
    w, d, sc, codes = _random_q6_k(rng, N, K)
    out, norm = oracle.gemm("q6_k", xq, w, M, N, K)
    nsb = K // 256
    wh = (d[:, :, None] * (np.repeat(sc, 16, axis=2) * (codes - 32))).reshape(N, K)
    da, _, qa = split_q8_1(xq)
    xh = (da[:, :, None] * qa).reshape(M, K)
    ref = xh @ wh.T
    scale = np.abs(xh) @ np.abs(wh).T
    assert np.all(np.abs(out - ref) <= 1e-12 * scale)
    assert np.all(norm >= np.abs(out) * (1 - 1e-15))


def test_q6_k_with_one_sub_scale_per_block_equals_q8_0():
    # both 16-element groups of every block share a sub-scale s_j in -3..3: the block is
    # the Q8_0 block with codes (q - 32) * s_j (|.| <= 96) and the super-block's d
    rng = np.random.default_rng(63)
    M, N, K = 2, 3, 512
    nsb = K // 256
    xq = oracle.quantize_q8_1(synth.activations(63, M, K, True))
    d = rng.uniform(1e-3, 1e-2, (N, nsb)).astype(np.float16)
    sj = rng.integers(-3, 4, (N, nsb, 8))
    codes = rng.integers(0, 64, (N, nsb, 256))
    w6 = np.stack([q6_k_super_block(int(d[n, s].view(np.uint16)), np.repeat(sj[n, s], 2), codes[n, s])
                   for n in range(N) for s in range(nsb)]).reshape(N, -1)
    c8 = ((codes.reshape(N, nsb, 8, 32) - 32) * sj[:, :, :, None]).astype(np.int8)
    w8 = np.zeros((N, nsb, 8, 34), dtype=np.uint8)
    w8[:, :, :, 0:2] = np.repeat(d[:, :, None], 8, axis=2).view(np.uint8).reshape(N, nsb, 8, 2)
    w8[:, :, :, 2:] = c8.view(np.uint8)
    w8 = w8.reshape(N, -1)
    o6, n6 = oracle.gemm("q6_k", xq, w6, M, N, K)
    o8, n8 = oracle.gemm("q8_0", xq, w8, M, N, K)
    assert np.array_equal(o6, o8) and np.array_equal(n6, n8)
    assert np.array_equal(oracle.block_dots("q6_k", xq, w6, M, N, K), oracle.block_dots("q8_0", xq, w8, M, N, K))
