"""Test-side helpers that BUILD Q4_K bytes from chosen values (the inverse direction of
the oracle's decoder), so that a transposed index or a wrong bit field in the decoder
shows up as a mismatch.  Written from the GGUF K-quant layout description: eight 6-bit
sub-scales and eight 6-bit sub-mins packed into 12 bytes, sub-blocks 4..7 split into a
low nibble (bytes 8..11) and two top bits (the spare top bits of bytes 0..7)."""
import numpy as np


def pack_scales(sc, m) -> np.ndarray:
    sc = [int(v) for v in sc]
    m = [int(v) for v in m]
    assert len(sc) == 8 and len(m) == 8 and all(0 <= v < 64 for v in sc + m)
    p = np.zeros(12, dtype=np.uint8)
    for j in range(4):
        p[j] = sc[j] | ((sc[j + 4] >> 4) << 6)
        p[j + 4] = m[j] | ((m[j + 4] >> 4) << 6)
        p[j + 8] = (sc[j + 4] & 15) | ((m[j + 4] & 15) << 4)
    return p


def pack_nibbles(codes) -> np.ndarray:
    """256 codes (0..15) in element order -> 128 bytes: byte 32c+i holds element 64c+i
    in its low half and element 64c+32+i in its high half."""
    codes = np.asarray(codes, dtype=np.uint8).reshape(4, 2, 32)
    assert codes.max() < 16
    return (codes[:, 0, :] | (codes[:, 1, :] << 4)).reshape(128).astype(np.uint8)


def super_block(d_f16: int, dmin_f16: int, sc, m, codes) -> np.ndarray:
    b = np.zeros(144, dtype=np.uint8)
    b[0:2] = np.array([d_f16], dtype=np.uint16).view(np.uint8)
    b[2:4] = np.array([dmin_f16], dtype=np.uint16).view(np.uint8)
    b[4:16] = pack_scales(sc, m)
    b[16:] = pack_nibbles(codes)
    return b


def q5_k_super_block(d_f16: int, dmin_f16: int, sc, m, codes) -> np.ndarray:
    """Q5_K super-block (176 B, the GGUF arrangement): f16 d, f16 dmin, the 12 scale bytes
    as Q4_K, 32 high-bit bytes, then the 128 nibble bytes of the low 4 bits.  Element
    64c + 32h + i (h = 0, 1) keeps its fifth bit in bit 2c + h of high-bit byte i."""
    codes = np.asarray(codes, dtype=np.int64).reshape(256)
    assert codes.min() >= 0 and codes.max() < 32
    b = np.zeros(176, dtype=np.uint8)
    b[0:2] = np.array([d_f16], dtype=np.uint16).view(np.uint8)
    b[2:4] = np.array([dmin_f16], dtype=np.uint16).view(np.uint8)
    b[4:16] = pack_scales(sc, m)
    qh = np.zeros(32, dtype=np.int64)
    for c in range(4):
        for h in range(2):
            qh |= ((codes[64 * c + 32 * h: 64 * c + 32 * h + 32] >> 4) & 1) << (2 * c + h)
    b[16:48] = qh.astype(np.uint8)
    b[48:] = pack_nibbles(codes & 15)
    return b


def q6_k_super_block(d_f16: int, sc, codes) -> np.ndarray:
    """Q6_K super-block (210 B, the GGUF arrangement) from 16 int8 sub-scales and 256
    codes (0..63) in element order: 128 bytes of low nibbles, 64 bytes of 2-bit high
    parts, the 16 sub-scales, f16 d.  Element 128h + 32t + l (t = 0..3, l = 0..31) keeps
    its low nibble in byte 64h + 32(t % 2) + l (the high half of the byte for t >= 2) and
    its top two bits in bits 2t, 2t + 1 of high-part byte 32h + l."""
    codes = np.asarray(codes, dtype=np.int64).reshape(2, 4, 32)   # [h][t][l]
    sc = np.asarray(sc, dtype=np.int64).reshape(16)
    assert codes.min() >= 0 and codes.max() < 64 and sc.min() >= -128 and sc.max() < 128
    b = np.zeros(210, dtype=np.uint8)
    for h in range(2):
        for tp in range(2):
            lo, hi = codes[h, tp] & 15, codes[h, tp + 2] & 15
            b[64 * h + 32 * tp: 64 * h + 32 * tp + 32] = (lo | (hi << 4)).astype(np.uint8)
        qh = np.zeros(32, dtype=np.int64)
        for t in range(4):
            qh |= (codes[h, t] >> 4) << (2 * t)
        b[128 + 32 * h: 160 + 32 * h] = qh.astype(np.uint8)
    b[192:208] = sc.astype(np.int8).view(np.uint8)
    b[208:210] = np.array([d_f16], dtype=np.uint16).view(np.uint8)
    return b
