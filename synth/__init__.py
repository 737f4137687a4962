"""Seeded synthetic operands for block-quantized int8 MMQ.

This module draws random numbers and lays them out as the byte formats the library
consumes.  It holds none of the method's arithmetic: no quantization, no scale
decoding, no dot products.  Both the oracle-based tests and the GPU path take their
inputs from here, so the two sides always see the same bytes.

Generator: splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014), used counter-style: output i of stream `seed` is
mix(seed + (i + 1) * 0x9E3779B97F4A7C15).  Uniform doubles take the top 53 bits;
normals use the Box-Muller transform in double precision, then cast to f32.

Value recipes (sizes are the projections of a 7B GQA transformer at 2K-token prefill):
  activations  x ~ N(0, 1) in f32; with `outliers`, each entry is multiplied by 20
               with probability 0.01 (independent Bernoulli).
  Q8_0 weights codes uniform in [-127, 127]; block scale d = f16(|N(0, 0.02)| / 127).
  Q4_K weights d, dmin = f16(U(1e-4, 2e-3)); the 12 packed scale bytes and the 128
               nibble bytes are uniform random bytes.  Every 96-bit pattern of the
               scale bytes is a valid set of eight 6-bit sub-scales and eight 6-bit
               sub-mins, and uniform bytes make each of them uniform on 0..63.
"""
from __future__ import annotations

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

QK = 32
QK_K = 256
Q8_1_BYTES = 36
Q8_0_BYTES = 34
Q4_K_BYTES = 144
Q5_K_BYTES = 176
Q6_K_BYTES = 210

BASE_SEED = 0x4D4D51


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """Outputs offset .. offset+n-1 of the splitmix64 stream started at `seed`."""
    out = np.empty(n, dtype=np.uint64)
    s = np.uint64(seed & 0xFFFFFFFFFFFFFFFF)
    with np.errstate(over="ignore"):
        for lo in range(0, n, _CHUNK):
            hi = min(n, lo + _CHUNK)
            i = np.arange(offset + lo + 1, offset + hi + 1, dtype=np.uint64)
            out[lo:hi] = _mix(s + i * _GOLDEN)
    return out


def substream(seed: int, tag: int) -> int:
    """A derived seed for an independent stream (one per array drawn)."""
    return int(splitmix64(seed ^ ((tag * 0xD1B54A32D192ED03) & 0xFFFFFFFFFFFFFFFF), 1)[0])


def uniform01(seed: int, n: int) -> np.ndarray:
    return (splitmix64(seed, n) >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def normal(seed: int, n: int) -> np.ndarray:
    u1 = uniform01(substream(seed, 1), n)
    u2 = uniform01(substream(seed, 2), n)
    return np.sqrt(-2.0 * np.log1p(-u1)) * np.cos(2.0 * np.pi * u2)


def random_bytes(seed: int, n: int) -> np.ndarray:
    words = splitmix64(seed, (n + 7) // 8)
    return words.view(np.uint8)[:n].copy()


def activations(seed: int, M: int, K: int, outliers: bool = True) -> np.ndarray:
    """f32 [M, K]: N(0, 1), with 1% of entries scaled by 20 when `outliers`."""
    x = normal(substream(seed, 10), M * K)
    if outliers:
        hit = uniform01(substream(seed, 11), M * K) < 0.01
        x = np.where(hit, x * 20.0, x)
    return x.astype(np.float32).reshape(M, K)


def q8_0_weights(seed: int, N: int, K: int) -> np.ndarray:
    """uint8 [N, K/32*34]: per block f16 d (little-endian) then 32 int8 codes."""
    assert K % QK == 0
    nb = K // QK
    codes = (splitmix64(substream(seed, 20), N * K) % np.uint64(255)).astype(np.int16) - 127
    d = (np.abs(normal(substream(seed, 21), N * nb)) * 0.02 / 127.0).astype(np.float16)
    blk = np.empty((N * nb, Q8_0_BYTES), dtype=np.uint8)
    blk[:, 0:2] = d.view(np.uint8).reshape(-1, 2)
    blk[:, 2:] = codes.astype(np.int8).view(np.uint8).reshape(-1, QK)
    return blk.reshape(N, nb * Q8_0_BYTES)


def q4_k_weights(seed: int, N: int, K: int) -> np.ndarray:
    """uint8 [N, K/256*144]: per super-block f16 d, f16 dmin, 12 scale bytes, 128 nibble bytes."""
    assert K % QK_K == 0
    nsb = K // QK_K
    u = uniform01(substream(seed, 30), 2 * N * nsb)
    dd = (1e-4 + u * (2e-3 - 1e-4)).astype(np.float16).reshape(-1, 2)
    blk = np.empty((N * nsb, Q4_K_BYTES), dtype=np.uint8)
    blk[:, 0:4] = dd.view(np.uint8).reshape(-1, 4)
    blk[:, 4:] = random_bytes(substream(seed, 31), N * nsb * 140).reshape(-1, 140)
    return blk.reshape(N, nsb * Q4_K_BYTES)


def q5_k_weights(seed: int, N: int, K: int) -> np.ndarray:
    """uint8 [N, K/256*176]: per super-block f16 d, f16 dmin, then 172 uniform bytes (12
    scale bytes, 32 high-bit bytes, 128 nibble bytes: every byte pattern is valid)."""
    assert K % QK_K == 0
    nsb = K // QK_K
    u = uniform01(substream(seed, 32), 2 * N * nsb)
    dd = (1e-4 + u * (2e-3 - 1e-4)).astype(np.float16).reshape(-1, 2)
    blk = np.empty((N * nsb, Q5_K_BYTES), dtype=np.uint8)
    blk[:, 0:4] = dd.view(np.uint8).reshape(-1, 4)
    blk[:, 4:] = random_bytes(substream(seed, 33), N * nsb * (Q5_K_BYTES - 4)).reshape(-1, Q5_K_BYTES - 4)
    return blk.reshape(N, nsb * Q5_K_BYTES)


def q6_k_weights(seed: int, N: int, K: int) -> np.ndarray:
    """uint8 [N, K/256*210]: per super-block 208 uniform bytes (128 low-nibble bytes, 64
    bytes of 2-bit high parts, 16 int8 sub-scales: every byte pattern is valid), then f16 d
    of either sign, |d| in [1e-5, 1e-4]."""
    assert K % QK_K == 0
    nsb = K // QK_K
    u = uniform01(substream(seed, 34), N * nsb)
    sign = np.where(uniform01(substream(seed, 35), N * nsb) < 0.5, -1.0, 1.0)
    d = (sign * (1e-5 + u * (1e-4 - 1e-5))).astype(np.float16)
    blk = np.empty((N * nsb, Q6_K_BYTES), dtype=np.uint8)
    blk[:, :208] = random_bytes(substream(seed, 36), N * nsb * 208).reshape(-1, 208)
    blk[:, 208:] = d.view(np.uint8).reshape(-1, 2)
    return blk.reshape(N, nsb * Q6_K_BYTES)


def weights(fmt: str, seed: int, N: int, K: int) -> np.ndarray:
    if fmt == "q8_0":
        return q8_0_weights(seed, N, K)
    if fmt == "q4_k":
        return q4_k_weights(seed, N, K)
    if fmt == "q5_k":
        return q5_k_weights(seed, N, K)
    if fmt == "q6_k":
        return q6_k_weights(seed, N, K)
    raise ValueError(f"unknown weight format {fmt!r}")


def row_bytes(fmt: str, K: int) -> int:
    return {"q8_0": K // QK * Q8_0_BYTES, "q4_k": K // QK_K * Q4_K_BYTES, "q5_k": K // QK_K * Q5_K_BYTES,
            "q6_k": K // QK_K * Q6_K_BYTES}[fmt]


# The five workloads: (format, M, N, K).  Seeds are BASE_SEED + index.
CONFIGS = {
    0: dict(name="q8_0 tiny", fmt="q8_0", M=64, N=256, K=512, outliers=False),
    1: dict(name="q8_0 attention-proj 512x3584x3584", fmt="q8_0", M=512, N=3584, K=3584, outliers=True),
    2: dict(name="q4_k ffn-up 2048x18944x3584", fmt="q4_k", M=2048, N=18944, K=3584, outliers=True),
    3: dict(name="q4_k ffn-down 2048x3584x18944", fmt="q4_k", M=2048, N=3584, K=18944, outliers=True),
}

# One 7B GQA layer's projections (N, K) at prefill, Q4_K weights.
LAYER_7B = [
    ("q", 3584, 3584),
    ("k", 512, 3584),
    ("v", 512, 3584),
    ("o", 3584, 3584),
    ("gate", 18944, 3584),
    ("up", 18944, 3584),
    ("down", 3584, 18944),
]
LAYERS_7B = 28
M_SWEEP = [1, 8, 32, 128, 512, 2048, 8192]


def config_operands(index: int, M: int | None = None):
    """(x f32 [M,K], w uint8 [N,rowbytes], spec) for config `index` (0..3)."""
    spec = dict(CONFIGS[index])
    if M is not None:
        spec["M"] = M
    seed = BASE_SEED + index
    x = activations(substream(seed, 100), spec["M"], spec["K"], spec["outliers"])
    w = weights(spec["fmt"], substream(seed, 200), spec["N"], spec["K"])
    return x, w, spec


def layer_weights(layer: int, proj: str, N: int, K: int) -> np.ndarray:
    seed = substream(BASE_SEED + 4, 1000 + 16 * layer + [p[0] for p in LAYER_7B].index(proj))
    return q4_k_weights(seed, N, K)


def layer_activations(layer: int, M: int, K: int, which: int) -> np.ndarray:
    return activations(substream(BASE_SEED + 4, 50000 + 16 * layer + which), M, K, True)
