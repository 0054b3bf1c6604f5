"""Seeded synthetic inputs (Q, K, V ~ N(0, 1)) shared by the tests, the
benchmark and the oracle checks.

This module holds none of the method's arithmetic: it only draws numbers.  It
imports nothing from the CUDA binding or from the oracle, so both sides can be
fed the same buffers.

Recipe (version-independent, so every machine draws the same bits):
  * pair p of normals uses a = sm(seed ^ 2p) and b = sm(seed ^ (2p+1)), where
    sm is the SplitMix64 output function used purely as a counter-based
    generator;
  * u1 = ((a >> 11) + 1) * 2^-53 in (0, 1],  u2 = (b >> 11) * 2^-53 in [0, 1);
  * Box-Muller in float64: z0 = sqrt(-2 ln u1) cos(2 pi u2),
    z1 = sqrt(-2 ln u1) sin(2 pi u2);
  * rounded to nearest float32, then (bf16 workloads) to nearest-even
    bfloat16;
  * Q, then K, then V are filled in flat [B][H][n][d] order from one running
    pair counter.
"""
from __future__ import annotations

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _sm(x: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = x + _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def normals(seed: int, count: int, first_pair: int = 0, chunk: int = 1 << 22) -> np.ndarray:
    """`count` float64 N(0,1) draws starting at pair index `first_pair`."""
    out = np.empty(count, dtype=np.float64)
    s = np.uint64(seed & 0xFFFFFFFFFFFFFFFF)
    pairs = (count + 1) // 2
    two_pi = 2.0 * np.pi
    for p0 in range(0, pairs, chunk):
        p = np.arange(first_pair + p0, first_pair + min(pairs, p0 + chunk), dtype=np.uint64)
        a = _sm(s ^ (p * np.uint64(2)))
        b = _sm(s ^ (p * np.uint64(2) + np.uint64(1)))
        u1 = ((a >> np.uint64(11)) + np.uint64(1)).astype(np.float64) * 2.0 ** -53
        u2 = (b >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
        rad = np.sqrt(-2.0 * np.log(u1))
        z = np.empty(2 * p.size, dtype=np.float64)
        z[0::2] = rad * np.cos(two_pi * u2)
        z[1::2] = rad * np.sin(two_pi * u2)
        lo = 2 * p0
        hi = min(count, lo + z.size)
        out[lo:hi] = z[: hi - lo]
    return out


def to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """Round float32 to nearest-even bfloat16; returns the uint16 bit patterns."""
    u = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32)
    rounding = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32)


def qkv(B: int, H: int, n: int, d: int, dtype: str, seed: int = 0):
    """Q, K, V of shape [B][H][n][d].

    dtype "fp32" -> float32 arrays; "bf16" -> uint16 arrays of bfloat16 bits.
    """
    per = B * H * n * d
    out = []
    first = 0
    for _ in range(3):
        z = normals(seed, per, first_pair=first).astype(np.float32).reshape(B, H, n, d)
        first += (per + 1) // 2
        out.append(to_bf16_bits(z) if dtype == "bf16" else z)
    return tuple(out)


def checksum(*arrays: np.ndarray) -> str:
    """Short content hash of input buffers (printed so runs can be compared)."""
    import hashlib
    h = hashlib.sha256()
    for a in arrays:
        h.update(np.ascontiguousarray(a).tobytes())
    return h.hexdigest()[:16]


def layer_inputs(B: int, n: int, D: int, H: int, seed: int = 0):
    """Input and synthetic weights of the module with its projections, as bf16
    bit patterns: X [B][n][D] ~ N(0, 1); Wqkv [3 H 64][D] and Wo [D][H 64] ~
    N(0, 1) scaled by the power of two nearest 1/sqrt(fan-in) (exact in bf16).
    Drawn from one running pair counter: X, then Wqkv, then Wo."""
    d = 64
    sizes = (B * n * D, 3 * H * d * D, D * H * d)
    scales = (1.0, 2.0 ** -round(np.log2(np.sqrt(D))), 2.0 ** -round(np.log2(np.sqrt(H * d))))
    shapes = ((B, n, D), (3 * H * d, D), (D, H * d))
    out, first = [], 0
    for size, scale, shape in zip(sizes, scales, shapes):
        z = (normals(seed, size, first_pair=first) * scale).astype(np.float32).reshape(shape)
        first += (size + 1) // 2
        out.append(to_bf16_bits(z))
    return tuple(out)
