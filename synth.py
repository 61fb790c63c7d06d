"""Seeded synthetic inputs for the reduce / scan workloads.

This module is shared by the tests, the bench and the oracle checks. It holds
none of the reduction or scan arithmetic: only a counter-based generator and
the mapping of its 64-bit words onto the value distributions of the workloads
(the shapes and distributions of the AcceleratedKernels.jl pull requests
"Finish whole-array reductions on the device" (#139, section "Numbers"), the
strided ``sum(x; dims=2)`` PR (#176, section "Timings") and the tile-scan PR
(#202, first two paragraphs)).

Generator: splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014), counter form: word i of a stream is
``mix(base + (i + 1) * GAMMA)`` with the published 64-bit finaliser ``mix``.
Each (seed, stream) pair gives an independent, reproducible sequence, so any
slice of an array can be regenerated without the rest of it.

Value mappings:
* uniform f32 in [-1, 1): ``k * 2**-23 - 1`` with k the top 24 bits, so every
  value sits on the 2**-23 grid and is exact in f32;
* uniform f64 in [0, 1): top 53 bits times 2**-53;
* integers in [lo, hi]: Lemire's multiply-shift on the top 32 bits;
* normal(0, 1): Box-Muller in f64 from two words, then rounded to the target
  type (f32 by IEEE cast, bf16 by torch's f32 -> bf16 conversion).
"""
from __future__ import annotations

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

# The modulus of the 2x2 matrix product workload: the Mersenne prime 2**31 - 1.
MODP = (1 << 31) - 1


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _base(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        s = np.array([(seed * 0x9E3779B97F4A7C15 + stream * 0xD1B54A32D192ED03 + 1)
                      & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
        return _mix(s)[0]


def words(n: int, seed: int = 0, stream: int = 0, offset: int = 0) -> np.ndarray:
    """n raw 64-bit words of stream (seed, stream), starting at word ``offset``."""
    out = np.empty(n, dtype=np.uint64)
    base = _base(seed, stream)
    with np.errstate(over="ignore"):
        for s in range(0, n, _CHUNK):
            e = min(n, s + _CHUNK)
            ctr = np.arange(offset + s + 1, offset + e + 1, dtype=np.uint64)
            out[s:e] = _mix(base + ctr * GAMMA)
    return out


def uniform_f32_pm1(n: int, seed: int = 0, stream: int = 0) -> np.ndarray:
    """f32 uniform on [-1, 1), on the 2**-23 grid (exact)."""
    out = np.empty(n, dtype=np.float32)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        k = (words(e - s, seed, stream, s) >> np.uint64(40)).astype(np.int64)
        out[s:e] = (k.astype(np.float64) * 2.0**-23 - 1.0).astype(np.float32)
    return out


def uniform_f64_01(n: int, seed: int = 0, stream: int = 0) -> np.ndarray:
    """f64 uniform on [0, 1): 53 random bits times 2**-53."""
    out = np.empty(n, dtype=np.float64)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        out[s:e] = (words(e - s, seed, stream, s) >> np.uint64(11)).astype(np.float64) * 2.0**-53
    return out


def uniform_int(n: int, lo: int, hi: int, dtype=np.int64, seed: int = 0, stream: int = 0) -> np.ndarray:
    """Integers uniform on [lo, hi] (hi - lo < 2**32) by multiply-shift."""
    span = hi - lo + 1
    assert 0 < span <= (1 << 32)
    out = np.empty(n, dtype=dtype)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        top = words(e - s, seed, stream, s) >> np.uint64(32)
        with np.errstate(over="ignore"):
            v = (top * np.uint64(span)) >> np.uint64(32)
        out[s:e] = (v.astype(np.int64) + lo).astype(dtype)
    return out


def normal_f64(n: int, seed: int = 0, stream: int = 0) -> np.ndarray:
    """normal(0, 1) in f64 by Box-Muller (one value per pair of words)."""
    out = np.empty(n, dtype=np.float64)
    for s in range(0, n, _CHUNK):
        e = min(n, s + _CHUNK)
        w = words(2 * (e - s), seed, stream, 2 * s)
        u1 = ((w[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0**-53  # (0, 1]
        u2 = (w[1::2] >> np.uint64(11)).astype(np.float64) * 2.0**-53         # [0, 1)
        out[s:e] = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    return out


def normal_f32(n: int, seed: int = 0, stream: int = 0) -> np.ndarray:
    return normal_f64(n, seed, stream).astype(np.float32)


def normal_bf16_bits(n: int, seed: int = 0, stream: int = 0) -> np.ndarray:
    """normal(0, 1) rounded to bf16, returned as the uint16 bit patterns."""
    import torch
    f = torch.from_numpy(normal_f32(n, seed, stream))
    return f.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def mat2_modp(n: int, seed: int = 0, stream: int = 0) -> np.ndarray:
    """n 2x2 matrices, entries uniform on [0, 2**31 - 1), as an (n, 4) int32
    array in column-major entry order (a11, a21, a12, a22)."""
    return uniform_int(4 * n, 0, MODP - 1, np.int32, seed, stream).reshape(n, 4)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to f32 (exact)."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
