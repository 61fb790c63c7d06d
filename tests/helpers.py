"""Shared helpers of the GPU parity tests: tolerances and comparisons.

Tolerances (stated by the problem for floating point):
* f32 sums: |gpu - oracle| <= 2^-20 * sum |f(x_i)| per output;
* bf16 outputs (f32 accumulate): within 1 bf16 ulp of the correctly rounded
  oracle value;
* f32 scans: per element <= 2^-20 * sum_{j<=i} |x_j| (the reduce rule applied
  to every prefix);
* f64 scans: per element <= 2^-36 * sum_{j<=i} |x_j| (a depth bound of about
  (tiles + tile length) * 2^-53 for 1e8 elements, with margin);
* integers, max / min and the 2x2 matrix product: bit-exact.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

F32_REL = 2.0**-20
F64_REL = 2.0**-36


def to_dev(a: np.ndarray, dtype=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def bf16_dev(bits: np.ndarray, rows_shape) -> torch.Tensor:
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).reshape(rows_shape).cuda()


def bf16_key(bits: np.ndarray) -> np.ndarray:
    """Monotonic integer key of bf16 bit patterns (adjacent values differ by 1)."""
    b = bits.astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b & 0x7FFF)


def assert_bf16_within_1ulp(got_bits: np.ndarray, exact_f64: np.ndarray):
    want = oracle.bf16_rne_array(exact_f64)
    d = np.abs(bf16_key(got_bits.ravel()) - bf16_key(want.ravel()))
    assert d.max(initial=0) <= 1, f"bf16 off by {d.max()} ulp at {np.argmax(d)}"


def assert_close_f32(got, want, absmass, rel=F32_REL):
    got = np.asarray(got, dtype=np.float64).ravel()
    want = np.asarray(want, dtype=np.float64).ravel()
    tol = rel * np.asarray(absmass, dtype=np.float64).ravel()
    err = np.abs(got - want)
    bad = err > tol
    assert not bad.any(), (f"{bad.sum()} of {bad.size} outside tolerance; first at {np.argmax(bad)}: "
                           f"got {got[np.argmax(bad)]!r} want {want[np.argmax(bad)]!r} tol {tol[np.argmax(bad)]!r}")


def assert_exact(got, want):
    got = np.asarray(got).ravel()
    want = np.asarray(want).ravel()
    assert got.shape == want.shape
    diff = got != want
    assert not diff.any(), f"{diff.sum()} mismatches; first at {np.argmax(diff)}: {got[np.argmax(diff)]} vs {want[np.argmax(diff)]}"


def colmajor_mass(x64: np.ndarray, shape, dims) -> np.ndarray:
    """sum |x| over the reduced column-major dims, flat in the output order."""
    arr = np.abs(x64).reshape(tuple(reversed(shape)))
    axes = tuple(len(shape) - 1 - d for d in dims)
    return arr.sum(axis=axes, keepdims=True).ravel()


def gen(kind: str, n: int, seed: int = 0, stream: int = 0, dist: str = "uniform"):
    """Seeded input of n elements of a kind, in the workload distributions."""
    if kind == "f32":
        return synth.normal_f32(n, seed, stream) if dist == "normal" else synth.uniform_f32_pm1(n, seed, stream)
    if kind == "f64":
        return synth.normal_f64(n, seed, stream) if dist == "normal" else synth.uniform_f64_01(n, seed, stream)
    if kind == "bf16":
        return synth.normal_bf16_bits(n, seed, stream)
    if kind == "i32":
        return synth.uniform_int(n, -1000, 1000, np.int32, seed, stream)
    if kind == "i64":
        return synth.uniform_int(n, -(2**20), 2**20, np.int64, seed, stream)
    if kind == "mat2":
        return synth.mat2_modp(n, seed, stream)
    raise ValueError(kind)


def dev_of(kind: str, a: np.ndarray) -> torch.Tensor:
    if kind == "bf16":
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()
