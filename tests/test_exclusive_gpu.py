"""GPU parity of the exclusive scan (ak_accumulate with opts.exclusive) against
the oracle: element i holds the fold of init and the elements before it.

Every scan kernel is covered: the TMA pipeline (long f32 / i32 / i64 lines),
the super-tile scan (f64, mixed types, Optional partials, the matrix
product), lines that fit one tile (dims=1), and lines along a strided
dimension; with init and with the neutral element standing in for it.
Integers, max and the matrix product are bit-exact; float sums within
2^-20 (f32) / 2^-36 (f64) of sum_{j<i} |x_j| + |init|.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import mapreduce_prefix_scan_gb300 as ak
import oracle
import synth
from helpers import F32_REL, F64_REL, assert_close_f32, assert_exact, dev_of, gen

pytestmark = pytest.mark.gpu


def _excl_mass(x64, shape, dim, init):
    a = np.abs(x64)
    if dim < 0:
        c = np.cumsum(a)
        return np.concatenate([[0.0], c[:-1]]) + abs(init)
    arr = a.reshape(tuple(reversed(shape)))
    ax = len(shape) - 1 - dim
    c = np.cumsum(arr, axis=ax)
    c = np.concatenate([np.zeros_like(np.take(c, [0], axis=ax)), np.delete(c, -1, axis=ax)], axis=ax)
    return c.ravel() + abs(init)


def _run(kind, x, shape, dim, op="add", init=None, acc=None, out=None, no_neutral=False):
    rows = tuple(reversed(shape))
    xd = dev_of(kind, x).reshape(rows + ((4,) if kind == "mat2" else ()))
    opts = ak.make_opts(no_neutral=no_neutral, exclusive=True, check=True)
    y = ak.ak_accumulate(xd, dim=dim, shape=shape, op=op, init=init, acc=acc, out=out,
                         elem="mat2" if kind == "mat2" else None, opts=opts)
    return y.cpu().numpy()


# (kind, shape, dim): which kernel runs follows from the shape
CASES = [
    ("f32", (256 * 32 * 3 + 17,), -1),       # TMA pipeline, ragged last row
    ("i64", (256 * 16 * 4 + 3,), -1),        # TMA pipeline, 8-byte elements
    ("i32", (256 * 32 * 2, 3), 0),           # TMA pipeline, several lines
    ("f64", (300_001,), -1),                 # super-tiles
    ("f32", (4096, 50), 0),                  # lines that fit one tile
    ("i32", (3000, 7), 0),
    ("f32", (33, 40, 5), 1),                 # strided dimension
    ("i64", (33, 40, 5), 2),
]


@pytest.mark.parametrize("kind,shape,dim", CASES)
@pytest.mark.parametrize("init", [None, 3])
def test_exclusive_sum_matches_oracle(kind, shape, dim, init):
    n = int(np.prod(shape))
    x = gen(kind, n, stream=80, dist="normal" if kind == "f32" else "uniform")
    y = _run(kind, x, shape, dim, init=init)
    want = oracle.scan(x, kind, shape, dim, exclusive=True, init=0 if init is None else init)
    if kind in ("f32", "f64"):
        rel = F32_REL if kind == "f32" else F64_REL
        assert_close_f32(y, want, _excl_mass(x.astype(np.float64), shape, dim, init or 0), rel=rel)
    else:
        assert_exact(y, want)
    # the first element of every line is exactly init (or +0)
    first = y.reshape(-1)[0]
    assert first == (0 if init is None else init)
    if kind in ("f32", "f64") and init is None:
        assert not np.signbit(first)


@pytest.mark.parametrize("kind,shape,dim", [("f32", (300_001,), -1), ("i64", (70_000,), -1), ("f32", (2000, 9), 0),
                                            ("i32", (17, 300, 3), 1)])
@pytest.mark.parametrize("op", ["max", "min"])
def test_exclusive_max_min_with_init(kind, shape, dim, op):
    n = int(np.prod(shape))
    x = gen(kind, n, stream=81, dist="normal" if kind == "f32" else "uniform")
    init = -5 if op == "max" else 5
    y = _run(kind, x, shape, dim, op=op, init=init)
    assert_exact(np.asarray(y, dtype=np.float64 if kind == "f32" else np.int64),
                 oracle.scan(x, kind, shape, dim, op=op, exclusive=True, init=init))


@pytest.mark.parametrize("n", [1, 1000, 10**6 + 3])
def test_exclusive_optional_partials_with_init(n):
    # operator with no neutral element: init makes the first output exist
    x = synth.normal_f32(n, stream=82)
    y = _run("f32", x, (n,), -1, op="max", init=0.5, no_neutral=True)
    assert_exact(y.astype(np.float64), oracle.scan(x, "f32", op="max", exclusive=True, init=0.5))


@pytest.mark.parametrize("shape,dim", [((10**6 + 1,), -1), ((7, 5000), 1), ((1000, 40), 0)])
def test_exclusive_mat2_product(shape, dim):
    n = int(np.prod(shape))
    x = synth.mat2_modp(n, stream=83)
    init = synth.mat2_modp(1, stream=84)[0]
    y = _run("mat2", x, shape, dim, op="matmul", init=init).view(np.uint32).reshape(-1, 4)
    assert_exact(y, oracle.scan(x, "mat2", shape, dim, exclusive=True, init=init))
    # without init the identity matrix is the first output
    y0 = _run("mat2", x, shape, dim, op="matmul").view(np.uint32).reshape(-1, 4)
    assert_exact(y0, oracle.scan(x, "mat2", shape, dim, exclusive=True, init=np.array([1, 0, 0, 1], np.uint32)))


def test_exclusive_mixed_types_and_in_place():
    x = synth.uniform_int(200_001, -1000, 1000, np.int32, stream=85)
    y = _run("i32", x, (x.size,), -1, acc="i64", out="i64", init=7)
    assert_exact(y, oracle.scan(x, "i32", exclusive=True, init=7, acc_bits=64))
    f = synth.normal_f32(100_000, stream=86)
    fd = dev_of("f32", f)
    ak.ak_accumulate(fd, dst=fd, exclusive=True)
    assert_close_f32(fd.cpu().numpy(), oracle.scan(f, "f32", exclusive=True, init=0.0),
                     _excl_mass(f.astype(np.float64), (f.size,), -1, 0.0))


def test_exclusive_without_a_neutral_element_is_refused():
    x = dev_of("f32", synth.normal_f32(1000, stream=87))
    for kw in (dict(op="max"), dict(op="add", opts=ak.make_opts(no_neutral=True, exclusive=True))):
        with pytest.raises(ak.AkError, match="empty reduction"):
            ak.ak_accumulate(x, exclusive=True, **kw)


def test_exclusive_full_size_f32_1e8():
    x = synth.normal_f32(10**8, seed=0, stream=65)
    y = ak.ak_accumulate(dev_of("f32", x), exclusive=True).cpu().numpy()
    want = oracle.scan(x, "f32", exclusive=True, init=0.0)
    assert_close_f32(y, want, _excl_mass(x.astype(np.float64), (x.size,), -1, 0.0))


def test_scan_status_reports_ok_and_a_silent_timeout():
    x = dev_of("f32", synth.normal_f32(256 * 32 * 8, stream=88))
    n = x.numel()
    ws = torch.empty(ak.ak_accumulate_workspace_size([n], -1, "f32", "f32"), dtype=torch.uint8, device="cuda")
    ak.ak_accumulate(x, workspace=ws)
    torch.cuda.synchronize()
    assert ak.ak_scan_status(ws) == 0
    # a tile that never publishes: without `check` the call itself says ok,
    # the status query reports the timeout once the stream has passed it
    o = ak.make_opts(wait_limit_ns=20_000_000, debug_skip_publish_tile=2)
    ak.ak_accumulate(x, workspace=ws, opts=o)
    torch.cuda.synchronize()
    assert ak.ak_scan_status(ws) == 6
    # the next call clears it
    ak.ak_accumulate(x, workspace=ws)
    torch.cuda.synchronize()
    assert ak.ak_scan_status(ws) == 0
    # a lines-kernel call (no waits) also leaves a clean status
    m = dev_of("f32", synth.normal_f32(4000, stream=89)).reshape(40, 100)
    ak.ak_accumulate(m, dim=0, workspace=ws)
    torch.cuda.synchronize()
    assert ak.ak_scan_status(ws) == 0


@pytest.mark.parametrize("exclusive", [False, True])
def test_long_single_lines_with_init(exclusive):
    # single lines outside the TMA scan, long enough that the tile prefixes
    # come from the one-block prefix scan rather than from each apply block
    n = 5 * 10**6 + 17                          # 40 MB of f64
    x = synth.uniform_f64_01(n, stream=90)
    y = ak.ak_accumulate(dev_of("f64", x), init=0.5, exclusive=exclusive).cpu().numpy()
    want = oracle.scan(x, "f64", init=0.5, exclusive=exclusive)
    mass = (_excl_mass(x, (n,), -1, 0.5) if exclusive else np.cumsum(x) + 0.5)
    assert_close_f32(y, want, mass, rel=F64_REL)
    m = 3 * 10**6 + 5                           # 48 MB of 2x2 matrices mod p
    xm = synth.mat2_modp(m, stream=91)
    init = synth.mat2_modp(1, stream=92)[0]
    ym = ak.ak_accumulate(dev_of("mat2", xm), op="matmul", elem="mat2", init=init, exclusive=exclusive)
    assert_exact(ym.cpu().numpy().view(np.uint32).reshape(-1, 4),
                 oracle.scan(xm, "mat2", init=init, exclusive=exclusive))
    k = 2 * 10**7 + 3                           # 80 MB of f32 under Optional partials
    xo = synth.normal_f32(k, stream=93)
    yo = ak.ak_accumulate(dev_of("f32", xo), op="max", init=-0.25, exclusive=exclusive,
                          opts=ak.make_opts(no_neutral=True, exclusive=exclusive)).cpu().numpy()
    assert_exact(yo.astype(np.float64), oracle.scan(xo, "f32", op="max", init=-0.25, exclusive=exclusive))
