"""GPU parity of ak_accumulate (inclusive scans) against the oracle.

The scan workloads at full size: cumsum of 1e8 f64; accumulate! of 1e7 f32
with max under Optional partials (no neutral element); cumsum along
dims=1 (Julia) of a 4096x4096 f32 matrix; the prefix product of 1e7 2x2
matrices mod 2^31-1, whole and along dims=1 of 1024x8192 matrices
(tile-scan PR #202: runs of each parity and partials of 4 to 16 bytes, whole
and along dims). Plus ragged sizes, init, in-place, strided dims, and the
bounded look-back wait running out on an injected missing publication.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mapreduce_prefix_scan_gb300 as ak
import oracle
import synth
from helpers import F32_REL, F64_REL, assert_close_f32, assert_exact, dev_of, gen

pytestmark = pytest.mark.gpu


def _mass_lines(x64, shape, dim):
    a = np.abs(x64)
    if dim < 0:
        return np.cumsum(a)
    return np.cumsum(a.reshape(tuple(reversed(shape))), axis=len(shape) - 1 - dim).ravel()


# --------------------------------------------------------------------------
# the scan workloads at full size
# --------------------------------------------------------------------------

def test_cumsum_1e8_f64():
    x = synth.uniform_f64_01(10**8, seed=0, stream=60)
    y = ak.ak_accumulate(dev_of("f64", x)).cpu().numpy()
    want = oracle.scan(x, "f64")
    assert_close_f32(y, want, np.cumsum(x), rel=F64_REL)


def test_cumsum_1e8_f32_and_i64():
    # the bench's f32 scan (the TMA pipeline) at full size, and the integer
    # scan through the same pipeline, bit-exact
    x = synth.normal_f32(10**8, seed=0, stream=65)
    y = ak.ak_accumulate(dev_of("f32", x)).cpu().numpy()
    assert_close_f32(y, oracle.scan(x, "f32"), np.cumsum(np.abs(x.astype(np.float64))))
    del x, y
    xi = synth.uniform_int(5 * 10**7, -(2**20), 2**20, np.int64, seed=0, stream=3)
    assert_exact(ak.ak_accumulate(dev_of("i64", xi)).cpu().numpy(), oracle.scan(xi, "i64"))


def test_accumulate_max_1e7_f32_no_neutral():
    x = synth.normal_f32(10**7, seed=0, stream=61)
    y = ak.ak_accumulate(dev_of("f32", x), op="max", opts=ak.make_opts(no_neutral=True)).cpu().numpy()
    assert_exact(y.astype(np.float64), oracle.scan(x, "f32", op="max"))


def test_cumsum_dims1_4096x4096_f32():
    shape = (4096, 4096)
    x = synth.normal_f32(4096 * 4096, seed=0, stream=62)
    y = ak.ak_accumulate(dev_of("f32", x).reshape(4096, 4096), dim=0).cpu().numpy()
    want = oracle.scan(x, "f32", shape, 0)
    assert_close_f32(y, want, _mass_lines(x.astype(np.float64), shape, 0))


def test_mat2_prefix_product_1e7():
    x = synth.mat2_modp(10**7, seed=0, stream=63)
    y = ak.ak_accumulate(dev_of("mat2", x), op="matmul", elem="mat2").cpu().numpy().view(np.uint32)
    assert_exact(y.reshape(-1, 4), oracle.scan(x, "mat2"))


def test_mat2_prefix_product_dims1_1024x8192():
    shape = (1024, 8192)
    x = synth.mat2_modp(1024 * 8192, seed=0, stream=64)
    xd = dev_of("mat2", x).reshape(8192, 1024, 4)
    y = ak.ak_accumulate(xd, op="matmul", elem="mat2", dim=0).cpu().numpy().view(np.uint32)
    assert_exact(y.reshape(-1, 4), oracle.scan(x, "mat2", shape, 0))


# --------------------------------------------------------------------------
# sizes, types, operators, init, in place
# --------------------------------------------------------------------------

SIZES = [1, 2, 31, 127, 128, 1023, 1024, 2047, 4096, 4097, 8191, 8192, 8193, 3 * 8192 + 5, 100_003, 1_234_567]


@pytest.mark.parametrize("n", SIZES)
def test_sizes_f32_f64_i64(n):
    x = gen("f32", n, stream=65, dist="normal")
    y = ak.ak_accumulate(dev_of("f32", x)).cpu().numpy()
    assert_close_f32(y, oracle.scan(x, "f32"), np.cumsum(np.abs(x.astype(np.float64))))
    xd = gen("f64", n, stream=66, dist="normal")
    y = ak.ak_accumulate(dev_of("f64", xd)).cpu().numpy()
    assert_close_f32(y, oracle.scan(xd, "f64"), np.cumsum(np.abs(xd)), rel=F64_REL)
    xi = gen("i64", n, stream=67)
    assert_exact(ak.ak_accumulate(dev_of("i64", xi)).cpu().numpy(), oracle.scan(xi, "i64"))


@pytest.mark.parametrize("n", [1, 100, 4096, 4097, 50_001])
@pytest.mark.parametrize("kind,acc,out", [("i32", "i32", "i32"), ("i32", "i64", "i64"), ("f32", "f64", "f64"),
                                          ("f32", "f64", "f32")])
@pytest.mark.parametrize("op", ["add", "max", "min", "mul"])
def test_types_ops(n, kind, acc, out, op):
    x = gen(kind, n, stream=68)
    if op == "mul":
        x = (np.sign(x) + (x == 0)).astype(x.dtype)  # +-1: products stay exact
    y = ak.ak_accumulate(dev_of(kind, x), op=op, acc=acc, out=out).cpu().numpy()
    if kind == "i32":
        assert_exact(y, oracle.scan(x, "i32", op=op, acc_bits=32 if acc == "i32" else 64))
    else:
        want = oracle.scan(x, "f32", op=op)
        if out == "f32" and op == "add":
            assert_close_f32(y, want, np.cumsum(np.abs(x.astype(np.float64))))
        elif op == "add":
            assert_close_f32(y, want, np.cumsum(np.abs(x.astype(np.float64))), rel=F64_REL)
        else:
            assert_exact(y.astype(np.float64), want)


@pytest.mark.parametrize("no_neutral", [False, True])
@pytest.mark.parametrize("op", ["add", "max", "min"])
def test_init_and_optional(no_neutral, op):
    n = 70_001
    x = gen("i64", n, stream=69)
    opts = ak.make_opts(no_neutral=no_neutral)
    y = ak.ak_accumulate(dev_of("i64", x), op=op, init=12345, opts=opts).cpu().numpy()
    assert_exact(y, oracle.scan(x, "i64", op=op, init=12345))
    y = ak.ak_accumulate(dev_of("i64", x), op=op, opts=opts).cpu().numpy()
    assert_exact(y, oracle.scan(x, "i64", op=op))


def test_in_place():
    x = gen("f64", 500_000, stream=70)
    xd = dev_of("f64", x)
    ak.ak_accumulate(xd, dst=xd)
    assert_close_f32(xd.cpu().numpy(), oracle.scan(x, "f64"), np.cumsum(np.abs(x)), rel=F64_REL)


@pytest.mark.parametrize("n", [1, 7, 8, 9, 1023, 1024, 1025, 3000, 123_457])
def test_mat2_sizes_and_init(n):
    x = synth.mat2_modp(n, stream=71)
    y = ak.ak_accumulate(dev_of("mat2", x), op="matmul", elem="mat2").cpu().numpy().view(np.uint32)
    assert_exact(y.reshape(-1, 4), oracle.scan(x, "mat2"))
    init = synth.mat2_modp(1, stream=72)[0]
    y = ak.ak_accumulate(dev_of("mat2", x), op="matmul", elem="mat2", init=init,
                         opts=ak.make_opts(no_neutral=True)).cpu().numpy().view(np.uint32)
    assert_exact(y.reshape(-1, 4), oracle.scan(x, "mat2", init=init))


# --------------------------------------------------------------------------
# long lines: the TMA tile scan (integer element types; lines of 128-byte
# rows, tiles of 256 rows: 8192 i32 or 4096 i64; a line's last tile may be
# partial or hold only a partial row; several lines must start on a row
# boundary) against the super-tile scan (forced by items_per_thread), and
# the super-tile scan on the same shapes for the other element types
# --------------------------------------------------------------------------

TMA_CASES = [("f32", 32), ("f64", 16), ("i64", 16), ("i32", 32), ("mat2", 8)]


def _scan_both(kind, x, shape, dim, **kw):
    """The default path and the super-tile path (forced by items_per_thread)."""
    items = {"f32": 32, "f64": 16, "i64": 16, "i32": 32, "mat2": 8}[kind]
    xd = dev_of(kind, x).reshape(tuple(reversed(shape)) + ((4,) if kind == "mat2" else ()))
    extra = {"op": "matmul", "elem": "mat2"} if kind == "mat2" else {}
    extra.update(kw)
    opts = extra.pop("opts", None)
    a = ak.ak_accumulate(xd, dim=dim, opts=opts, **extra)
    o2 = ak.make_opts(items_per_thread=items, no_neutral=bool(opts is not None and opts.no_neutral))
    b = ak.ak_accumulate(xd, dim=dim, opts=o2, **extra)
    return a.cpu().numpy(), b.cpu().numpy()


def _check_scan(kind, x, shape, dim, got, op="add"):
    if kind == "mat2":
        assert_exact(got.view(np.uint32).reshape(-1, 4), oracle.scan(x, "mat2", shape, dim))
    elif kind == "i32":
        assert_exact(got, oracle.scan(x, "i32", shape, dim, op=op, acc_bits=32))
    elif kind == "i64" or op != "add":
        assert_exact(got.astype(np.float64) if kind != "i64" else got, oracle.scan(x, kind, shape, dim, op=op))
    else:
        mass = _mass_lines(x.astype(np.float64), shape, dim)
        assert_close_f32(got, oracle.scan(x, kind, shape, dim), mass, rel=F64_REL if kind == "f64" else F32_REL)


@pytest.mark.parametrize("kind,rl", TMA_CASES)
@pytest.mark.parametrize("rows", [256 * 3, 256 * 3 + 1, 256 * 5 + 77])
@pytest.mark.parametrize("tail", [0, 1, 5])
def test_tma_single_line(kind, rl, rows, tail):
    n = rows * rl + tail
    x = synth.mat2_modp(n, stream=80) if kind == "mat2" else gen(kind, n, stream=80)
    a, b = _scan_both(kind, x, (n,), -1)
    _check_scan(kind, x, (n,), -1, a)
    _check_scan(kind, x, (n,), -1, b)


@pytest.mark.parametrize("kind,rl", TMA_CASES)
@pytest.mark.parametrize("rows,lines", [(256 * 2 + 5, 3), (256 * 4, 2), (300, 7)])
def test_tma_lines_along_dim1(kind, rl, rows, lines):
    shape = (rows * rl, lines)
    n = rows * rl * lines
    x = synth.mat2_modp(n, stream=81) if kind == "mat2" else gen(kind, n, stream=81)
    a, b = _scan_both(kind, x, shape, 0)
    _check_scan(kind, x, shape, 0, a)
    _check_scan(kind, x, shape, 0, b)


@pytest.mark.parametrize("op", ["max", "min", "add"])
def test_tma_optional_partials_and_init(op):
    n = 8192 * 6 + 40
    x = gen("f32", n, stream=82, dist="normal")
    opts = ak.make_opts(no_neutral=True)
    y = ak.ak_accumulate(dev_of("f32", x), op=op, opts=opts).cpu().numpy()
    _check_scan("f32", x, (n,), -1, y, op=op)
    xi = gen("i64", n, stream=83)
    y = ak.ak_accumulate(dev_of("i64", xi), op=op, init=-77, opts=opts).cpu().numpy()
    assert_exact(y, oracle.scan(xi, "i64", op=op, init=-77))


def test_f64_scan_special_values():
    # the long-line f64 scan folds rows in 64-bit fixed point; rows of only
    # zeros / subnormals and rows with an infinity take the plain f64 fold
    n = 4096 * 9 + 7
    z = np.full(n, -0.0)
    y = ak.ak_accumulate(dev_of("f64", z)).cpu().numpy()
    assert np.all(y == 0) and np.all(np.signbit(y))  # every prefix of -0.0 is -0.0
    k = synth.uniform_int(n, -1000, 1000, np.int64, stream=86)
    x = np.ldexp(synth.normal_f64(n, stream=87), k)  # exponents over the whole range
    x[5000:5100] = 0.0
    x[6016:6032] = 4.9e-322 * np.arange(1, 17)  # a row of subnormals only
    x[20000:20016] = -0.0
    want = oracle.scan(x, "f64")
    for opts in (None, ak.make_opts(items_per_thread=16)):
        y = ak.ak_accumulate(dev_of("f64", x), opts=opts).cpu().numpy()
        assert_close_f32(y, want, np.cumsum(np.abs(x)), rel=F64_REL)
    x[n - 100] = np.inf
    y = ak.ak_accumulate(dev_of("f64", x)).cpu().numpy()
    assert np.all(np.isfinite(y[: n - 100])) and np.all(y[n - 100:] == np.inf)
    assert_close_f32(y[: n - 100], want[: n - 100], np.cumsum(np.abs(x[: n - 100])), rel=F64_REL)


@pytest.mark.parametrize("exclusive", [False, True])
def test_f64_scan_magnitude_jumps(exclusive):
    # f64 sums on the TMA scan keep row prefixes in wide fixed point and scan
    # each row with FP64 additions, some of them backwards from the next
    # row's prefix; magnitudes that jump by 2^20 .. 2^60 inside a row, a warp
    # of rows or a tile, and zero-mean data whose prefix keeps returning near
    # zero, must all stay within the tolerance of the mass before each output
    n = 4096 * 50 + 5
    e = np.zeros(n, dtype=np.int64)
    e[np.arange(n) % 16 >= 8] = 20              # second half of every row 2^20 larger
    e[(np.arange(n) // 16) % 32 == 31] += 40    # the last row of every warp of rows larger again
    e[(np.arange(n) // 4096) % 3 == 2] -= 300   # every third tile tiny
    x = np.ldexp(synth.normal_f64(n, stream=88), e)
    x[: 4096 * 2] = synth.normal_f64(4096 * 2, stream=89)  # zero-mean start, prefix near 0
    init = 0.25 if exclusive else None
    y = ak.ak_accumulate(dev_of("f64", x), init=init, exclusive=exclusive).cpu().numpy()
    want = oracle.scan(x, "f64", init=init, exclusive=exclusive)
    a = np.abs(x)
    mass = (np.concatenate([[0.0], np.cumsum(a)[:-1]]) if exclusive else np.cumsum(a)) + abs(init or 0.0)
    assert_close_f32(y, want, mass, rel=F64_REL)


def test_tma_unaligned_views_fall_back():
    n = 8192 * 4 + 3
    x = gen("f32", n + 1, stream=84, dist="normal")
    xd = dev_of("f32", x)[1:]
    y = ak.ak_accumulate(xd).cpu().numpy()
    _check_scan("f32", x[1:], (n,), -1, y)
    out = torch.empty(n + 1, device="cuda")
    ak.ak_accumulate(dev_of("f32", x[1:]), dst=out[1:])
    _check_scan("f32", x[1:], (n,), -1, out[1:].cpu().numpy())


def test_tma_in_place_ragged():
    n = 4096 * 7 + 9
    x = gen("i64", n, stream=85)
    xd = dev_of("i64", x)
    ak.ak_accumulate(xd, dst=xd, op="max")
    assert_exact(xd.cpu().numpy(), oracle.scan(x, "i64", op="max"))


# --------------------------------------------------------------------------
# along dimensions
# --------------------------------------------------------------------------

@pytest.mark.parametrize("shape,dim", [((5000, 7), 0), ((100, 300), 1), ((33, 40, 5), 1), ((33, 40, 5), 2),
                                       ((7, 9000), 0), ((20_000, 3), 0), ((3, 20_000), 1), ((1, 50_000), 1),
                                       ((4097, 2), 0), ((2, 3, 4, 5), 3)])
def test_along_dims(shape, dim):
    n = int(np.prod(shape))
    x = gen("f32", n, stream=73, dist="normal")
    xd = dev_of("f32", x).reshape(tuple(reversed(shape)))
    y = ak.ak_accumulate(xd, dim=dim).cpu().numpy()
    assert_close_f32(y, oracle.scan(x, "f32", shape, dim), _mass_lines(x.astype(np.float64), shape, dim))
    xi = gen("i64", n, stream=74)
    y = ak.ak_accumulate(dev_of("i64", xi).reshape(tuple(reversed(shape))), dim=dim, op="max").cpu().numpy()
    assert_exact(y, oracle.scan(xi, "i64", shape, dim, op="max"))
    xm = synth.mat2_modp(n, stream=75)
    xmd = dev_of("mat2", xm).reshape(tuple(reversed(shape)) + (4,))
    y = ak.ak_accumulate(xmd, dim=dim, op="matmul", elem="mat2").cpu().numpy().view(np.uint32)
    assert_exact(y.reshape(-1, 4), oracle.scan(xm, "mat2", shape, dim))


@pytest.mark.parametrize("shape,dim", [((4096, 2048), 1), ((64, 3000), 1), ((5, 70_000), 1), ((300, 40, 77), 1)])
@pytest.mark.parametrize("exclusive", [False, True])
def test_strided_dims_in_chunks(shape, dim, exclusive):
    # few columns along a long strided dimension: the dimension is cut into
    # chunks (fold, then apply from the chunk totals before each chunk)
    n = int(np.prod(shape))
    rows = tuple(reversed(shape))
    x = gen("f32", n, stream=76, dist="normal")
    y = ak.ak_accumulate(dev_of("f32", x).reshape(rows), dim=dim, init=0.5, exclusive=exclusive).cpu().numpy()
    want = oracle.scan(x, "f32", shape, dim, init=0.5, exclusive=exclusive)
    mass = _mass_lines(x.astype(np.float64), shape, dim) + 0.5
    assert_close_f32(y, want, mass)
    xi = gen("i64", n, stream=77)
    o = ak.make_opts(no_neutral=True, exclusive=exclusive)
    y = ak.ak_accumulate(dev_of("i64", xi).reshape(rows), dim=dim, op="max", init=-3, opts=o).cpu().numpy()
    assert_exact(y, oracle.scan(xi, "i64", shape, dim, op="max", init=-3, exclusive=exclusive))
    xm = synth.mat2_modp(n, stream=78)
    init = synth.mat2_modp(1, stream=79)[0]
    y = ak.ak_accumulate(dev_of("mat2", xm).reshape(rows + (4,)), dim=dim, op="matmul", elem="mat2", init=init,
                         exclusive=exclusive).cpu().numpy().view(np.uint32)
    assert_exact(y.reshape(-1, 4), oracle.scan(xm, "mat2", shape, dim, init=init, exclusive=exclusive))


# --------------------------------------------------------------------------
# bounded waits
# --------------------------------------------------------------------------

def test_lookback_wait_runs_out_and_gpu_stays_usable():
    # Tile 5 never publishes its state (fault injection); its successor's
    # bounded wait runs out after 20 ms, the kernel records the failure and
    # every block leaves. The call reports AK_ERR_TIMEOUT; the next call works.
    x = gen("f64", 40 * 4096, stream=76)
    xd = dev_of("f64", x)
    opts = ak.make_opts(check=True, wait_limit_ns=20_000_000, debug_skip_publish_tile=5)
    with pytest.raises(ak.AkError) as ei:
        ak.ak_accumulate(xd, opts=opts)
    assert ei.value.status == 6
    y = ak.ak_accumulate(xd, opts=ak.make_opts(check=True)).cpu().numpy()
    assert_close_f32(y, oracle.scan(x, "f64"), np.cumsum(np.abs(x)), rel=F64_REL)


def test_lookback_wait_runs_out_on_the_tma_path():
    # The same injected missing publication on the TMA pipeline (i64, 4096
    # elements per tile): the look-back warp that needs tile 5's aggregate
    # gives up after 20 ms, every other role sees the error word and leaves,
    # the producer lets its copies land; the next call is correct.
    x = gen("i64", 40 * 4096 + 17, stream=77)
    xd = dev_of("i64", x)
    opts = ak.make_opts(check=True, wait_limit_ns=20_000_000, debug_skip_publish_tile=5)
    with pytest.raises(ak.AkError) as ei:
        ak.ak_accumulate(xd, opts=opts)
    assert ei.value.status == 6
    y = ak.ak_accumulate(xd, opts=ak.make_opts(check=True)).cpu().numpy()
    assert_exact(y, oracle.scan(x, "i64"))


def _mat2_hitting_p(n):
    # alternating [[1, p-1], [0, 1]] and [[1, 1], [0, 1]] (column-major
    # a11, a21, a12, a22): every second prefix has a12 = p - 1 + 1 = 0 mod p,
    # which an uncanonicalised product leaves as p
    p = synth.MODP
    x = np.zeros((n, 4), dtype=np.int32)
    x[:, 0] = 1
    x[:, 3] = 1
    x[0::2, 2] = p - 1
    x[1::2, 2] = 1
    return x


@pytest.mark.parametrize("shape,dim", [((50_001,), -1), ((1000, 40), 0), ((3, 20_000), 1), ((20_000, 3), 0)])
def test_mat2_results_are_canonical(shape, dim):
    n = int(np.prod(shape))
    x = _mat2_hitting_p(n)
    xd = dev_of("mat2", x).reshape(tuple(reversed(shape)) + (4,))
    y = ak.ak_accumulate(xd, dim=dim, op="matmul", elem="mat2").cpu().numpy().view(np.uint32).reshape(-1, 4)
    assert y.max() < synth.MODP
    assert_exact(y, oracle.scan(x, "mat2", shape, dim))
