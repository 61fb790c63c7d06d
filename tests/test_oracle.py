"""Pins of the CPU oracle against facts that do not come from the oracle:
closed forms, library routines (math.fsum, numpy integer sums, exact Python
integer matrix products, torch's bf16 conversion), hand-derived golden
fixtures, invariants, and brute force over association trees.

Every pin is chosen so that a plausible mistake in the oracle (a dropped
term, a wrong sign or index, a transposed operand, a double rounding, a
missing wrap) fails at least one of them.
"""
from __future__ import annotations

import functools
import itertools
import math
import os

import numpy as np
import pytest

import oracle
import synth

P = oracle.MODP
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 2, 7, 1000, 100_000])
def test_sum_one_to_n_int64(n):
    x = np.arange(1, n + 1, dtype=np.int64)
    assert oracle.reduce(x, "i64") == n * (n + 1) // 2


def test_sum_int32_wraps_mod_2_32():
    n = 100_000  # n(n+1)/2 = 5_000_050_000 > 2^31
    x = np.arange(1, n + 1, dtype=np.int32)
    exact = n * (n + 1) // 2
    wrapped = ((exact + 2**31) % 2**32) - 2**31
    assert oracle.reduce(x, "i32") == wrapped
    assert oracle.reduce(x, "i32", acc_bits=64) == exact


@pytest.mark.parametrize("kind", ["f32", "f64"])
def test_sum_one_to_n_float_exact(kind):
    n = 4096
    x = np.arange(1, n + 1).astype(np.float32 if kind == "f32" else np.float64)
    assert oracle.reduce(x, kind) == n * (n + 1) / 2


def test_abs2_and_abs_closed_forms():
    n = 3000
    x = -np.arange(1, n + 1, dtype=np.float32)
    assert oracle.reduce(x, "f32", map="abs2") == n * (n + 1) * (2 * n + 1) // 6
    assert oracle.reduce(x, "f32", map="abs") == n * (n + 1) // 2
    xi = -np.arange(1, n + 1, dtype=np.int64)
    assert oracle.reduce(xi, "i64", map="abs2") == n * (n + 1) * (2 * n + 1) // 6
    assert oracle.reduce(xi, "i64", map="abs") == n * (n + 1) // 2
    assert oracle.reduce(xi, "i64") == -n * (n + 1) // 2


def test_products_closed_forms():
    x = np.full(40, 2.0)
    assert oracle.reduce(x, "f64", op="mul") == 2.0**40
    xi = np.full(40, 2, dtype=np.int64)
    assert oracle.reduce(xi, "i64", op="mul") == 2**40
    assert oracle.reduce(xi[:33].astype(np.int32), "i32", op="mul") == 0  # 2^33 wraps to 0
    assert oracle.reduce(xi[:31].astype(np.int32), "i32", op="mul") == -(2**31)  # 2^31 wraps to INT32_MIN


def test_max_min_of_permutation():
    rng = np.random.default_rng(3)
    x = rng.permutation(10_000).astype(np.int64) - 5000
    assert oracle.reduce(x, "i64", op="max") == 4999
    assert oracle.reduce(x, "i64", op="min") == -5000
    xf = x.astype(np.float32)
    assert oracle.reduce(xf, "f32", op="max") == 4999.0
    assert oracle.reduce(xf, "f32", op="min") == -5000.0


@pytest.mark.parametrize("kind", ["f32", "f64", "i32", "i64"])
def test_scan_of_ones(kind):
    n = 5000
    x = np.ones(n, dtype={"f32": np.float32, "f64": np.float64, "i32": np.int32, "i64": np.int64}[kind])
    y = oracle.scan(x, kind)
    assert np.array_equal(y, np.arange(1, n + 1))


def test_init_applied_once_at_left():
    x = np.arange(1, 11, dtype=np.int64)
    assert oracle.reduce(x, "i64", init=100) == 155
    assert oracle.reduce(x, "i64", op="max", init=100) == 100
    assert oracle.reduce(x, "i64", op="max", init=-100) == 10
    y = oracle.scan(x, "i64", init=100)
    assert np.array_equal(y, 100 + np.cumsum(x))
    xf = np.arange(1, 11, dtype=np.float64)
    assert oracle.reduce(xf, "f64", init=0.5) == 55.5
    assert oracle.reduce(xf, "f64", op="mul", init=2.0) == 2.0 * math.factorial(10)


def test_empty_inputs():
    e = np.zeros(0, dtype=np.float32)
    assert oracle.reduce(e, "f32") is None
    assert oracle.reduce(e, "f32", init=3.0) == 3.0
    assert oracle.reduce(np.zeros(0, np.int64), "i64", op="max") is None
    assert oracle.reduce(np.zeros((0, 4), np.uint32), "mat2") is None
    assert oracle.scan(e, "f32").size == 0


# --------------------------------------------------------------------------
# library routines
# --------------------------------------------------------------------------

def test_float_sum_matches_fsum_on_grid_data():
    # uniform[-1,1) f32 lives on the 2^-23 grid: the f64 sum is exact and must
    # equal the correctly rounded exact sum from math.fsum bit for bit.
    x = synth.uniform_f32_pm1(200_000, seed=0, stream=11)
    assert oracle.reduce(x, "f32") == math.fsum(x.astype(np.float64))
    assert oracle.reduce(x, "f32", map="abs2") == math.fsum((x.astype(np.float64)) ** 2)
    assert oracle.reduce(x, "f32", map="abs") == math.fsum(np.abs(x.astype(np.float64)))


def test_float_sum_close_to_fsum_on_general_f64():
    x = synth.normal_f64(100_000, stream=12) * np.exp(synth.normal_f64(100_000, stream=13) * 10)
    r = oracle.reduce(x, "f64")
    ref = math.fsum(x)
    assert abs(r - ref) <= 2 * np.spacing(abs(ref)) + 1e-30


def test_bf16_input_sum_matches_fsum():
    bits = synth.normal_bf16_bits(4096, stream=14)
    vals = synth.bf16_bits_to_f32(bits).astype(np.float64)
    assert oracle.reduce(bits, "bf16") == math.fsum(vals)


@pytest.mark.parametrize("shape,dims", [((5, 7), (1,)), ((5, 7), (0,)), ((4, 6, 3), (1,)),
                                        ((4, 6, 3), (0, 2)), ((3, 1, 5, 2), (1, 3)),
                                        ((8, 9), (0, 1)), ((6, 0, 2), (0,))])
def test_reduce_dims_int_matches_numpy(shape, dims):
    n = int(np.prod(shape))
    x = synth.uniform_int(n, -1000, 1000, np.int64, stream=15)
    got = oracle.reduce_dims(x, "i64", shape, dims)
    arr = x.reshape(tuple(reversed(shape)))  # row-major view of the column-major array
    axes = tuple(len(shape) - 1 - d for d in dims)
    ref = arr.sum(axis=axes, keepdims=True)
    assert np.array_equal(got, np.ravel(ref))
    got_max = oracle.reduce_dims(x, "i64", shape, dims, op="max")
    if all(shape[d] > 0 for d in dims):
        assert np.array_equal(got_max, np.ravel(arr.max(axis=axes, keepdims=True)))
    else:
        assert got_max is None


def test_reduce_dims_float_matches_fsum_per_output():
    shape = (6, 50, 4)
    x = synth.uniform_f32_pm1(int(np.prod(shape)), stream=16)
    got = oracle.reduce_dims(x, "f32", shape, (1,), map="abs2")
    arr = x.astype(np.float64).reshape(4, 50, 6)
    for k in range(4):
        for i in range(6):
            assert got[i + 6 * k] == math.fsum(arr[k, :, i] ** 2)


def test_reduce_dims_all_equals_whole_reduce():
    x = synth.uniform_int(600, -50, 50, np.int32, stream=17)
    assert oracle.reduce_dims(x, "i32", (10, 6, 10), (0, 1, 2))[0] == oracle.reduce(x, "i32")


@pytest.mark.parametrize("shape,dim", [((1000,), -1), ((7, 9), 0), ((7, 9), 1), ((3, 4, 5), 1),
                                       ((3, 4, 5), 2), ((3, 4, 5), -1)])
def test_int_scan_matches_numpy_cumsum(shape, dim):
    n = int(np.prod(shape))
    x = synth.uniform_int(n, -(2**20), 2**20, np.int64, stream=18)
    y = oracle.scan(x, "i64", shape, dim)
    if dim < 0:
        ref = np.cumsum(x)
    else:
        ref = np.cumsum(x.reshape(tuple(reversed(shape))), axis=len(shape) - 1 - dim).ravel()
    assert np.array_equal(y, ref)
    ym = oracle.scan(x, "i64", shape, dim, op="max")
    if dim < 0:
        refm = np.maximum.accumulate(x)
    else:
        refm = np.maximum.accumulate(x.reshape(tuple(reversed(shape))), axis=len(shape) - 1 - dim).ravel()
    assert np.array_equal(ym, refm)


def test_float_scan_matches_fsum_prefixes():
    x = synth.normal_f64(400, stream=19)
    y = oracle.scan(x, "f64")
    for i in range(len(x)):
        assert abs(y[i] - math.fsum(x[: i + 1])) <= np.spacing(abs(y[i])) + 1e-300


def test_f32_scan_exact_on_grid_data():
    x = synth.uniform_f32_pm1(50_000, stream=20)
    y = oracle.scan(x, "f32")
    ref = np.cumsum(x.astype(np.float64))  # every prefix is exact in f64 on this grid
    assert np.array_equal(y, ref)


def test_int32_scan_wraps():
    x = np.full(10, 2**30, dtype=np.int32)
    y = oracle.scan(x, "i32")
    ref = [((k * 2**30 + 2**31) % 2**32) - 2**31 for k in range(1, 11)]
    assert list(y) == ref


# --------------------------------------------------------------------------
# bf16 rounding
# --------------------------------------------------------------------------

def test_bf16_rne_golden():
    with open(os.path.join(GOLDEN, "bf16_rne.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            v, want = line.split()
            assert oracle.bf16_rne(float.fromhex(v)) == int(want, 16), v
    assert oracle.bf16_rne(float("nan")) & 0x7f80 == 0x7f80
    assert oracle.bf16_rne(float("inf")) == 0x7f80
    assert oracle.bf16_rne(float("-inf")) == 0xff80


def test_bf16_rne_matches_torch_on_f32_values():
    torch = pytest.importorskip("torch")
    f = np.concatenate([synth.normal_f32(20_000, stream=21),
                        synth.normal_f32(5_000, stream=22) * np.float32(1e-38),
                        synth.normal_f32(5_000, stream=23) * np.float32(1e30)])
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_rne_array(f.astype(np.float64))
    assert np.array_equal(got, ref)


# --------------------------------------------------------------------------
# max / min semantics
# --------------------------------------------------------------------------

def test_julia_max_min_semantics():
    assert math.isnan(oracle.fmax(float("nan"), 1.0))
    assert math.isnan(oracle.fmax(1.0, float("nan")))
    assert math.isnan(oracle.fmin(float("nan"), -1.0))
    assert math.copysign(1.0, oracle.fmax(-0.0, 0.0)) == 1.0
    assert math.copysign(1.0, oracle.fmax(0.0, -0.0)) == 1.0
    assert math.copysign(1.0, oracle.fmin(-0.0, 0.0)) == -1.0
    assert math.copysign(1.0, oracle.fmin(0.0, -0.0)) == -1.0
    x = np.array([1.0, float("nan"), 3.0], dtype=np.float32)
    assert math.isnan(oracle.reduce(x, "f32", op="max"))
    y = oracle.scan(x, "f32", op="max")
    assert y[0] == 1.0 and math.isnan(y[1]) and math.isnan(y[2])


def test_running_max_properties():
    x = synth.normal_f32(20_000, stream=24)
    y = oracle.scan(x, "f32", op="max")
    assert np.all(np.diff(y) >= 0)
    assert y[0] == x[0]
    prev = np.concatenate([[-np.inf], y[:-1]])
    assert np.all((y == prev) | (y == x.astype(np.float64)))
    assert y[-1] == oracle.reduce(x, "f32", op="max")
    assert np.array_equal(y, np.maximum.accumulate(x.astype(np.float64)))


# --------------------------------------------------------------------------
# 2x2 matrices mod p
# --------------------------------------------------------------------------

def _as_matrix(v):
    """Column-major entries (a11, a21, a12, a22) -> exact Python-int 2x2."""
    a11, a21, a12, a22 = (int(t) for t in v)
    return np.array([[a11, a12], [a21, a22]], dtype=object)


def _exact_product(ms):
    """Left-to-right product over the integers (numpy object matmul), then mod p."""
    prod = functools.reduce(np.matmul, [_as_matrix(m) for m in ms])
    prod = prod % P
    return [int(prod[0, 0]), int(prod[1, 0]), int(prod[0, 1]), int(prod[1, 1])]


def test_mat2_golden():
    with open(os.path.join(GOLDEN, "mat2_modp.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            lhs, rhs = line.split("->")
            ops = [np.array([int(t) for t in part.split()], dtype=np.uint32) for part in lhs.split(";")]
            want = [int(t) for t in rhs.split()]
            got = oracle.reduce(np.stack(ops), "mat2")
            assert list(got) == want, line
            if len(ops) == 2:
                assert list(oracle.mat2_mul(ops[0], ops[1])) == want


def test_mat2_product_matches_exact_integer_product():
    x = synth.mat2_modp(24, stream=25)
    got = oracle.reduce(x, "mat2")
    assert list(got) == _exact_product(x)
    rev = _exact_product(x[::-1])
    assert list(got) != rev  # order matters: a swapped operand order is caught
    y = oracle.scan(x, "mat2")
    for i in range(len(x)):
        assert list(y[i]) == _exact_product(x[: i + 1])


def test_mat2_fibonacci_powers():
    # [[1,1],[1,0]]^n = [[F(n+1), F(n)], [F(n), F(n-1)]] (Fibonacci by recurrence).
    n = 5000
    q = np.tile(np.array([1, 1, 1, 0], dtype=np.uint32), (n, 1))
    y = oracle.scan(q, "mat2")
    fib = [0, 1]
    for _ in range(n + 1):
        fib.append(fib[-1] + fib[-2])
    for k in (1, 2, 10, 100, 1000, n):
        assert list(y[k - 1]) == [fib[k + 1] % P, fib[k] % P, fib[k] % P, fib[k - 1] % P]


def test_mat2_unipotent_sum_and_layout():
    # [[1,a_i],[0,1]] products = [[1, sum a_i],[0,1]]: stored (1, 0, sum, 1).
    a = synth.uniform_int(3000, 0, P - 1, np.int64, stream=26)
    x = np.zeros((3000, 4), dtype=np.uint32)
    x[:, 0] = 1
    x[:, 2] = a
    x[:, 3] = 1
    y = oracle.scan(x, "mat2")
    assert np.array_equal(y[:, 2].astype(np.int64), np.cumsum(a) % P)
    assert np.all(y[:, 0] == 1) and np.all(y[:, 1] == 0) and np.all(y[:, 3] == 1)


def test_mat2_init_on_the_left():
    x = synth.mat2_modp(5, stream=27)
    init = synth.mat2_modp(1, stream=28)[0]
    got = oracle.reduce(x, "mat2", init=init)
    assert list(got) == _exact_product([init] + list(x))
    y = oracle.scan(x, "mat2", init=init)
    assert list(y[-1]) == list(got)


def test_mat2_dims_and_scan_along_dims():
    shape = (3, 5)
    x = synth.mat2_modp(15, stream=29)
    r = oracle.reduce_dims(x, "mat2", shape, (0,))
    for j in range(5):
        assert list(r[j]) == _exact_product(x[3 * j: 3 * j + 3])
    r2 = oracle.reduce_dims(x, "mat2", shape, (1,))
    for i in range(3):
        assert list(r2[i]) == _exact_product(x[i::3])
    y = oracle.scan(x, "mat2", shape, dim=1)
    for i in range(3):
        for j in range(5):
            assert list(y[i + 3 * j]) == _exact_product(x[i: i + 3 * j + 1: 3])


# --------------------------------------------------------------------------
# invariants and brute force
# --------------------------------------------------------------------------

@pytest.mark.parametrize("kind,op", [("i64", "add"), ("i64", "max"), ("i32", "mul"), ("f32", "max"),
                                     ("f32", "min"), ("f64", "add"), ("mat2", "matmul")])
def test_last_scan_element_equals_reduce(kind, op):
    n = 3333
    if kind == "mat2":
        x = synth.mat2_modp(n, stream=30)
    elif kind == "i64":
        x = synth.uniform_int(n, -(2**20), 2**20, np.int64, stream=30)
    elif kind == "i32":
        x = synth.uniform_int(n, -3, 3, np.int32, stream=30)
    elif kind == "f32":
        x = synth.normal_f32(n, stream=30)
    else:
        x = synth.uniform_f64_01(n, stream=30)
    y = oracle.scan(x, kind, op=op)
    r = oracle.reduce(x, kind, op=op)
    if kind == "mat2":
        assert list(y[-1]) == list(r)
    else:
        assert y[-1] == r


def _all_trees(items, combine):
    if len(items) == 1:
        yield items[0]
        return
    for k in range(1, len(items)):
        for left in _all_trees(items[:k], combine):
            for right in _all_trees(items[k:], combine):
                yield combine(left, right)


@pytest.mark.parametrize("n", [2, 3, 5, 6])
def test_every_association_tree_agrees(n):
    x = synth.mat2_modp(n, stream=31 + n)
    want = list(oracle.reduce(x, "mat2"))
    for t in _all_trees([np.array(m) for m in x], oracle.mat2_mul):
        assert list(t) == want
    xi = synth.uniform_int(n, -(2**31), 2**31 - 1, np.int32, stream=40 + n)
    wi = oracle.reduce(xi, "i32", op="mul")

    def wmul(a, b):
        return ((a * b + 2**31) % 2**32) - 2**31

    for t in _all_trees([int(v) for v in xi], wmul):
        assert t == wi


def test_synth_is_deterministic_and_on_grid():
    a = synth.uniform_f32_pm1(1000, seed=0, stream=1)
    b = synth.uniform_f32_pm1(1000, seed=0, stream=1)
    c = synth.uniform_f32_pm1(1000, seed=0, stream=2)
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    assert np.all(a >= -1) and np.all(a < 1)
    assert np.all((a.astype(np.float64) * 2**23) % 1 == 0)
    # a slice regenerates from its offset
    w = synth.words(100, stream=5)
    assert np.array_equal(w[40:60], synth.words(20, stream=5, offset=40))
    i = synth.uniform_int(10_000, -1000, 1000, np.int32)
    assert i.min() == -1000 and i.max() == 1000


def test_signed_zero_follows_the_left_fold():
    # IEEE addition: -0 + -0 = -0 and -0 + +0 = +0; the left fold (and every
    # prefix of it) keeps those signs, for sums and scans in f64 and f32 inputs
    for kind, dt in (("f64", np.float64), ("f32", np.float32)):
        x = np.full(7, -0.0, dtype=dt)
        assert np.signbit(oracle.reduce(x, kind))
        assert np.all(np.signbit(oracle.scan(x, kind)))
        y = oracle.scan(np.array([-0.0, 0.0, -0.0], dtype=dt), kind)
        assert list(np.signbit(y)) == [True, False, False]
    # with an init of -0.0 the fold of -0.0 stays -0.0; a +0.0 init makes it +0.0
    assert np.signbit(oracle.reduce(np.full(3, -0.0), "f64", init=-0.0))
    assert not np.signbit(oracle.reduce(np.full(3, -0.0), "f64", init=0.0))


# --------------------------------------------------------------------------
# init in dims reductions and in float scans; float scans along a dimension
# (init applied exactly once, at the left of each output's fold: "Finish
# whole-array reductions on the device", section "Compatibility")
# --------------------------------------------------------------------------

def _colmajor_axes(shape, dims):
    return tuple(len(shape) - 1 - d for d in dims)


@pytest.mark.parametrize("shape,dims", [((5, 7), (1,)), ((5, 7), (0,)), ((4, 6, 3), (1,)),
                                        ((4, 6, 3), (0, 2)), ((3, 1, 5, 2), (1, 3))])
def test_reduce_dims_int_init_once_per_output(shape, dims):
    n = int(np.prod(shape))
    x = synth.uniform_int(n, -1000, 1000, np.int64, stream=50)
    arr = x.reshape(tuple(reversed(shape)))
    axes = _colmajor_axes(shape, dims)
    init = 123_457
    got = oracle.reduce_dims(x, "i64", shape, dims, init=init)
    assert np.array_equal(got, arr.sum(axis=axes, keepdims=True).ravel() + init)
    # max: an init above every element wins everywhere, one below none
    assert np.all(oracle.reduce_dims(x, "i64", shape, dims, op="max", init=5000) == 5000)
    assert np.array_equal(oracle.reduce_dims(x, "i64", shape, dims, op="max", init=-5000),
                          arr.max(axis=axes, keepdims=True).ravel())
    # product: init * prod(x) per output, wrapped to 64 bits (exact Python ints)
    xs = synth.uniform_int(n, -3, 3, np.int64, stream=51)
    got = oracle.reduce_dims(xs, "i64", shape, dims, op="mul", init=7)
    prods = np.ravel(np.prod(xs.reshape(tuple(reversed(shape))).astype(object), axis=axes, keepdims=True))
    assert [int(v) for v in got] == [((7 * int(p) + 2**63) % 2**64) - 2**63 for p in prods]


def test_reduce_dims_float_init_once_per_output():
    shape = (6, 50, 4)
    x = synth.uniform_f32_pm1(int(np.prod(shape)), stream=52)
    arr = x.astype(np.float64).reshape(4, 50, 6)
    for init in (0.375, -1.5):
        got = oracle.reduce_dims(x, "f32", shape, (1,), init=init)
        for k in range(4):
            for i in range(6):
                assert got[i + 6 * k] == math.fsum([init] + list(arr[k, :, i]))
    # abs2 applies to the elements, not to init
    got = oracle.reduce_dims(x, "f32", shape, (1,), map="abs2", init=-2.0)
    assert got[0] == math.fsum([-2.0] + list(arr[0, :, 0] ** 2))
    # empty reduced extent: every output is init
    assert np.all(oracle.reduce_dims(np.zeros(0, np.float32), "f32", (3, 0), (1,), init=2.5) == 2.5)


def test_reduce_dims_mat2_init_on_the_left():
    shape = (3, 5)
    x = synth.mat2_modp(15, stream=53)
    init = synth.mat2_modp(1, stream=54)[0]
    r = oracle.reduce_dims(x, "mat2", shape, (1,), init=init)
    for i in range(3):
        assert list(r[i]) == _exact_product([init] + list(x[i::3]))
    r = oracle.reduce_dims(x, "mat2", shape, (0,), init=init)
    for j in range(5):
        assert list(r[j]) == _exact_product([init] + list(x[3 * j: 3 * j + 3]))


@pytest.mark.parametrize("shape,dim", [((5, 7), 0), ((5, 7), 1), ((3, 4, 5), 1), ((3, 4, 5), 2)])
def test_float_scan_along_dim_matches_fsum_prefixes(shape, dim):
    n = int(np.prod(shape))
    x = synth.uniform_f32_pm1(n, stream=55)  # 2^-23 grid: every prefix is exact in f64
    arr = x.astype(np.float64).reshape(tuple(reversed(shape)))
    ax = len(shape) - 1 - dim
    for init in (None, 0.75):
        y = oracle.scan(x, "f32", shape, dim, init=init).reshape(arr.shape)
        moved = np.moveaxis(arr, ax, -1)
        ym = np.moveaxis(y, ax, -1)
        for idx in np.ndindex(moved.shape[:-1]):
            line = list(moved[idx])
            head = [] if init is None else [init]
            for j in range(len(line)):
                assert ym[idx][j] == math.fsum(head + line[: j + 1]), (idx, j)


def test_float_scan_init_once_at_the_left():
    x = synth.uniform_f32_pm1(2000, stream=56)
    xd = x.astype(np.float64)
    y = oracle.scan(x, "f32", init=-3.25)
    assert np.array_equal(y, np.cumsum(np.concatenate([[-3.25], xd]))[1:])
    # max with init: the running max never falls below init
    ym = oracle.scan(x, "f32", op="max", init=0.5)
    assert np.array_equal(ym, np.maximum.accumulate(np.maximum(xd, 0.5)))
    # f64 product with init: exact powers of two
    p = np.full(20, 2.0)
    assert list(oracle.scan(p, "f64", op="mul", init=3.0)) == [3.0 * 2.0**k for k in range(1, 21)]


# --------------------------------------------------------------------------
# exclusive scans: element i is the fold of init and x_1 .. x_{i-1}
# --------------------------------------------------------------------------

def test_exclusive_scan_of_ones_closed_form():
    for kind, dt in (("i64", np.int64), ("i32", np.int32), ("f64", np.float64), ("f32", np.float32)):
        y = oracle.scan(np.ones(1000, dtype=dt), kind, exclusive=True, init=5)
        assert list(y) == [5 + i for i in range(1000)]


@pytest.mark.parametrize("shape,dim", [((1000,), -1), ((7, 9), 0), ((7, 9), 1), ((3, 4, 5), 1)])
def test_exclusive_int_scan_matches_numpy(shape, dim):
    n = int(np.prod(shape))
    x = synth.uniform_int(n, -(2**20), 2**20, np.int64, stream=60)
    init = 77
    y = oracle.scan(x, "i64", shape, dim, exclusive=True, init=init)
    arr = x.reshape(tuple(reversed(shape))) if dim >= 0 else x
    ax = len(shape) - 1 - dim if dim >= 0 else 0
    inc = np.cumsum(arr, axis=ax)
    ref = np.concatenate([np.zeros_like(np.take(inc, [0], axis=ax)), np.delete(inc, -1, axis=ax)], axis=ax) + init
    assert np.array_equal(y, ref.ravel())
    ym = oracle.scan(x, "i64", shape, dim, op="max", exclusive=True, init=-(2**62))
    incm = np.maximum.accumulate(arr, axis=ax)
    refm = np.concatenate([np.full_like(np.take(incm, [0], axis=ax), -(2**62)), np.delete(incm, -1, axis=ax)],
                          axis=ax)
    assert np.array_equal(ym, refm.ravel())


def test_exclusive_float_scan_matches_fsum():
    x = synth.uniform_f32_pm1(3000, stream=61)
    xd = list(x.astype(np.float64))
    y = oracle.scan(x, "f32", exclusive=True, init=0.25)
    for i in (0, 1, 2, 999, 2999):
        assert y[i] == math.fsum([0.25] + xd[:i])
    assert y[0] == 0.25


def test_exclusive_mat2_scan_is_the_exact_product_of_the_elements_before():
    x = synth.mat2_modp(9, stream=62)
    init = synth.mat2_modp(1, stream=63)[0]
    y = oracle.scan(x, "mat2", exclusive=True, init=init)
    assert list(y[0]) == [int(v) for v in init]
    for i in range(1, 9):
        assert list(y[i]) == _exact_product([init] + list(x[:i]))


# --------------------------------------------------------------------------
# findall
# --------------------------------------------------------------------------

@pytest.mark.parametrize("kind", ["u8", "i32", "i64", "f32", "f64"])
def test_findall_matches_flatnonzero(kind):
    n = 10_000
    w = synth.uniform_int(n, 0, 3, np.int64, stream=64)
    x = np.where(w == 0, 0, w).astype({"u8": np.uint8, "i32": np.int32, "i64": np.int64, "f32": np.float32,
                                       "f64": np.float64}[kind])
    idx = oracle.findall(x, kind)
    assert np.array_equal(idx, np.flatnonzero(x))
    assert idx.size == int(np.count_nonzero(x))
    assert np.all(np.diff(idx) > 0)


def test_findall_special_values_and_empty():
    x = np.array([0.0, -0.0, np.nan, 1.0, -2.0, 0.0], dtype=np.float32)
    assert list(oracle.findall(x, "f32")) == [2, 3, 4]
    assert oracle.findall(np.zeros(0, np.uint8), "u8").size == 0
    assert oracle.findall(np.zeros(7, np.uint8), "u8").size == 0
    assert list(oracle.findall(np.full(5, 255, np.uint8), "u8")) == [0, 1, 2, 3, 4]


# --------------------------------------------------------------------------
# fused two-source reductions
# --------------------------------------------------------------------------

def test_reduce2_closed_forms():
    n = 2000
    k = np.arange(1, n + 1)
    for kind, dt in (("i64", np.int64), ("f64", np.float64), ("f32", np.float32)):
        x = k.astype(dt)
        y = (n + 1 - k).astype(dt)
        # sum k (n+1-k) = n(n+1)(n+2)/6
        assert oracle.reduce2(x, y, kind, "mul") == n * (n + 1) * (n + 2) // 6
        # (k - (k+1))^2 = 1
        assert oracle.reduce2(x, (k + 1).astype(dt), kind, "sqdiff") == n
        # |2k - (n+1)|, summed
        assert oracle.reduce2(x, y, kind, "absdiff") == sum(abs(2 * int(t) - (n + 1)) for t in k)
        assert oracle.reduce2(x, y, kind, "mul", op="max") == max(int(t) * (n + 1 - int(t)) for t in k)
        assert oracle.reduce2(x, y, kind, "mul", init=10) == n * (n + 1) * (n + 2) // 6 + 10


def test_reduce2_matches_fsum_and_numpy():
    x = synth.uniform_f32_pm1(5000, stream=65)
    y = synth.uniform_f32_pm1(5000, stream=66)
    xd, yd = x.astype(np.float64), y.astype(np.float64)
    assert oracle.reduce2(x, y, "f32", "mul") == math.fsum(xd * yd)       # products exact in f64
    assert oracle.reduce2(x, y, "f32", "sqdiff") == math.fsum((xd - yd) ** 2)
    xi = synth.uniform_int(5000, -1000, 1000, np.int32, stream=67)
    yi = synth.uniform_int(5000, -1000, 1000, np.int32, stream=68)
    assert oracle.reduce2(xi, yi, "i32", "mul") == int(np.dot(xi.astype(np.int64), yi.astype(np.int64)))
    assert oracle.reduce2(xi, yi, "i32", "absdiff") == int(np.abs(xi.astype(np.int64) - yi).sum())
    assert oracle.reduce2(np.zeros(0, np.float32), np.zeros(0, np.float32), "f32") is None


# --------------------------------------------------------------------------
# strided views
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dims", [(1,), (0,), (0, 1)])
def test_reduce_dims_of_a_strided_view_matches_numpy(dims):
    # a 6 x 5 column-major view into a 10 x 8 buffer, starting at (2, 1)
    buf = synth.uniform_int(80, -1000, 1000, np.int64, stream=69)
    base = 2 + 10 * 1
    shape, strides = (6, 5), (1, 10)
    flat = buf[base:]
    got = oracle.reduce_dims(flat, "i64", shape, dims, strides=strides)
    view = buf.reshape(8, 10)[1:6, 2:8]  # row-major view of the column-major sub-block
    axes = tuple(1 - d for d in dims)
    assert np.array_equal(got, view.sum(axis=axes, keepdims=True).ravel())
    # a transposed view (strides swapped) and a view with a stride-2 inner dimension
    got_t = oracle.reduce_dims(buf, "i64", (8, 10), (1,), strides=(10, 1))
    assert np.array_equal(got_t, buf.reshape(8, 10).sum(axis=1))
    got_2 = oracle.reduce_dims(buf, "i64", (5, 8), (0,), strides=(2, 10))
    assert np.array_equal(got_2, buf.reshape(8, 10)[:, ::2].sum(axis=1))
    xf = synth.uniform_f32_pm1(80, stream=70)
    got_f = oracle.reduce_dims(xf[base:], "f32", shape, (1,), strides=strides)
    vf = xf.astype(np.float64).reshape(8, 10)[1:6, 2:8]
    assert list(got_f) == [math.fsum(vf[:, i]) for i in range(6)]


# --------------------------------------------------------------------------
# affine maps mod p (the template API's user operator)
# --------------------------------------------------------------------------

def test_affine_scan_applied_to_a_value_equals_iteration():
    n = 500
    x = np.stack([synth.uniform_int(n, 0, P - 1, np.int64, stream=71),
                  synth.uniform_int(n, 0, P - 1, np.int64, stream=72)], axis=1).astype(np.uint32)
    y = oracle.scan_affine(x)
    v0 = 12345
    v = v0
    for i in range(n):
        v = (int(x[i, 0]) * v + int(x[i, 1])) % P
        assert (int(y[i, 0]) * v0 + int(y[i, 1])) % P == v
    assert list(oracle.reduce_affine(x)) == list(y[-1])
    # composition order matters: the reversed product differs
    assert list(oracle.reduce_affine(x[::-1].copy())) != list(y[-1])


def test_affine_special_cases_and_exclusive():
    n = 300
    b = synth.uniform_int(n, 0, P - 1, np.int64, stream=73)
    x = np.stack([np.ones(n, np.int64), b], axis=1).astype(np.uint32)  # translations: b's prefix sums
    y = oracle.scan_affine(x)
    assert np.array_equal(y[:, 1].astype(np.int64), np.cumsum(b) % P) and np.all(y[:, 0] == 1)
    init = np.array([3, 5], np.uint32)
    ye = oracle.scan_affine(x, init=init, exclusive=True)
    assert list(ye[0]) == [3, 5]
    # element i of the exclusive scan, then x_i, is element i of the inclusive scan with init
    yi = oracle.scan_affine(x, init=init)
    for i in range(n):
        assert list(oracle.affine_compose(ye[i], x[i])) == list(yi[i])
    assert list(yi[0]) == [3, (5 + int(b[0])) % P]
