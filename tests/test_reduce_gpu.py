"""GPU parity of ak_reduce (whole-array mapreduce) against the oracle.

Covers the whole-array workloads at full size (1e6 f32 / i32 sums to host
and device; 1e8 f32 abs2 sum and 1e8 i64 sum and max into device arrays),
one tile / one pass / two passes, misaligned and ragged inputs, init / fold /
overwrite stores, accumulators wider than the output, Optional partials,
the order-preserving matrix product, workspace reuse and the empty rules
(reduction PR #139, section "Compatibility" and its last paragraph).
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import mapreduce_prefix_scan_gb300 as ak
import oracle
import synth
from helpers import assert_close_f32, assert_exact, dev_of, gen

pytestmark = pytest.mark.gpu

P = oracle.MODP


def _absmass(x, kind, f):
    x64 = synth.bf16_bits_to_f32(x).astype(np.float64) if kind == "bf16" else x.astype(np.float64)
    if f == "abs2":
        x64 = x64 * x64
    return float(np.abs(x64).sum())


# --------------------------------------------------------------------------
# the whole-array workloads at full size
# --------------------------------------------------------------------------

def test_sum_1e6_f32_host_and_device():
    x = synth.uniform_f32_pm1(10**6, seed=0, stream=0)
    xd = dev_of("f32", x)
    r = torch.full((1,), 123.0, device="cuda")
    ak.ak_reduce(xd, dst=r, init=0.0)
    h = ak.ak_reduce(xd, to_host=True, init=0.0)
    want = oracle.reduce(x, "f32", init=0.0)
    m = _absmass(x, "f32", "identity")
    assert abs(r.item() - want) <= 2.0**-20 * m
    assert abs(h - want) <= 2.0**-20 * m


def test_sum_1e6_i32_bit_exact():
    x = synth.uniform_int(10**6, -1000, 1000, np.int32, seed=0, stream=1)
    xd = dev_of("i32", x)
    r = torch.zeros(1, dtype=torch.int32, device="cuda")
    ak.ak_reduce(xd, dst=r)
    assert r.item() == oracle.reduce(x, "i32")
    assert ak.ak_reduce(xd, to_host=True) == oracle.reduce(x, "i32")


@pytest.fixture(scope="module")
def big_f32():
    return synth.uniform_f32_pm1(10**8, seed=0, stream=2)


@pytest.fixture(scope="module")
def big_i64():
    return synth.uniform_int(10**8, -(2**20), 2**20, np.int64, seed=0, stream=3)


def test_abs2_sum_1e8_f32(big_f32):
    xd = dev_of("f32", big_f32)
    r = torch.empty(1, dtype=torch.float32, device="cuda")
    ak.ak_reduce(xd, f="abs2", dst=r)
    want = oracle.reduce(big_f32, "f32", map="abs2")
    assert abs(r.item() - want) <= 2.0**-20 * want


@pytest.mark.parametrize("op", ["add", "max"])
def test_i64_1e8_bit_exact(big_i64, op):
    xd = dev_of("i64", big_i64)
    r = torch.empty(1, dtype=torch.int64, device="cuda")
    ak.ak_reduce(xd, op=op, dst=r)
    assert r.item() == oracle.reduce(big_i64, "i64", op=op)


# --------------------------------------------------------------------------
# sizes, alignment, types, ops, maps
# --------------------------------------------------------------------------

SIZES = [1, 2, 7, 31, 32, 33, 1000, 16384, 16385, 100_003, (1 << 20) + 13]


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("kind,acc,out", [("f32", "f32", "f32"), ("f32", "f64", "f64"), ("f64", "f64", "f64"),
                                          ("bf16", "f32", "f32"), ("i32", "i32", "i32"), ("i32", "i64", "i64"),
                                          ("i64", "i64", "i64")])
def test_sizes_types(n, kind, acc, out):
    x = gen(kind, n, stream=10 + n % 97)
    xd = dev_of(kind, x)
    for op, f in [("add", "identity"), ("max", "identity"), ("min", "abs"), ("add", "abs2")]:
        got = ak.ak_reduce(xd, op=op, f=f, acc=acc, out=out, to_host=True)
        if acc in ("i32", "i64"):
            want = oracle.reduce(x, kind, op=op, map=f, acc_bits=32 if acc == "i32" else 64)
            assert got == want, (n, kind, op, f)
        else:
            want = oracle.reduce(x, kind, op=op, map=f)
            if op in ("max", "min"):
                assert got == want
            else:
                rel = 2.0**-20 if acc == "f32" else 2.0**-45
                assert abs(got - want) <= rel * _absmass(x, kind, f), (n, kind, op, f)


@pytest.mark.parametrize("offset", [1, 2, 3, 5, 7])
def test_misaligned_source(offset):
    n = 200_001
    x = gen("f32", n + offset, stream=20)
    xd = dev_of("f32", x)[offset:]
    got = ak.ak_reduce(xd, to_host=True)
    want = oracle.reduce(x[offset:], "f32")
    assert abs(got - want) <= 2.0**-20 * _absmass(x[offset:], "f32", "identity")
    xi = gen("i64", n + offset, stream=21)
    assert ak.ak_reduce(dev_of("i64", xi)[offset:], to_host=True) == oracle.reduce(xi[offset:], "i64")


def test_int_mul_wraps():
    x = synth.uniform_int(5000, -3, 3, np.int32, stream=22)
    x[x == 0] = 1
    xd = dev_of("i32", x)
    assert ak.ak_reduce(xd, op="mul", to_host=True) == oracle.reduce(x, "i32", op="mul")
    assert ak.ak_reduce(xd, op="mul", acc="i64", to_host=True) == oracle.reduce(x, "i32", op="mul", acc_bits=64)


def test_bf16_input_bf16_output():
    bits = synth.normal_bf16_bits(777_777, stream=23)
    xd = dev_of("bf16", bits)
    r = torch.empty(1, dtype=torch.bfloat16, device="cuda")
    ak.ak_reduce(xd, acc="f32", out="bf16", dst=r)
    got = r.view(torch.int16).cpu().numpy().view(np.uint16)
    want = oracle.bf16_rne(oracle.reduce(bits, "bf16"))
    from helpers import bf16_key
    assert abs(int(bf16_key(got)[0]) - int(bf16_key(np.array([want], np.uint16))[0])) <= 1


# --------------------------------------------------------------------------
# store modes, init, fold, host finish, Optional partials
# --------------------------------------------------------------------------

@pytest.mark.parametrize("n", [100, 50_000, 3_000_000])
def test_store_modes(n):
    x = gen("i64", n, stream=24)
    xd = dev_of("i64", x)
    s = oracle.reduce(x, "i64")
    r = torch.tensor([1000], dtype=torch.int64, device="cuda")
    ak.ak_reduce(xd, dst=r, mode="fold")
    assert r.item() == 1000 + s
    ak.ak_reduce(xd, dst=r, mode="init", init=-7)
    assert r.item() == s - 7
    ak.ak_reduce(xd, dst=r, mode="overwrite")
    assert r.item() == s
    assert ak.ak_reduce(xd, to_host=True, mode="fold", host_old=5) == s + 5
    assert ak.ak_reduce(xd, op="max", to_host=True, init=10**9) == 10**9
    r2 = torch.tensor([10**12], dtype=torch.int64, device="cuda")
    assert ak.ak_reduce(xd, op="max", dst=r2, mode="fold", to_host=True) == 10**12


@pytest.mark.parametrize("n", [1, 33, 20_000, 1_000_003])
@pytest.mark.parametrize("op", ["add", "max", "min", "mul"])
def test_no_neutral_optional_partials(n, op):
    x = gen("f32", n, stream=25, dist="normal") if op != "mul" else np.ones(n, np.float32)
    xd = dev_of("f32", x)
    opts = ak.make_opts(no_neutral=True)
    got = ak.ak_reduce(xd, op=op, to_host=True, opts=opts)
    dev = torch.empty(1, device="cuda")
    ak.ak_reduce(xd, op=op, dst=dev, opts=opts)
    want = oracle.reduce(x, "f32", op=op)
    if op in ("max", "min", "mul"):
        assert got == want and dev.item() == want
    else:
        m = _absmass(x, "f32", "identity")
        assert abs(got - want) <= 2.0**-20 * m and abs(dev.item() - want) <= 2.0**-20 * m


def test_empty_rules():
    e = torch.empty(0, device="cuda")
    assert ak.ak_reduce(e, to_host=True) == 0.0
    assert ak.ak_reduce(e, op="mul", to_host=True) == 1.0
    assert ak.ak_reduce(e, init=2.5, to_host=True) == 2.5
    with pytest.raises(ak.AkError) as ei:
        ak.ak_reduce(e, op="max", to_host=True)
    assert ei.value.status == 4
    with pytest.raises(ak.AkError):
        ak.ak_reduce(e, to_host=True, opts=ak.make_opts(no_neutral=True))
    r = torch.tensor([3.0], device="cuda")
    ak.ak_reduce(e, dst=r, mode="fold")
    assert r.item() == 3.0
    ak.ak_reduce(e, dst=r)
    assert r.item() == 0.0
    m = torch.empty((0, 4), dtype=torch.int32, device="cuda")
    assert ak.ak_reduce(m, op="matmul", elem="mat2", to_host=True) == (1, 0, 0, 1)


def test_max_nan_and_signed_zero():
    x = np.array([-0.0, 0.0, -0.0], dtype=np.float32)
    got = ak.ak_reduce(dev_of("f32", x), op="max", to_host=True)
    assert got == 0.0 and math.copysign(1.0, got) == 1.0
    got = ak.ak_reduce(dev_of("f32", x), op="min", to_host=True)
    assert math.copysign(1.0, got) == -1.0
    x = gen("f32", 300_000, stream=26)
    x[123_457] = np.nan
    assert math.isnan(ak.ak_reduce(dev_of("f32", x), op="max", to_host=True))
    assert math.isnan(ak.ak_reduce(dev_of("f32", x), op="min", to_host=True))


def test_sum_of_single_negative_zero():
    x = np.array([-0.0], dtype=np.float32)
    got = ak.ak_reduce(dev_of("f32", x), to_host=True)
    assert math.copysign(1.0, got) == -1.0


# --------------------------------------------------------------------------
# order-preserving matrix product, workspace reuse
# --------------------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 2, 255, 256, 257, 10_000, 1_000_001])
def test_mat2_product_in_order(n):
    x = synth.mat2_modp(n, stream=27)
    xd = dev_of("mat2", x)
    got = ak.ak_reduce(xd, op="matmul", elem="mat2", to_host=True)
    assert got == tuple(int(v) for v in oracle.reduce(x, "mat2"))
    d = torch.zeros(4, dtype=torch.int32, device="cuda")
    ak.ak_reduce(xd, op="matmul", elem="mat2", dst=d)
    assert tuple(int(v) for v in d.cpu().numpy().view(np.uint32)) == got
    init = synth.mat2_modp(1, stream=28)[0]
    got_i = ak.ak_reduce(xd, op="matmul", elem="mat2", init=init, to_host=True)
    assert got_i == tuple(int(v) for v in oracle.reduce(x, "mat2", init=init))


def test_workspace_reuse_and_target_blocks():
    x = gen("f64", 2_000_000, stream=29)
    xd = dev_of("f64", x)
    size = ak.ak_reduce_workspace_size(x.size, "f64", "f64")
    ws = torch.empty(size, dtype=torch.uint8, device="cuda")
    want = oracle.reduce(x, "f64")
    for tb in (0, 1, 7, 152, 10_000):
        opts = ak.make_opts(target_blocks=tb)
        got = ak.ak_reduce(xd, to_host=True, workspace=ws, opts=opts)
        assert abs(got - want) <= 2.0**-45 * _absmass(x, "f64", "identity")


def test_mat2_reduction_results_are_canonical():
    # a product whose lazily reduced entries land on p (see the scan test of
    # the same name): the stored result is reduced below p, device and host
    p = synth.MODP
    for n in (10_000, 1_000_001):
        x = np.zeros((n, 4), dtype=np.int32)
        x[:, 0] = 1
        x[:, 3] = 1
        x[0::2, 2] = p - 1
        x[1::2, 2] = 1
        xd = dev_of("mat2", x)
        want = tuple(int(v) for v in oracle.reduce(x, "mat2"))
        d = torch.empty(4, dtype=torch.int32, device="cuda")
        ak.ak_reduce(xd, op="matmul", elem="mat2", dst=d)
        assert tuple(int(v) for v in d.cpu().numpy().view(np.uint32)) == want
        assert ak.ak_reduce(xd, op="matmul", elem="mat2", to_host=True) == want
