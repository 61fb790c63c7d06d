"""GPU parity of ak_reduce_dims against the oracle.

The strided workloads at full size (strided-reduction PR #176, section
"Timings": 3072x2048 bf16, 768x1024x8 bf16 and f32, 64x4096x32 f32,
8192x8192 f32, all sum(x; dims=2) in column-major order), every kernel
shape forced on ragged shapes, integer and matrix operators bit-exact,
contiguous (dims=1) and general masks, store modes and empty reductions.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mapreduce_prefix_scan_gb300 as ak
import oracle
import synth
from helpers import assert_bf16_within_1ulp, assert_close_f32, assert_exact, colmajor_mass, dev_of, gen

pytestmark = pytest.mark.gpu


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _run(x, kind, shape, dims, **kw):
    xd = dev_of(kind, x).reshape(tuple(reversed(shape)) + ((4,) if kind == "mat2" else ()))
    return ak.ak_reduce_dims(xd, dims, elem="mat2" if kind == "mat2" else None, **kw)


def _check_float(x, kind, shape, dims, out, f="identity", init=None):
    want = oracle.reduce_dims(x, kind, shape, dims, map=f, init=init)
    x64 = synth.bf16_bits_to_f32(x).astype(np.float64) if kind == "bf16" else x.astype(np.float64)
    if f == "abs2":
        x64 = x64 * x64
    mass = colmajor_mass(x64, shape, dims) + (abs(init) if init is not None else 0.0)
    if out.dtype == torch.bfloat16:
        assert_bf16_within_1ulp(_bits(out), want)
    else:
        assert_close_f32(out.cpu().numpy(), want, mass)


# --------------------------------------------------------------------------
# the strided workloads at full size
# --------------------------------------------------------------------------

@pytest.mark.parametrize("cluster", [False, True])
def test_3072x2048_bf16_dims2(cluster):
    shape = (3072, 2048)
    x = synth.normal_bf16_bits(3072 * 2048, seed=0, stream=40)
    out = _run(x, "bf16", shape, [1], opts=ak.make_opts(dims_cluster=cluster))
    assert out.dtype == torch.bfloat16 and out.shape == (1, 3072)
    _check_float(x, "bf16", shape, [1], out)


@pytest.mark.parametrize("kind", ["bf16", "f32"])
def test_768x1024x8_middle_dim(kind):
    shape = (768, 1024, 8)
    x = synth.normal_bf16_bits(768 * 1024 * 8, stream=41) if kind == "bf16" else synth.normal_f32(768 * 1024 * 8, stream=41)
    out = _run(x, kind, shape, [1])
    assert out.shape == (8, 1, 768)
    _check_float(x, kind, shape, [1], out)


def test_64x4096x32_f32_middle_dim():
    shape = (64, 4096, 32)
    x = synth.normal_f32(64 * 4096 * 32, stream=42)
    _check_float(x, "f32", shape, [1], _run(x, "f32", shape, [1]))


def test_8192x8192_f32_dims2():
    shape = (8192, 8192)
    x = synth.normal_f32(8192 * 8192, stream=43)
    _check_float(x, "f32", shape, [1], _run(x, "f32", shape, [1]))


# --------------------------------------------------------------------------
# every shape, ragged extents, misalignment
# --------------------------------------------------------------------------

SHAPES3 = [(1000, 37, 3), (17, 3000, 2), (130, 129, 5), (4100, 65, 1), (5, 70_000, 1), (3, 9, 4000),
           (256, 31, 7), (2, 2, 2)]


@pytest.mark.parametrize("shape", SHAPES3)
@pytest.mark.parametrize("forced", ["auto", "thread", "tiled", "columns", "cluster"])
def test_forced_shapes_f32_and_i64(shape, forced):
    n = int(np.prod(shape))
    opts = ak.make_opts(dims_cluster=True) if forced == "cluster" else ak.make_opts(dims_shape=forced)
    x = gen("f32", n, stream=44, dist="normal")
    _check_float(x, "f32", shape, [1], _run(x, "f32", shape, [1], opts=opts))
    xi = gen("i64", n, stream=45)
    got = _run(xi, "i64", shape, [1], opts=opts)
    assert_exact(got.cpu().numpy(), oracle.reduce_dims(xi, "i64", shape, [1]))
    got = _run(xi, "i64", shape, [1], op="max", opts=opts)
    assert_exact(got.cpu().numpy(), oracle.reduce_dims(xi, "i64", shape, [1], op="max"))


@pytest.mark.parametrize("shape", [(257, 300, 3), (1001, 64, 2), (8, 2048, 1)])
def test_bf16_outputs_ragged(shape):
    n = int(np.prod(shape))
    x = gen("bf16", n, stream=46)
    for forced in ("auto", "thread", "columns", "cluster"):
        opts = ak.make_opts(dims_cluster=True) if forced == "cluster" else ak.make_opts(dims_shape=forced)
        _check_float(x, "bf16", shape, [1], _run(x, "bf16", shape, [1], opts=opts))


def test_misaligned_source_falls_back_to_scalar_rows():
    shape = (513, 700)
    n = 513 * 700
    x = gen("f32", n + 1, stream=47)
    xd = dev_of("f32", x)[1:].reshape(700, 513)
    out = ak.ak_reduce_dims(xd, [1])
    want = oracle.reduce_dims(x[1:], "f32", shape, [1])
    assert_close_f32(out.cpu().numpy(), want, colmajor_mass(x[1:].astype(np.float64), shape, [1]))


@pytest.mark.parametrize("shape", [(40, 600, 3), (7, 50, 9), (300, 2000, 1)])
def test_mat2_dims_in_order(shape):
    n = int(np.prod(shape))
    x = synth.mat2_modp(n, stream=48)
    for forced in ("auto", "thread", "columns", "cluster"):
        opts = ak.make_opts(dims_cluster=True) if forced == "cluster" else ak.make_opts(dims_shape=forced)
        got = _run(x, "mat2", shape, [1], op="matmul", opts=opts)
        assert_exact(got.cpu().numpy().view(np.uint32).reshape(-1, 4),
                     oracle.reduce_dims(x, "mat2", shape, [1]))


@pytest.mark.parametrize("kind,acc,out", [("i32", "i32", "i32"), ("i32", "i64", "i64"), ("f32", "f64", "f64"),
                                          ("f64", "f64", "f64"), ("bf16", "f32", "f32")])
def test_types(kind, acc, out):
    shape = (300, 411, 2)
    n = int(np.prod(shape))
    x = gen(kind, n, stream=49)
    got = _run(x, kind, shape, [1], acc=acc, out=out, f="abs2")
    if kind in ("i32", "i64"):
        want = oracle.reduce_dims(x, kind, shape, [1], map="abs2", acc_bits=32 if acc == "i32" else 64)
        assert_exact(got.cpu().numpy(), want)
    else:
        _check_float(x, kind, shape, [1], got, f="abs2")


# --------------------------------------------------------------------------
# other masks: contiguous (dims=0), general, whole, none
# --------------------------------------------------------------------------

@pytest.mark.parametrize("shape,dims", [((5000, 40), [0]), ((100_003, 3), [0]), ((33, 4, 5), [0, 2]),
                                        ((6, 7, 8, 9), [1, 3]), ((64, 64), [0, 1]), ((9, 10), []),
                                        ((1, 5000, 1), [1]), ((4, 1, 6), [1])])
def test_masks(shape, dims):
    n = int(np.prod(shape))
    x = gen("f32", n, stream=50, dist="normal")
    _check_float(x, "f32", shape, dims, _run(x, "f32", shape, dims))
    xi = gen("i32", n, stream=51)
    assert_exact(_run(xi, "i32", shape, dims).cpu().numpy(), oracle.reduce_dims(xi, "i32", shape, dims))
    xm = synth.mat2_modp(n, stream=52)
    got = _run(xm, "mat2", shape, dims, op="matmul")
    assert_exact(got.cpu().numpy().view(np.uint32).reshape(-1, 4), oracle.reduce_dims(xm, "mat2", shape, dims))


def test_store_modes_and_no_neutral():
    shape = (1000, 300, 2)
    n = int(np.prod(shape))
    x = gen("i64", n, stream=53)
    want = oracle.reduce_dims(x, "i64", shape, [1])
    dst = torch.full((2, 1, 1000), 5, dtype=torch.int64, device="cuda")
    _run(x, "i64", shape, [1], dst=dst, mode="fold")
    assert_exact(dst.cpu().numpy(), want + 5)
    _run(x, "i64", shape, [1], dst=dst, init=-3)
    assert_exact(dst.cpu().numpy(), want - 3)
    got = _run(x, "i64", shape, [1], op="max", opts=ak.make_opts(no_neutral=True))
    assert_exact(got.cpu().numpy(), oracle.reduce_dims(x, "i64", shape, [1], op="max"))


def test_empty_reductions():
    x = torch.empty((0, 5), device="cuda")  # column-major (5, 0): reduce dim 1 (extent 0)
    out = ak.ak_reduce_dims(x, [1])
    assert out.shape == (1, 5) and torch.all(out == 0)
    out = ak.ak_reduce_dims(x, [1], init=2.0)
    assert torch.all(out == 2.0)
    with pytest.raises(ak.AkError):
        ak.ak_reduce_dims(x, [1], op="max")
    out = ak.ak_reduce_dims(torch.empty((3, 0), device="cuda"), [1])  # no outputs
    assert out.numel() == 0


def test_mat2_dims_results_are_canonical():
    p = synth.MODP
    shape = (40, 600, 3)
    n = int(np.prod(shape))
    x = np.zeros((n, 4), dtype=np.int32)
    x[:, 0] = 1
    x[:, 3] = 1
    # along the reduced (middle) dimension the a12 entries alternate p-1, 1
    j = (np.arange(n) // shape[0]) % shape[1]
    x[:, 2] = np.where(j % 2 == 0, p - 1, 1)
    for forced in ("auto", "thread", "columns"):
        got = _run(x, "mat2", shape, [1], op="matmul", opts=ak.make_opts(dims_shape=forced))
        g = got.cpu().numpy().view(np.uint32).reshape(-1, 4)
        assert g.max() < p
        assert_exact(g, oracle.reduce_dims(x, "mat2", shape, [1]))
