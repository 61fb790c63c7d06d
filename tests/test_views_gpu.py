"""GPU parity of reductions over strided views (ak_reduce_dims with strides,
and ak_reduce of a non-contiguous tensor) against the oracle.

Views are described by their strides and reduced in place, nothing is
copied ("Finish whole-array reductions on the device": its tests cover offset
views). Covered: sub-matrix and padded 3-d views (strided / row kernels with
16-byte loads), transposes and stepped slices (the general kernel, one
thread per output or blocks per output with a split), single outputs over a
non-contiguous view, and 2x2 matrices. Tolerances as everywhere: f32 sums
within 2^-20 * sum |x|, bf16 within 1 ulp, integers and products bit-exact.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mapreduce_prefix_scan_gb300 as ak
import oracle
import synth
from helpers import assert_bf16_within_1ulp, assert_close_f32, assert_exact, gen

pytestmark = pytest.mark.gpu


def _view_args(t: torch.Tensor, base: torch.Tensor):
    """Column-major shape / strides of a view and the flat host buffer that
    starts at its first element."""
    shape = list(reversed(t.shape))
    strides = list(reversed(t.stride()))
    off = t.storage_offset() - base.storage_offset()
    return shape, strides, off


def _mass(flat64, shape, strides, dims):
    return oracle.reduce_dims(np.abs(flat64), "f64", shape, dims, strides=strides)


def _check(kind, host_flat, t, base, dims, out):
    shape, strides, off = _view_args(t, base)
    buf = host_flat[off:]
    if kind == "bf16":
        want = oracle.reduce_dims(buf, "bf16", shape, dims, strides=strides)
        assert_bf16_within_1ulp(out.view(torch.int16).cpu().numpy().view(np.uint16), want)
    elif kind == "f32":
        want = oracle.reduce_dims(buf, "f32", shape, dims, strides=strides)
        assert_close_f32(out.cpu().numpy(), want, _mass(buf.astype(np.float64), shape, strides, dims))
    else:
        assert_exact(out.cpu().numpy().ravel(), oracle.reduce_dims(buf, kind, shape, dims, strides=strides))


@pytest.mark.parametrize("kind", ["f32", "bf16", "i64"])
@pytest.mark.parametrize("dims", [[0], [1], [0, 1]])
def test_submatrix_view(kind, dims):
    rows, cols = 4100, 3000
    host = gen(kind, rows * cols, stream=120, dist="normal")
    big = (torch.from_numpy(host.view(np.int16)).view(torch.bfloat16) if kind == "bf16"
           else torch.from_numpy(host)).reshape(rows, cols).cuda()
    v = big[5:4005, 8:2056]              # column-major 2048 x 4000, column stride 3000
    assert not v.is_contiguous()
    out = ak.ak_reduce_dims(v, dims)
    _check(kind, host, v, big, dims, out)


@pytest.mark.parametrize("kind", ["f32", "bf16"])
def test_padded_3d_middle_dim(kind):
    # the 768 x 1024 x 8 workload as a view of rows padded to 800 elements
    host = gen(kind, 8 * 1024 * 800, stream=121, dist="normal")
    big = (torch.from_numpy(host.view(np.int16)).view(torch.bfloat16) if kind == "bf16"
           else torch.from_numpy(host)).reshape(8, 1024, 800).cuda()
    v = big[:, :, :768]
    out = ak.ak_reduce_dims(v, [1])
    _check(kind, host, v, big, [1], out)


@pytest.mark.parametrize("case", ["transpose", "step2", "step3_rows", "permuted3d"])
def test_general_views(case):
    host = synth.normal_f32(600 * 700, stream=122)
    big = torch.from_numpy(host).reshape(600, 700).cuda()
    if case == "transpose":
        v, dims = big.t(), [1]
    elif case == "step2":
        v, dims = big[:, ::2], [1]
    elif case == "step3_rows":
        v, dims = big[::3, 1:], [0]
    else:
        v, dims = big.reshape(6, 100, 700).permute(2, 0, 1), [0, 2]
    out = ak.ak_reduce_dims(v, dims)
    _check("f32", host, v, big, dims, out)
    # init, max and an integer view through the same paths
    hi = synth.uniform_int(600 * 700, -1000, 1000, np.int64, stream=123)
    bi = torch.from_numpy(hi).reshape(600, 700).cuda()
    vi = {"transpose": bi.t(), "step2": bi[:, ::2], "step3_rows": bi[::3, 1:],
          "permuted3d": bi.reshape(6, 100, 700).permute(2, 0, 1)}[case]
    shape, strides, off = _view_args(vi, bi)
    out = ak.ak_reduce_dims(vi, dims, init=11)
    assert_exact(out.cpu().numpy().ravel(), oracle.reduce_dims(hi[off:], "i64", shape, dims, init=11, strides=strides))
    out = ak.ak_reduce_dims(vi, dims, op="max")
    assert_exact(out.cpu().numpy().ravel(), oracle.reduce_dims(hi[off:], "i64", shape, dims, op="max",
                                                               strides=strides))


def test_single_output_over_strided_views():
    # whole-array reductions of non-contiguous views: general blocks with a split
    host = synth.uniform_f32_pm1(3 * 10**6, stream=124)
    x = torch.from_numpy(host).cuda()
    got = ak.ak_reduce(x[::3], to_host=True)
    want = oracle.reduce(host[::3].copy(), "f32")
    assert abs(got - want) <= 2.0**-20 * float(np.abs(host[::3].astype(np.float64)).sum())
    hi = synth.uniform_int(2000 * 1500, -(2**20), 2**20, np.int64, stream=125)
    m = torch.from_numpy(hi).reshape(2000, 1500).cuda()[10:1990, 3:1400]
    assert ak.ak_reduce(m, to_host=True) == int(hi.reshape(2000, 1500)[10:1990, 3:1400].sum())
    assert ak.ak_reduce(m, op="max", to_host=True) == int(hi.reshape(2000, 1500)[10:1990, 3:1400].max())


def test_mat2_view_keeps_order():
    host = synth.mat2_modp(300 * 40, stream=126)
    big = torch.from_numpy(host.view(np.int32)).reshape(300, 40, 4).cuda()
    v = big[:, 5:35]                       # column-major 30 x 300 matrices, column stride 40
    out = ak.ak_reduce_dims(v, [1], op="matmul", elem="mat2")
    shape, strides = [30, 300], [1, 40]
    want = oracle.reduce_dims(host[5:], "mat2", shape, [1], strides=strides)
    assert_exact(out.cpu().numpy().view(np.uint32).reshape(-1, 4), want)
    out = ak.ak_reduce_dims(big.transpose(0, 1), [0], op="matmul", elem="mat2")  # 300 x 40, stride (40, 1)
    want = oracle.reduce_dims(host, "mat2", [300, 40], [0], strides=[40, 1])
    assert_exact(out.cpu().numpy().view(np.uint32).reshape(-1, 4), want)
