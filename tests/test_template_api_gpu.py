"""GPU parity of the C++ template API (include/ak.hpp) with operators the C
ABI does not offer, compiled into a caller's own translation unit
(tests/user_op/user_ops.cu) and checked against the oracle.

* Affine maps mod p, v -> a*v + b, composed left to right: a non-commutative
  operator with 8-byte elements, declared with and without an identity (the
  second runs on Optional partials). Reduce, reductions over dimensions,
  inclusive and exclusive scans are bit-exact against the oracle's
  sequential composition (per output slice for the dimensions).
* UserAdd: float addition declared by the caller, which takes the TMA tile
  scan; within 2^-20 * sum |x| of the f64 oracle.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import F32_REL, assert_close_f32, assert_exact

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "user_op", "user_ops.cu")
OUT = os.path.join(ROOT, "tests", "_build", "libuserops.so")
P = oracle.MODP


@pytest.fixture(scope="module")
def U():
    from mapreduce_prefix_scan_gb300 import _abi, build

    lib = build.build()
    _abi.load()  # libak.so first: the user library links against it
    deps = [SRC, os.path.join(ROOT, "include", "ak.hpp")] + [
        os.path.join(ROOT, "mapreduce_prefix_scan_gb300", "csrc", f)
        for f in ("reduce.cuh", "reduce_dims.cuh", "scan.cuh", "ak_internal.h")]
    if not os.path.exists(OUT) or os.path.getmtime(OUT) < max(os.path.getmtime(d) for d in deps + [lib]):
        os.makedirs(os.path.dirname(OUT), exist_ok=True)
        libdir = os.path.dirname(lib)
        cmd = [build._nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "-O2",
               "--expt-relaxed-constexpr", "-Xcompiler", "-fPIC", "-shared", "-cudart", "shared",
               "-I", os.path.join(ROOT, "include"), SRC, "-o", OUT + ".tmp", "-L", libdir, "-lak",
               "-Xlinker", "-rpath", "-Xlinker", libdir]
        r = subprocess.run(cmd, capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
        os.replace(OUT + ".tmp", OUT)
    L = ctypes.CDLL(OUT)
    Pv, I64, I32, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    L.user_affine_ws.argtypes = [I64, I32, I32, ctypes.POINTER(SZ)]
    L.user_affine_reduce.argtypes = [Pv, I64, Pv, Pv, I32, Pv, SZ, Pv]
    L.user_affine_scan.argtypes = [Pv, Pv, I64, Pv, I32, I32, Pv, SZ, Pv]
    PI64 = ctypes.POINTER(I64)
    L.user_affine_dims_ws.argtypes = [I32, PI64, PI64, ctypes.c_uint32, I32, ctypes.POINTER(SZ)]
    L.user_affine_dims.argtypes = [Pv, I32, PI64, PI64, ctypes.c_uint32, Pv, Pv, I32, Pv, SZ, Pv]
    L.user_add_ws.argtypes = [I64, I32, ctypes.POINTER(SZ)]
    L.user_add_reduce.argtypes = [Pv, I64, Pv, Pv, SZ, Pv]
    L.user_add_scan.argtypes = [Pv, Pv, I64, I32, Pv, SZ, Pv]
    return L


def _affine(n, stream):
    a = synth.uniform_int(n, 0, P - 1, np.int64, stream=stream)
    b = synth.uniform_int(n, 0, P - 1, np.int64, stream=stream + 1000)
    return np.stack([a, b], axis=1).astype(np.uint32)


def _ws(nbytes):
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device="cuda")


def _stream():
    return torch.cuda.current_stream().cuda_stream


@pytest.mark.parametrize("n", [1, 5, 1000, 16385, 1_000_003])
@pytest.mark.parametrize("no_id", [0, 1])
@pytest.mark.parametrize("with_init", [False, True])
def test_affine_reduce(U, n, no_id, with_init):
    x = _affine(n, 130)
    xd = torch.from_numpy(x.view(np.int32)).cuda()
    init = np.array([3, 5], np.uint32) if with_init else None
    b = ctypes.c_size_t()
    assert U.user_affine_ws(n, 0, no_id, ctypes.byref(b)) == 0
    ws = _ws(b.value)
    out = torch.empty(2, dtype=torch.int32, device="cuda")
    st = U.user_affine_reduce(xd.data_ptr(), n, out.data_ptr(), None if init is None else init.ctypes.data, no_id,
                              ws.data_ptr(), ws.numel(), _stream())
    assert st == 0
    assert list(out.cpu().numpy().view(np.uint32)) == list(oracle.reduce_affine(x, init=init))


@pytest.mark.parametrize("n", [1, 700, 4096, 4097, 3_000_005])
@pytest.mark.parametrize("no_id", [0, 1])
@pytest.mark.parametrize("mode", ["inclusive", "inclusive_init", "exclusive_init"])
def test_affine_scan(U, n, no_id, mode):
    x = _affine(n, 131)
    xd = torch.from_numpy(x.view(np.int32)).cuda()
    y = torch.empty_like(xd)
    init = np.array([7, 11], np.uint32) if mode != "inclusive" else None
    excl = mode.startswith("exclusive")
    b = ctypes.c_size_t()
    assert U.user_affine_ws(n, 1, no_id, ctypes.byref(b)) == 0
    ws = _ws(b.value)
    st = U.user_affine_scan(xd.data_ptr(), y.data_ptr(), n, None if init is None else init.ctypes.data, int(excl),
                            no_id, ws.data_ptr(), ws.numel(), _stream())
    assert st == 0
    want = oracle.scan_affine(x, init=init, exclusive=excl)
    assert_exact(y.cpu().numpy().view(np.uint32).reshape(-1, 2), want)


# (column-major shape, reduced dims): strided middle / leading / trailing
# dimensions, several reduced blocks, everything, and a strided view
DIMS_CASES = [((300, 40, 3), (1,)), ((64, 2048), (1,)), ((2048, 64), (0,)), ((17, 5, 33, 4), (0, 2)),
              ((1000, 33), (0, 1)), ((3, 70000), (1,)), ((9, 11, 7), (0, 1, 2))]


@pytest.mark.parametrize("shape,dims", DIMS_CASES)
@pytest.mark.parametrize("no_id", [0, 1])
@pytest.mark.parametrize("with_init", [False, True])
def test_affine_reduce_dims(U, shape, dims, no_id, with_init):
    n = int(np.prod(shape))
    x = _affine(n, 134)
    xd = torch.from_numpy(x.view(np.int32)).cuda()
    init = np.array([13, 17], np.uint32) if with_init else None
    mask = sum(1 << d for d in dims)
    shp = (ctypes.c_int64 * len(shape))(*shape)
    b = ctypes.c_size_t()
    assert U.user_affine_dims_ws(len(shape), shp, None, mask, no_id, ctypes.byref(b)) == 0
    ws = _ws(b.value)
    kept = [e for d, e in enumerate(shape) if d not in dims]
    nout = int(np.prod(kept)) if kept else 1
    out = torch.empty(2 * nout, dtype=torch.int32, device="cuda")
    st = U.user_affine_dims(xd.data_ptr(), len(shape), shp, None, mask, out.data_ptr(),
                            None if init is None else init.ctypes.data, no_id, ws.data_ptr(), ws.numel(), _stream())
    assert st == 0
    got = out.cpu().numpy().view(np.uint32).reshape(-1, 2)
    # the oracle's fold of each output's slice, reduced elements in column-major order
    arr = x.reshape(tuple(reversed(shape)) + (2,))            # numpy axis a = dim ndim-1-a
    red_axes = sorted(len(shape) - 1 - d for d in dims)      # highest dimension slowest
    kept_axes = [a for a in range(len(shape)) if a not in red_axes]
    moved = np.transpose(arr, kept_axes + red_axes + [len(shape)])
    moved = moved.reshape(nout, -1, 2)                         # outputs in column-major order of the kept dims
    for o in range(0, nout, max(1, nout // 64)):              # a sample of the outputs
        assert list(got[o]) == list(oracle.reduce_affine(np.ascontiguousarray(moved[o]), init=init)), o
    assert got.shape[0] == nout


def test_affine_reduce_dims_strided_view(U):
    # a column-major 60 x 50 x 4 array viewed with every other column: shape
    # (60, 25, 4), strides (1, 120, 3000); reduce over dimension 1
    base = _affine(60 * 50 * 4, 135)
    xd = torch.from_numpy(base.view(np.int32)).cuda()
    shape, strides = (60, 25, 4), (1, 120, 3000)
    shp = (ctypes.c_int64 * 3)(*shape)
    std = (ctypes.c_int64 * 3)(*strides)
    b = ctypes.c_size_t()
    assert U.user_affine_dims_ws(3, shp, std, 2, 0, ctypes.byref(b)) == 0
    ws = _ws(b.value)
    out = torch.empty(2 * 60 * 4, dtype=torch.int32, device="cuda")
    assert U.user_affine_dims(xd.data_ptr(), 3, shp, std, 2, out.data_ptr(), None, 0, ws.data_ptr(), ws.numel(),
                              _stream()) == 0
    got = out.cpu().numpy().view(np.uint32).reshape(4, 60, 2)
    full = base.reshape(4, 50, 60, 2)
    for k in range(4):
        for i in (0, 7, 59):
            assert list(got[k, i]) == list(oracle.reduce_affine(np.ascontiguousarray(full[k, ::2, i])))


def test_affine_exclusive_without_init(U):
    n = 200_001
    x = _affine(n, 132)
    xd = torch.from_numpy(x.view(np.int32)).cuda()
    y = torch.empty_like(xd)
    b = ctypes.c_size_t()
    U.user_affine_ws(n, 1, 1, ctypes.byref(b))
    ws = _ws(b.value)
    # with an identity, (1, 0) stands for init
    assert U.user_affine_scan(xd.data_ptr(), y.data_ptr(), n, None, 1, 0, ws.data_ptr(), ws.numel(), _stream()) == 0
    want = oracle.scan_affine(x, init=np.array([1, 0], np.uint32), exclusive=True)
    assert_exact(y.cpu().numpy().view(np.uint32).reshape(-1, 2), want)
    # without one the first output has no value
    assert U.user_affine_scan(xd.data_ptr(), y.data_ptr(), n, None, 1, 1, ws.data_ptr(), ws.numel(), _stream()) == 4


@pytest.mark.parametrize("n", [1000, 10**7 + 7])
def test_user_add_takes_the_tma_scan(U, n):
    x = synth.normal_f32(n, stream=133)
    xd = torch.from_numpy(x).cuda()
    y = torch.empty_like(xd)
    b = ctypes.c_size_t()
    assert U.user_add_ws(n, 1, ctypes.byref(b)) == 0
    ws = _ws(b.value)
    assert U.user_add_scan(xd.data_ptr(), y.data_ptr(), n, 0, ws.data_ptr(), ws.numel(), _stream()) == 0
    x64 = x.astype(np.float64)
    assert_close_f32(y.cpu().numpy(), oracle.scan(x, "f32"), np.cumsum(np.abs(x64)))
    assert U.user_add_scan(xd.data_ptr(), y.data_ptr(), n, 1, ws.data_ptr(), ws.numel(), _stream()) == 0
    assert_close_f32(y.cpu().numpy(), oracle.scan(x, "f32", exclusive=True, init=0.0),
                     np.concatenate([[0.0], np.cumsum(np.abs(x64))[:-1]]))
    assert U.user_add_ws(n, 0, ctypes.byref(b)) == 0
    ws = _ws(b.value)
    r = torch.empty(1, dtype=torch.float32, device="cuda")
    assert U.user_add_reduce(xd.data_ptr(), n, r.data_ptr(), ws.data_ptr(), ws.numel(), _stream()) == 0
    assert abs(float(r.item()) - oracle.reduce(x, "f32")) <= F32_REL * float(np.abs(x64).sum())
