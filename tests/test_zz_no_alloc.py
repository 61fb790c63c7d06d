"""ak_reduce_noalloc: the reduction for callers that cannot allocate.

Some callers must not allocate device memory when they reduce -- a
real-time loop that cannot afford cudaMalloc's implicit synchronisation, a
process whose device memory another allocator has already reserved, code
with a fixed memory budget. ak_reduce_noalloc serves them with its scratch
in a fixed array inside the library. This test calls it through the C ABI
(ctypes, plain pointers, no workspace argument) and checks that two calls
in a row give the same results as ak_reduce, within the tolerances of the
other reduce tests (bit-exact for integers, max and the matrix product;
2^-20 * sum |f(x)| for f32 sums). It runs last (file name) and needs nothing
from the other test files, so it passes alone in a fresh process too.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _setup():
    from mapreduce_prefix_scan_gb300 import build

    build.build()
    from mapreduce_prefix_scan_gb300 import _abi

    return _abi, _abi.load()


def _reduce_ref(L, _abi, x, n, kind, f, op, out_t, init=None):
    """The existing entry point, with a caller-allocated workspace."""
    D = _abi.DTYPES
    size = ctypes.c_size_t()
    assert L.ak_reduce_workspace_size(n, D[kind], D[kind], None, ctypes.byref(size)) == 0
    ws = torch.empty(size.value, dtype=torch.uint8, device="cuda")
    r = torch.empty(4 if kind == "mat2" else 1, dtype=out_t, device="cuda")
    st = L.ak_reduce(x.data_ptr(), n, D[kind], _abi.MAPS[f], _abi.OPS[op], D[kind], D[kind], init,
                     _abi.STORES["init" if init is not None else "overwrite"], r.data_ptr(), None, ws.data_ptr(),
                     size.value, None, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    return r


def _reduce_noalloc(L, _abi, x, n, kind, f, op, out_t, init=None):
    D = _abi.DTYPES
    r = torch.empty(4 if kind == "mat2" else 1, dtype=out_t, device="cuda")
    st = L.ak_reduce_noalloc(x.data_ptr(), n, D[kind], _abi.MAPS[f], _abi.OPS[op], D[kind], D[kind], init,
                             _abi.STORES["init" if init is not None else "overwrite"], r.data_ptr(), None, None,
                             torch.cuda.current_stream().cuda_stream)
    assert st == 0, L.ak_status_string(st)
    return r


@pytest.mark.parametrize("case", ["f32_abs2_sum", "i64_max", "i32_sum_small", "mat2_product"])
def test_noalloc_matches_ak_reduce_twice(case):
    _abi, L = _setup()
    rng = np.random.default_rng(7)
    init = None
    if case == "f32_abs2_sum":
        n, kind, f, op, out_t = 3_000_001, "f32", "abs2", "add", torch.float32
        host = rng.uniform(-1, 1, n).astype(np.float32)
    elif case == "i64_max":
        n, kind, f, op, out_t = 5_000_000, "i64", "identity", "max", torch.int64
        host = rng.integers(-(2**40), 2**40, n, dtype=np.int64)
    elif case == "i32_sum_small":
        n, kind, f, op, out_t = 1000, "i32", "identity", "add", torch.int32
        host = rng.integers(-1000, 1001, n, dtype=np.int32)
        init = ctypes.create_string_buffer(np.array([17], np.int32).tobytes(), 16)
    else:
        n, kind, f, op, out_t = 200_000, "mat2", "identity", "matmul", torch.int32
        host = rng.integers(0, 2**31 - 1, (n, 4), dtype=np.int64).astype(np.int32)
    x = torch.from_numpy(host).cuda()
    want = _reduce_ref(L, _abi, x, n, kind, f, op, out_t, init).cpu().numpy()
    for _ in range(2):  # two calls in a row share the fixed scratch
        got = _reduce_noalloc(L, _abi, x, n, kind, f, op, out_t, init).cpu().numpy()
        if kind == "f32":
            tol = 2.0**-20 * float(np.sum(host.astype(np.float64) ** 2))
            assert abs(float(got[0]) - float(want[0])) <= tol
        else:
            assert np.array_equal(got, want)


def test_noalloc_host_result_and_empty():
    _abi, L = _setup()
    D = _abi.DTYPES
    host = np.arange(1, 100_001, dtype=np.int64)
    x = torch.from_numpy(host).cuda()
    out = ctypes.c_int64(0)
    s = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        st = L.ak_reduce_noalloc(x.data_ptr(), host.size, D["i64"], 0, 0, D["i64"], D["i64"], None, 0, None,
                                 ctypes.byref(out), None, s)
        assert st == 0 and out.value == 100_000 * 100_001 // 2
    st = L.ak_reduce_noalloc(None, 0, D["i64"], 0, 2, D["i64"], D["i64"], None, 0, None, ctypes.byref(out), None, s)
    assert st == _abi.AK_ERR_EMPTY_NO_INIT

