"""CPU checks of the C ABI: the library loads, exports every symbol that
include/ak.h declares, and validates arguments before touching a device.
The dims shape selector and the scan workspace plan are pure host logic."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from mapreduce_prefix_scan_gb300 import build
    build.build()
    from mapreduce_prefix_scan_gb300 import _abi
    return _abi.load()


def _declared():
    src = open(os.path.join(ROOT, "include", "ak.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ak_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    from mapreduce_prefix_scan_gb300 import _abi
    names = _declared()
    assert set(names) == set(_abi.EXPORTS)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings_and_sizes(L):
    for s in range(7):
        assert L.ak_status_string(s)
    assert L.ak_status_string(99) == b"unknown status"
    assert [L.ak_dtype_size(t) for t in range(7)] == [4, 8, 2, 4, 8, 16, 1]
    assert L.ak_dtype_size(17) == 0


def test_opts_default(L):
    from mapreduce_prefix_scan_gb300 import _abi
    o = _abi.ak_opts()
    o.no_neutral = 7
    L.ak_opts_default(ctypes.byref(o))
    assert o.no_neutral == 0 and o.dims_shape == 0 and o.debug_skip_publish_tile == -1
    assert ctypes.sizeof(_abi.ak_opts) == 48 and o.exclusive == 0 and o.reserved == 0


def _reduce(L, src=0x1000, n=10, in_t=0, f=0, op=0, acc=0, out=0, init=None, mode=0, dst=0x2000, host=None):
    return L.ak_reduce(src, n, in_t, f, op, acc, out, init, mode, dst, host, 0x4000, 1 << 20, None, None)


def test_reduce_validates_before_device(L):
    from mapreduce_prefix_scan_gb300._abi import AK_ERR_INVALID_ARG as INV, AK_ERR_UNSUPPORTED as UNS
    assert _reduce(L, in_t=9) == INV
    assert _reduce(L, f=5) == INV
    assert _reduce(L, op=8) == INV
    assert _reduce(L, n=-1) == INV
    assert _reduce(L, src=None) == INV
    assert _reduce(L, dst=None, host=None) == INV
    assert _reduce(L, mode=3) == INV
    assert _reduce(L, mode=1, init=None) == INV            # init mode without init
    assert _reduce(L, src=0x1001) == INV                   # misaligned f32 source
    assert _reduce(L, in_t=5, acc=5, out=5, op=0) == UNS    # matrices only multiply
    assert _reduce(L, in_t=0, acc=0, out=0, op=4) == UNS    # matmul needs matrices
    assert _reduce(L, in_t=5, acc=5, out=5, op=4, f=2) == UNS
    assert _reduce(L, in_t=2, acc=2, out=2) == UNS          # bf16 accumulator
    assert _reduce(L, in_t=4, acc=3, out=3) == UNS          # narrowing accumulator


def test_reduce_dims_validates_before_device(L):
    from mapreduce_prefix_scan_gb300._abi import AK_ERR_INVALID_ARG as INV
    sh = (ctypes.c_int64 * 3)(4, 5, 6)
    call = lambda ndim=3, shape=sh, mask=2, mode=0, init=None, strides=None: L.ak_reduce_dims(
        0x1000, ndim, shape, strides, mask, 0, 0, 0, 0, 0, init, mode, 0x2000, 0x4000, 1 << 20, None, None)
    assert call(ndim=0) == INV
    assert call(ndim=9) == INV
    assert call(mask=1 << 3) == INV
    assert call(shape=None) == INV
    assert call(shape=(ctypes.c_int64 * 3)(4, -1, 6)) == INV
    assert call(mode=1) == INV
    assert call(strides=(ctypes.c_int64 * 3)(1, -4, 20)) == INV   # negative strides are refused


def test_accumulate_validates_and_plans_on_host(L):
    from mapreduce_prefix_scan_gb300._abi import AK_ERR_INVALID_ARG as INV, AK_ERR_UNSUPPORTED as UNS
    sh = (ctypes.c_int64 * 2)(4096, 4096)
    acc = lambda dim=0, src=0x1000, dst=0x800000, in_t=0, op=0, a=0, o=0: L.ak_accumulate(
        src, dst, 2, sh, dim, in_t, op, a, o, None, 0x4000, 1 << 20, None, None)
    assert acc(dim=2) == INV
    assert acc(dim=-2) == INV
    assert acc(src=None) == INV
    assert acc(dst=0x1000 + 64) == INV        # partial overlap
    assert acc(in_t=5, a=5, o=5, op=0) == UNS
    from mapreduce_prefix_scan_gb300 import _abi
    for field, bad in (("exclusive", 2), ("exclusive", -1), ("reserved", 1)):
        o = _abi.ak_opts()
        L.ak_opts_default(ctypes.byref(o))
        setattr(o, field, bad)
        assert L.ak_accumulate(0x1000, 0x800000, 2, sh, 0, 0, 0, 0, 0, None, 0x4000, 1 << 20,
                               ctypes.byref(o), None) == INV
    assert L.ak_scan_status(None) == INV
    assert L.ak_scan_status(0x4001) == INV
    b = ctypes.c_size_t()
    # whole-array f64 scan of 1e8: super-tiles of 256 threads x 64 elements,
    # one 32-byte state record each (tag, check word, value)
    n = (ctypes.c_int64 * 1)(10**8)
    assert L.ak_accumulate_workspace_size(1, n, -1, 1, 1, 0, None, ctypes.byref(b)) == 0
    tiles = -(-10**8 // (256 * 64))
    assert b.value >= 256 + tiles * 32
    # columns of 4096 f32 fit one tile each: no tile state needed
    assert L.ak_accumulate_workspace_size(2, sh, 0, 0, 0, 0, None, ctypes.byref(b)) == 0
    assert b.value == 256


def test_dims_selector(L):
    import mapreduce_prefix_scan_gb300 as ak
    # 3072 x 2048 bf16, dims=2 (12.6 MB, latency-bound): 16-byte vectors of 8,
    # 16 threads across a 128-output row segment, 16 row groups of 8 rows, the
    # reduction split 16 ways and the split blocks of an output tile combined
    # in a thread-block cluster: 384 blocks of 32 KB, all resident at once
    shape, tile, groups, split = ak.ak_dims_select(3072, 2048, 1, 2, 8, 152)
    assert shape == "columns" and tile == 128 and groups == 16 and split == 16
    assert (3072 // tile) * split == 384 and 2048 // (split * groups) == 8
    # a larger input: a warp across a 256-output row segment, 8 row groups,
    # split through the workspace and a second pass, >= 1 block per SM
    shape, tile, groups, split = ak.ak_dims_select(3072, 8192, 1, 2, 8, 152)
    assert shape == "columns" and tile == 256 and groups == 8 and split > 1
    assert -(-3072 // tile) * split >= 152
    # middle dim of 64 x 4096 x 32 f32: 16 threads cover the 64 outputs of a run
    shape, tile, groups, split = ak.ak_dims_select(64, 4096, 32, 4, 4, 152)
    assert shape == "columns" and tile == 64 and groups == 16 and split > 1
    # short reductions take one thread per output vector
    assert ak.ak_dims_select(100_000, 16, 1, 4, 4, 152)[0] == "thread"
    # forced shapes are honoured
    assert ak.ak_dims_select(3072, 2048, 1, 2, 8, 152, "tiled")[3] == 1
    assert ak.ak_dims_select(3072, 2048, 1, 2, 8, 152, "thread")[2] == 1
    with pytest.raises(ak.AkError):
        ak.ak_dims_select(0, 1, 1, 4, 4, 152)


def test_missing_library_fails_loudly():
    # no CPU or PyTorch fallback: without libak.so every entry point raises
    import subprocess
    import sys

    code = ("import mapreduce_prefix_scan_gb300._abi as a; a.LIB_PATH = '/nonexistent/libak.so'; "
            "import mapreduce_prefix_scan_gb300 as ak; ak.ak_reduce_workspace_size(100, \"f32\", \"f32\")")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0
    assert "libak.so not built" in r.stderr


def test_findall_validates_and_plans_on_host(L):
    from mapreduce_prefix_scan_gb300._abi import AK_ERR_INVALID_ARG as INV, AK_ERR_UNSUPPORTED as UNS
    cnt = ctypes.c_int64()
    call = lambda src=0x1000, n=100, t=6, idx=0x8000, cd=0x9000, ch=None: L.ak_findall(
        src, n, t, idx, cd, ch, 0x4000, 1 << 20, None, None)
    assert call(n=-1) == INV
    assert call(t=9) == INV
    assert call(cd=None, ch=None) == INV
    assert call(src=None) == INV
    assert call(idx=None) == INV
    assert call(idx=0x8004) == INV          # int64 indices need 8-byte alignment
    assert call(src=0x1002, t=0) == INV     # misaligned f32 source
    assert call(t=2) == UNS                 # bf16
    assert call(t=5) == UNS                 # matrices
    # empty input: count 0 on the host, nothing launched
    assert L.ak_findall(None, 0, 6, None, None, ctypes.byref(cnt), None, 0, None, None) == 0 and cnt.value == 0
    # one 32-byte record per tile of 16 K flags, after the 256-byte header
    b = ctypes.c_size_t()
    assert L.ak_findall_workspace_size(10**8, 6, None, ctypes.byref(b)) == 0
    assert b.value >= 256 + (-(-10**8 // 16384)) * 32 + 8
