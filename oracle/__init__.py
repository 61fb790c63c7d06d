"""Python view of the sequential CPU oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, ``__graft_entry__.smoke()``
and the bench's CPU-baseline / reference arm, never by the library. It shares
no code with the CUDA path.

Arrays are passed as flat numpy buffers holding a column-major array of the
given shape (the memory of a contiguous row-major torch tensor of the
reversed shape). Element kinds: 'f32', 'f64', 'bf16' (uint16 bit patterns),
'i32', 'i64', 'mat2' (four uint32 entries per element, column-major
a11, a21, a12, a22), 'u8' (Bool flags, findall only). Ops: 'add', 'mul', 'max', 'min', and 'matmul' for mat2.
Maps: 'identity', 'abs', 'abs2'.

Results: float kinds -> f64 values; integer kinds -> int64 values wrapped to
the accumulator width; mat2 -> uint32 entries. A reduction with no element
and no init has no value and returns None.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_KIND = {"f32": 0, "f64": 1, "bf16": 2, "i32": 3, "i64": 4, "mat2": 5, "u8": 6}
_MAP2 = {"mul": 0, "sqdiff": 1, "absdiff": 2}
_MAP = {"identity": 0, "abs": 1, "abs2": 2}
_OP = {"add": 0, "mul": 1, "max": 2, "min": 3, "matmul": 4}
_NP = {"f32": np.float32, "f64": np.float64, "bf16": np.uint16, "i32": np.int32,
       "i64": np.int64, "mat2": np.uint32, "u8": np.uint8}
MODP = 2147483647

_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P, I64, I32, U32, D = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint32,
                               ctypes.c_double)
        PI64 = ctypes.POINTER(ctypes.c_int64)
        L.orc_bf16_rne.argtypes = [D]
        L.orc_bf16_rne.restype = ctypes.c_uint16
        L.orc_fmax.argtypes = [D, D]
        L.orc_fmax.restype = D
        L.orc_fmin.argtypes = [D, D]
        L.orc_fmin.restype = D
        L.orc_mat2_mul.argtypes = [P, P, P]
        L.orc_reduce_float.argtypes = [P, I64, I32, I32, I32, I32, D, P]
        L.orc_reduce_int.argtypes = [P, I64, I32, I32, I32, I32, I32, I64, P]
        L.orc_reduce_mat2.argtypes = [P, I64, P, P]
        L.orc_reduce_dims_float.argtypes = [P, I32, PI64, U32, I32, I32, I32, I32, D, P]
        L.orc_reduce_dims_int.argtypes = [P, I32, PI64, U32, I32, I32, I32, I32, I32, I64, P]
        L.orc_reduce_dims_mat2.argtypes = [P, I32, PI64, U32, P, P]
        L.orc_scan_float.argtypes = [P, I32, PI64, I32, I32, I32, I32, D, P]
        L.orc_scan_int.argtypes = [P, I32, PI64, I32, I32, I32, I32, I32, I64, P]
        L.orc_scan_mat2.argtypes = [P, I32, PI64, I32, P, P]
        L.orc_reduce_dims_float_s.argtypes = [P, I32, PI64, PI64, U32, I32, I32, I32, I32, D, P]
        L.orc_reduce_dims_int_s.argtypes = [P, I32, PI64, PI64, U32, I32, I32, I32, I32, I32, I64, P]
        L.orc_reduce_dims_mat2_s.argtypes = [P, I32, PI64, PI64, U32, P, P]
        L.orc_scan_excl_float.argtypes = [P, I32, PI64, I32, I32, I32, D, P]
        L.orc_scan_excl_int.argtypes = [P, I32, PI64, I32, I32, I32, I32, I64, P]
        L.orc_scan_excl_mat2.argtypes = [P, I32, PI64, I32, P, P]
        L.orc_findall.argtypes = [P, I64, I32, P]
        L.orc_findall.restype = I64
        L.orc_reduce2_float.argtypes = [P, P, I64, I32, I32, I32, I32, D, P]
        L.orc_reduce2_int.argtypes = [P, P, I64, I32, I32, I32, I32, I32, I64, P]
        L.orc_affine_compose.argtypes = [P, P, P]
        L.orc_affine_compose.restype = None
        L.orc_scan_affine.argtypes = [P, I64, P, I32, P]
        L.orc_reduce_affine.argtypes = [P, I64, P, P]
        for name in ("orc_reduce_float", "orc_reduce_int", "orc_reduce_mat2", "orc_reduce_dims_float",
                     "orc_reduce_dims_int", "orc_reduce_dims_mat2", "orc_scan_float", "orc_scan_int",
                     "orc_scan_mat2", "orc_reduce_dims_float_s", "orc_reduce_dims_int_s",
                     "orc_reduce_dims_mat2_s", "orc_scan_excl_float", "orc_scan_excl_int",
                     "orc_scan_excl_mat2", "orc_reduce2_float", "orc_reduce2_int", "orc_scan_affine",
                     "orc_reduce_affine"):
            getattr(L, name).restype = I32
        _lib = L
    return _lib


def _buf(x: np.ndarray, kind: str) -> np.ndarray:
    a = np.ascontiguousarray(x)
    want = _NP[kind]
    if kind == "mat2" and a.dtype == np.int32:
        a = a.view(np.uint32)
    if kind == "bf16" and a.dtype == np.int16:
        a = a.view(np.uint16)
    if a.dtype != want:
        raise TypeError(f"oracle: {kind} input must be {np.dtype(want)}, got {a.dtype}")
    return a


def _shape(shape) -> ctypes.Array:
    return (ctypes.c_int64 * len(shape))(*[int(s) for s in shape])


def _acc_bits(kind: str, acc_bits):
    if acc_bits is None:
        return 32 if kind == "i32" else 64
    return int(acc_bits)


def _check(rc: int):
    if rc < 0:
        raise ValueError("oracle: bad argument")
    return rc


def bf16_rne(v: float) -> int:
    """f64 -> bf16 bit pattern, one correct rounding (nearest, ties to even)."""
    return int(lib().orc_bf16_rne(float(v)))


def bf16_rne_array(v: np.ndarray) -> np.ndarray:
    f = lib().orc_bf16_rne
    return np.array([f(float(t)) for t in np.ravel(v)], dtype=np.uint16).reshape(np.shape(v))


def fmax(a: float, b: float) -> float:
    return lib().orc_fmax(a, b)


def fmin(a: float, b: float) -> float:
    return lib().orc_fmin(a, b)


def mat2_mul(a, b) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.uint32)
    b = np.ascontiguousarray(b, dtype=np.uint32)
    c = np.zeros(4, dtype=np.uint32)
    lib().orc_mat2_mul(a.ctypes.data, b.ctypes.data, c.ctypes.data)
    return c


def reduce(x: np.ndarray, kind: str, op: str = "add", map: str = "identity", init=None,
           acc_bits=None):
    """Whole-array left fold ``op(init, f(x_1), ..., f(x_n))``."""
    L = lib()
    a = _buf(x, kind)
    if kind == "mat2":
        n = a.size // 4
        out = np.zeros(4, dtype=np.uint32)
        ini = None if init is None else np.ascontiguousarray(init, dtype=np.uint32)
        rc = _check(L.orc_reduce_mat2(a.ctypes.data, n, None if ini is None else ini.ctypes.data,
                                      out.ctypes.data))
        return None if rc == 1 else out
    if kind in ("f32", "f64", "bf16"):
        out = ctypes.c_double()
        rc = _check(L.orc_reduce_float(a.ctypes.data, a.size, _KIND[kind], _MAP[map], _OP[op],
                                       init is not None, 0.0 if init is None else float(init),
                                       ctypes.byref(out)))
        return None if rc == 1 else out.value
    out = ctypes.c_int64()
    rc = _check(L.orc_reduce_int(a.ctypes.data, a.size, _KIND[kind], _acc_bits(kind, acc_bits),
                                 _MAP[map], _OP[op], init is not None,
                                 0 if init is None else int(init), ctypes.byref(out)))
    return None if rc == 1 else out.value


def reduce_dims(x: np.ndarray, kind: str, shape, dims, op: str = "add", map: str = "identity",
                init=None, acc_bits=None, strides=None):
    """Fold over the 0-based column-major dimensions ``dims``; returns a flat
    column-major output of the kept extents (reduced extents become 1).
    ``strides`` (elements per dimension) reads ``x`` as a strided view of its
    flat buffer instead of the dense column-major layout."""
    L = lib()
    a = _buf(x, kind)
    st = None if strides is None else _shape(strides)
    mask = 0
    for d in dims:
        mask |= 1 << int(d)
    nout = 1
    for d, s in enumerate(shape):
        if not (mask >> d) & 1:
            nout *= int(s)
    sh = _shape(shape)
    if kind == "mat2":
        out = np.zeros((nout, 4), dtype=np.uint32)
        ini = None if init is None else np.ascontiguousarray(init, dtype=np.uint32)
        rc = _check(L.orc_reduce_dims_mat2_s(a.ctypes.data, len(shape), sh, st, mask,
                                             None if ini is None else ini.ctypes.data, out.ctypes.data))
    elif kind in ("f32", "f64", "bf16"):
        out = np.zeros(nout, dtype=np.float64)
        rc = _check(L.orc_reduce_dims_float_s(a.ctypes.data, len(shape), sh, st, mask, _KIND[kind],
                                              _MAP[map], _OP[op], init is not None,
                                              0.0 if init is None else float(init), out.ctypes.data))
    else:
        out = np.zeros(nout, dtype=np.int64)
        rc = _check(L.orc_reduce_dims_int_s(a.ctypes.data, len(shape), sh, st, mask, _KIND[kind],
                                            _acc_bits(kind, acc_bits), _MAP[map], _OP[op],
                                            init is not None, 0 if init is None else int(init),
                                            out.ctypes.data))
    return None if rc == 1 else out


def scan(x: np.ndarray, kind: str, shape=None, dim: int = -1, op: str = "add", init=None,
         acc_bits=None, exclusive: bool = False):
    """Inclusive scan, whole array (dim = -1) or along 0-based column-major
    dimension ``dim``; returns a flat array in the input's layout. With
    ``exclusive`` (init required) element i holds the fold of init and the
    elements before it."""
    if exclusive:
        return _scan_excl(x, kind, shape, dim, op, init, acc_bits)
    L = lib()
    a = _buf(x, kind)
    if shape is None:
        shape = (a.size // 4,) if kind == "mat2" else (a.size,)
    sh = _shape(shape)
    n = 1
    for s in shape:
        n *= int(s)
    if kind == "mat2":
        y = np.zeros((n, 4), dtype=np.uint32)
        ini = None if init is None else np.ascontiguousarray(init, dtype=np.uint32)
        _check(L.orc_scan_mat2(a.ctypes.data, len(shape), sh, dim,
                               None if ini is None else ini.ctypes.data, y.ctypes.data))
    elif kind in ("f32", "f64", "bf16"):
        y = np.zeros(n, dtype=np.float64)
        _check(L.orc_scan_float(a.ctypes.data, len(shape), sh, dim, _KIND[kind], _OP[op],
                                init is not None, 0.0 if init is None else float(init),
                                y.ctypes.data))
    else:
        y = np.zeros(n, dtype=np.int64)
        _check(L.orc_scan_int(a.ctypes.data, len(shape), sh, dim, _KIND[kind],
                              _acc_bits(kind, acc_bits), _OP[op], init is not None,
                              0 if init is None else int(init), y.ctypes.data))
    return y


def _scan_excl(x, kind, shape, dim, op, init, acc_bits):
    if init is None:
        raise ValueError("oracle: an exclusive scan needs init")
    L = lib()
    a = _buf(x, kind)
    if shape is None:
        shape = (a.size // 4,) if kind == "mat2" else (a.size,)
    sh = _shape(shape)
    n = 1
    for s in shape:
        n *= int(s)
    if kind == "mat2":
        y = np.zeros((n, 4), dtype=np.uint32)
        ini = np.ascontiguousarray(init, dtype=np.uint32)
        _check(L.orc_scan_excl_mat2(a.ctypes.data, len(shape), sh, dim, ini.ctypes.data, y.ctypes.data))
    elif kind in ("f32", "f64", "bf16"):
        y = np.zeros(n, dtype=np.float64)
        _check(L.orc_scan_excl_float(a.ctypes.data, len(shape), sh, dim, _KIND[kind], _OP[op], float(init),
                                     y.ctypes.data))
    else:
        y = np.zeros(n, dtype=np.int64)
        _check(L.orc_scan_excl_int(a.ctypes.data, len(shape), sh, dim, _KIND[kind], _acc_bits(kind, acc_bits),
                                   _OP[op], int(init), y.ctypes.data))
    return y


def findall(x: np.ndarray, kind: str) -> np.ndarray:
    """0-based indices of the nonzero elements of a flat array, increasing
    ('u8' Bool flags, 'i32', 'i64', 'f32', 'f64')."""
    a = _buf(x, kind)
    idx = np.zeros(max(a.size, 1), dtype=np.int64)
    c = lib().orc_findall(a.ctypes.data, a.size, _KIND[kind], idx.ctypes.data)
    if c < 0:
        raise ValueError("oracle: bad argument")
    return idx[:c].copy()


def reduce2(x: np.ndarray, y: np.ndarray, kind: str, map2: str = "mul", op: str = "add", init=None,
            acc_bits=None):
    """Left fold ``op(init, f(x_1, y_1), ..., f(x_n, y_n))`` of two sources of
    the same kind and length; f: 'mul' (x*y), 'sqdiff' ((x-y)^2), 'absdiff'
    (|x-y|)."""
    L = lib()
    a = _buf(x, kind)
    b = _buf(y, kind)
    if a.size != b.size:
        raise ValueError("oracle: sources of different lengths")
    if kind in ("f32", "f64", "bf16"):
        out = ctypes.c_double()
        rc = _check(L.orc_reduce2_float(a.ctypes.data, b.ctypes.data, a.size, _KIND[kind], _MAP2[map2], _OP[op],
                                        init is not None, 0.0 if init is None else float(init), ctypes.byref(out)))
        return None if rc == 1 else out.value
    out = ctypes.c_int64()
    rc = _check(L.orc_reduce2_int(a.ctypes.data, b.ctypes.data, a.size, _KIND[kind], _acc_bits(kind, acc_bits),
                                  _MAP2[map2], _OP[op], init is not None, 0 if init is None else int(init),
                                  ctypes.byref(out)))
    return None if rc == 1 else out.value


def affine_compose(f, g) -> np.ndarray:
    """op(f, g) of two affine maps mod p, (a, b) = v -> a*v + b: f first, then g."""
    f = np.ascontiguousarray(f, dtype=np.uint32)
    g = np.ascontiguousarray(g, dtype=np.uint32)
    out = np.zeros(2, dtype=np.uint32)
    lib().orc_affine_compose(f.ctypes.data, g.ctypes.data, out.ctypes.data)
    return out


def scan_affine(x: np.ndarray, init=None, exclusive: bool = False) -> np.ndarray:
    """Inclusive (or exclusive, init required) scan of affine maps mod p; x is
    (n, 2) uint32."""
    a = np.ascontiguousarray(x, dtype=np.uint32).reshape(-1, 2)
    y = np.zeros_like(a)
    ini = None if init is None else np.ascontiguousarray(init, dtype=np.uint32)
    _check(lib().orc_scan_affine(a.ctypes.data, a.shape[0], None if ini is None else ini.ctypes.data,
                                 int(bool(exclusive)), y.ctypes.data))
    return y


def reduce_affine(x: np.ndarray, init=None):
    a = np.ascontiguousarray(x, dtype=np.uint32).reshape(-1, 2)
    out = np.zeros(2, dtype=np.uint32)
    ini = None if init is None else np.ascontiguousarray(init, dtype=np.uint32)
    rc = _check(lib().orc_reduce_affine(a.ctypes.data, a.shape[0], None if ini is None else ini.ctypes.data,
                                        out.ctypes.data))
    return None if rc == 1 else out
