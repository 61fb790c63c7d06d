"""ctypes prototypes of include/ak.h (plain pointers and sizes).

Loading fails loudly when the in-tree library has not been built: there is
no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libak.so")

# enums of include/ak.h
AK_OK, AK_ERR_INVALID_ARG, AK_ERR_UNSUPPORTED, AK_ERR_WORKSPACE, AK_ERR_EMPTY_NO_INIT, AK_ERR_CUDA, \
    AK_ERR_TIMEOUT = range(7)
DTYPES = {"f32": 0, "f64": 1, "bf16": 2, "i32": 3, "i64": 4, "mat2": 5, "u8": 6}
MAPS = {"identity": 0, "abs": 1, "abs2": 2}
MAPS2 = {"mul": 0, "sqdiff": 1, "absdiff": 2}
OPS = {"add": 0, "mul": 1, "max": 2, "min": 3, "matmul": 4}
STORES = {"overwrite": 0, "init": 1, "fold": 2}
SHAPES = {"auto": 0, "thread": 1, "tiled": 2, "columns": 3}
FLAG_DIMS_CLUSTER = 1

# every symbol include/ak.h declares
EXPORTS = ("ak_opts_default", "ak_status_string", "ak_dtype_size", "ak_last_cuda_error",
           "ak_kernel_launch_count", "ak_reduce_workspace_size", "ak_reduce", "ak_reduce2",
           "ak_reduce_dims_workspace_size", "ak_reduce_dims", "ak_accumulate_workspace_size",
           "ak_accumulate", "ak_scan_status", "ak_findall_workspace_size", "ak_findall", "ak_dims_select",
           "ak_reduce_noalloc")


class ak_opts(ctypes.Structure):
    _fields_ = [("no_neutral", ctypes.c_int32), ("target_blocks", ctypes.c_int32),
                ("items_per_thread", ctypes.c_int32), ("dims_shape", ctypes.c_int32),
                ("check", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("exclusive", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("wait_limit_ns", ctypes.c_int64), ("debug_skip_publish_tile", ctypes.c_int64)]


_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libak.so (LIB_PATH unless a path is given) and declare its
    prototypes. There is no fallback: without the library every call raises."""
    global _lib
    if path is None:
        if _lib is not None:
            return _lib
        path = LIB_PATH
    if not os.path.exists(path):
        raise ImportError(f"libak.so not built ({path}); run __graft_entry__.build() or "
                          "python -m mapreduce_prefix_scan_gb300.build")
    L = ctypes.CDLL(path)
    P, I32, I64, U32, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_uint32, ctypes.c_size_t
    PI64 = ctypes.POINTER(ctypes.c_int64)
    PSZ = ctypes.POINTER(ctypes.c_size_t)
    PO = ctypes.POINTER(ak_opts)
    PI32 = ctypes.POINTER(ctypes.c_int32)
    L.ak_opts_default.argtypes = [PO]
    L.ak_opts_default.restype = None
    L.ak_status_string.argtypes = [I32]
    L.ak_status_string.restype = ctypes.c_char_p
    L.ak_dtype_size.argtypes = [I32]
    L.ak_dtype_size.restype = SZ
    L.ak_last_cuda_error.argtypes = []
    L.ak_last_cuda_error.restype = I32
    L.ak_kernel_launch_count.argtypes = []
    L.ak_kernel_launch_count.restype = ctypes.c_uint64
    L.ak_reduce_workspace_size.argtypes = [I64, I32, I32, PO, PSZ]
    L.ak_reduce.argtypes = [P, I64, I32, I32, I32, I32, I32, P, I32, P, P, P, SZ, PO, P]
    L.ak_reduce2.argtypes = [P, P, I64, I32, I32, I32, I32, I32, P, I32, P, P, P, SZ, PO, P]
    L.ak_reduce_dims_workspace_size.argtypes = [I32, PI64, PI64, U32, I32, I32, PO, PSZ]
    L.ak_reduce_dims.argtypes = [P, I32, PI64, PI64, U32, I32, I32, I32, I32, I32, P, I32, P, P, SZ, PO, P]
    L.ak_accumulate_workspace_size.argtypes = [I32, PI64, I32, I32, I32, I32, PO, PSZ]
    L.ak_accumulate.argtypes = [P, P, I32, PI64, I32, I32, I32, I32, I32, P, P, SZ, PO, P]
    L.ak_scan_status.argtypes = [P]
    L.ak_findall_workspace_size.argtypes = [I64, I32, PO, PSZ]
    L.ak_findall.argtypes = [P, I64, I32, P, P, P, P, SZ, PO, P]
    L.ak_dims_select.argtypes = [I64, I64, I64, I32, I32, I32, I32, PI32, PI32, PI32, PI32]
    L.ak_reduce_noalloc.argtypes = [P, I64, I32, I32, I32, I32, I32, P, I32, P, P, PO, P]
    for f in ("ak_reduce_workspace_size", "ak_reduce", "ak_reduce2", "ak_reduce_dims_workspace_size", "ak_reduce_dims",
              "ak_accumulate_workspace_size", "ak_accumulate", "ak_scan_status", "ak_findall_workspace_size",
              "ak_findall", "ak_dims_select", "ak_reduce_noalloc"):
        getattr(L, f).restype = I32
    if path == LIB_PATH:
        _lib = L
    return L
