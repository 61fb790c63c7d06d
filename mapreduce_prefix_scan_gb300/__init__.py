"""GB300 (sm_103a) device-wide reduce and inclusive prefix scan.

A thin binding over the C ABI of include/ak.h (libak.so): every function
here only marshals arguments; all work runs in the library's CUDA kernels.
PyTorch supplies device memory and the current stream.

Arrays follow the C ABI's convention: a contiguous tensor holds a
column-major array of ``shape`` (default: the tensor's shape reversed), and
dimensions are numbered 0-based in that column-major shape (Julia's
``dims=2`` is ``1`` here). Element kinds: ``'f32'``, ``'f64'``, ``'bf16'``,
``'i32'``, ``'i64'``, and ``'mat2'`` (an int32 tensor whose last extent is 4:
2x2 matrices mod 2**31 - 1, entries a11, a21, a12, a22).
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

from . import _abi
from ._abi import DTYPES, MAPS, MAPS2, OPS, SHAPES, STORES

__all__ = ["AkError", "ak_reduce", "ak_reduce2", "ak_reduce_dims", "ak_accumulate", "ak_reduce_workspace_size",
           "ak_reduce_dims_workspace_size", "ak_accumulate_workspace_size", "ak_status_string",
           "ak_kernel_launch_count", "ak_dims_select", "ak_scan_status", "ak_findall",
           "ak_findall_workspace_size", "make_opts", "lib"]

_TORCH = {torch.float32: "f32", torch.float64: "f64", torch.bfloat16: "bf16", torch.int32: "i32",
          torch.int64: "i64", torch.uint8: "u8", torch.bool: "u8"}
_TORCH_OF = {"f32": torch.float32, "f64": torch.float64, "bf16": torch.bfloat16, "i32": torch.int32,
             "i64": torch.int64, "mat2": torch.int32, "u8": torch.uint8}
_NP_OF = {"f32": np.float32, "f64": np.float64, "i32": np.int32, "i64": np.int64}
_DEFAULT_ACC = {"f32": "f32", "f64": "f64", "bf16": "f32", "i32": "i32", "i64": "i64", "mat2": "mat2"}


class AkError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = lib().ak_status_string(status).decode()
        if status == _abi.AK_ERR_CUDA:
            msg += f" (cudaError {lib().ak_last_cuda_error()})"
        super().__init__(f"{where}: {msg}")


def lib() -> ctypes.CDLL:
    return _abi.load()


def _check(status: int, where: str) -> None:
    if status != _abi.AK_OK:
        raise AkError(status, where)


def ak_status_string(status: int) -> str:
    return lib().ak_status_string(status).decode()


def ak_kernel_launch_count() -> int:
    return int(lib().ak_kernel_launch_count())


def make_opts(no_neutral=False, target_blocks=0, items_per_thread=0, dims_shape="auto", check=False,
              wait_limit_ns=0, debug_skip_publish_tile=-1, dims_cluster=False, exclusive=False) -> _abi.ak_opts:
    o = _abi.ak_opts()
    lib().ak_opts_default(ctypes.byref(o))
    o.no_neutral = int(bool(no_neutral))
    o.target_blocks = int(target_blocks)
    o.items_per_thread = int(items_per_thread)
    o.dims_shape = SHAPES[dims_shape] if isinstance(dims_shape, str) else int(dims_shape)
    o.check = int(bool(check))
    o.wait_limit_ns = int(wait_limit_ns)
    o.debug_skip_publish_tile = int(debug_skip_publish_tile)
    o.flags = _abi.FLAG_DIMS_CLUSTER if dims_cluster else 0
    o.exclusive = int(bool(exclusive))
    return o


def _opts_ptr(opts):
    if opts is None:
        return None
    if isinstance(opts, dict):
        opts = make_opts(**opts)
    return ctypes.byref(opts)


def _kind(t: torch.Tensor, elem):
    if elem == "mat2":
        if t.dtype != torch.int32 or t.shape[-1] != 4:
            raise ValueError("mat2 arrays are int32 tensors whose last extent is 4")
        return "mat2"
    if elem is not None and elem != _TORCH.get(t.dtype):
        raise ValueError(f"tensor dtype {t.dtype} does not hold {elem} elements")
    if t.dtype not in _TORCH:
        raise ValueError(f"unsupported tensor dtype {t.dtype}")
    return _TORCH[t.dtype]


def _count(t: torch.Tensor, kind: str) -> int:
    return t.numel() // 4 if kind == "mat2" else t.numel()


def _colmajor_shape(t: torch.Tensor, kind: str, shape):
    if shape is not None:
        return [int(s) for s in shape]
    dims = list(t.shape[:-1]) if kind == "mat2" else list(t.shape)
    return [int(s) for s in reversed(dims)] or [1]


def _value_bytes(v, kind: str):
    """Host buffer holding one value of an accumulator kind (or None)."""
    if v is None:
        return None
    if kind == "mat2":
        a = np.asarray(v, dtype=np.uint32).reshape(4)
    elif kind == "bf16":
        raise ValueError("bf16 is not an accumulator type")
    else:
        a = np.array([v], dtype=_NP_OF[kind])
    return ctypes.create_string_buffer(a.tobytes(), 16)


def _from_bytes(buf, kind: str):
    raw = bytes(buf)[:16]
    if kind == "mat2":
        return tuple(int(t) for t in np.frombuffer(raw[:16], dtype=np.uint32))
    if kind == "bf16":
        bits = np.frombuffer(raw[:2], dtype=np.uint16)[0]
        return float(np.array([int(bits) << 16], dtype=np.uint32).view(np.float32)[0])
    a = np.frombuffer(raw[: np.dtype(_NP_OF[kind]).itemsize], dtype=_NP_OF[kind])[0]
    return float(a) if kind in ("f32", "f64") else int(a)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _require_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("arrays must be contiguous CUDA tensors")


def _workspace(nbytes: int, device, workspace):
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError("workspace too small")
        return workspace.data_ptr(), workspace.numel() * workspace.element_size(), workspace
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
    return ws.data_ptr(), ws.numel(), ws


# ---------------------------------------------------------------------------
# ak_reduce
# ---------------------------------------------------------------------------

def ak_reduce_workspace_size(n: int, in_kind: str, acc: str, opts=None) -> int:
    b = ctypes.c_size_t()
    _check(lib().ak_reduce_workspace_size(int(n), DTYPES[in_kind], DTYPES[acc], _opts_ptr(opts),
                                          ctypes.byref(b)), "ak_reduce_workspace_size")
    return b.value


def ak_reduce(src: torch.Tensor, *, f: str = "identity", op: str = "add", acc: str | None = None,
              out: str | None = None, init=None, mode: str | None = None, dst: torch.Tensor | None = None,
              to_host: bool = False, host_old=None, elem: str | None = None, workspace=None, opts=None,
              stream=None):
    """Whole-array mapreduce ``op(f(x_1), ..., f(x_n))``.

    Stores into ``dst`` (a one-element device tensor) and/or returns the host
    value when ``to_host`` is set. ``mode``: 'overwrite', 'init' (needs
    ``init``) or 'fold' (into dst's previous value, or ``host_old`` for a
    host-only fold). Default: 'init' when ``init`` is given, else
    'overwrite'.
    """
    if src.is_cuda and not src.is_contiguous():
        # a strided view: all of its dimensions through ak_reduce_dims
        kind = _kind(src, elem)
        sh, _ = _view_of(src, kind, None, None)
        r = dst if dst is not None else torch.empty(4 if (out or acc or _DEFAULT_ACC[kind]) == "mat2" else 1,
                                                    dtype=_TORCH_OF[out or acc or _DEFAULT_ACC[kind]],
                                                    device=src.device)
        if to_host and host_old is not None and mode == "fold":
            r.fill_(host_old)
        ak_reduce_dims(src, list(range(len(sh))), f=f, op=op, acc=acc, out=out, init=init, mode=mode, dst=r,
                       elem=elem, workspace=workspace, opts=opts, stream=stream)
        if to_host:
            v = r.cpu()
            return tuple(int(t) for t in v.view(torch.int32).numpy().view("uint32")) if v.numel() == 4 else v.item()
        return r
    _require_cuda(src, dst)
    kind = _kind(src, elem)
    acc = acc or _DEFAULT_ACC[kind]
    out = out or acc
    mode = mode or ("init" if init is not None else "overwrite")
    n = _count(src, kind)
    L = lib()
    size = ak_reduce_workspace_size(n, kind, acc, opts)
    wp, wb, _keep = _workspace(size, src.device, workspace)
    ib = _value_bytes(init, acc)
    hb = None
    if to_host:
        hb = ctypes.create_string_buffer(16)
        if host_old is not None:
            ctypes.memmove(hb, _value_bytes(host_old, out if out != "bf16" else "f32"), 16)
    _check(L.ak_reduce(src.data_ptr() if n else None, n, DTYPES[kind], MAPS[f], OPS[op], DTYPES[acc], DTYPES[out],
                       ib, STORES[mode], dst.data_ptr() if dst is not None else None, hb, wp, wb,
                       _opts_ptr(opts), _stream(stream)), "ak_reduce")
    if to_host:
        return _from_bytes(hb, out)
    return dst


def ak_reduce2(a: torch.Tensor, b: torch.Tensor, *, f: str = "mul", op: str = "add", acc: str | None = None,
               out: str | None = None, init=None, mode: str | None = None, dst: torch.Tensor | None = None,
               to_host: bool = False, host_old=None, workspace=None, opts=None, stream=None):
    """Whole-array mapreduce of a fused two-source element,
    ``op(f(a_1, b_1), ..., f(a_n, b_n))`` with f 'mul' (a*b), 'sqdiff'
    ((a-b)^2) or 'absdiff' (|a-b|); a and b have the same dtype and size.
    Stores and returns like ak_reduce."""
    _require_cuda(a, b, dst)
    kind = _kind(a, None)
    if _kind(b, None) != kind or a.numel() != b.numel():
        raise ValueError("both sources need the same dtype and number of elements")
    acc = acc or _DEFAULT_ACC[kind]
    out = out or acc
    mode = mode or ("init" if init is not None else "overwrite")
    n = a.numel()
    size = ak_reduce_workspace_size(n, kind, acc, opts)
    wp, wb, _keep = _workspace(size, a.device, workspace)
    hb = None
    if to_host:
        hb = ctypes.create_string_buffer(16)
        if host_old is not None:
            ctypes.memmove(hb, _value_bytes(host_old, out if out != "bf16" else "f32"), 16)
    _check(lib().ak_reduce2(a.data_ptr() if n else None, b.data_ptr() if n else None, n, DTYPES[kind], MAPS2[f],
                            OPS[op], DTYPES[acc], DTYPES[out], _value_bytes(init, acc), STORES[mode],
                            dst.data_ptr() if dst is not None else None, hb, wp, wb, _opts_ptr(opts),
                            _stream(stream)), "ak_reduce2")
    if to_host:
        return _from_bytes(hb, out)
    return dst


# ---------------------------------------------------------------------------
# ak_reduce_dims
# ---------------------------------------------------------------------------

def _mask(dims) -> int:
    m = 0
    for d in dims:
        m |= 1 << int(d)
    return m


def ak_reduce_dims_workspace_size(shape, dims, in_kind: str, acc: str, opts=None, strides=None) -> int:
    sh = (ctypes.c_int64 * len(shape))(*shape)
    st = None if strides is None else (ctypes.c_int64 * len(strides))(*strides)
    b = ctypes.c_size_t()
    _check(lib().ak_reduce_dims_workspace_size(len(shape), sh, st, _mask(dims), DTYPES[in_kind], DTYPES[acc],
                                               _opts_ptr(opts), ctypes.byref(b)), "ak_reduce_dims_workspace_size")
    return b.value


def _view_of(t: torch.Tensor, kind: str, shape, strides):
    """Column-major shape and element strides of a (possibly non-contiguous)
    tensor; None strides for a contiguous one."""
    if shape is not None:
        return [int(v) for v in shape], (None if strides is None else [int(v) for v in strides])
    if t.is_contiguous():
        return _colmajor_shape(t, kind, None), None
    if kind == "mat2":
        if t.stride(-1) != 1:
            raise ValueError("a view of 2x2 matrices must keep each matrix's four entries together")
        dims, sts = list(t.shape[:-1]), [s // 4 for s in t.stride()[:-1]]
        if any(s % 4 for s in t.stride()[:-1]):
            raise ValueError("a view of 2x2 matrices must step by whole matrices")
    else:
        dims, sts = list(t.shape), list(t.stride())
    return [int(v) for v in reversed(dims)] or [1], [int(v) for v in reversed(sts)] or [1]


def ak_reduce_dims(src: torch.Tensor, dims, *, shape=None, f: str = "identity", op: str = "add",
                   acc: str | None = None, out: str | None = None, init=None, mode: str | None = None,
                   dst: torch.Tensor | None = None, elem: str | None = None, workspace=None, opts=None,
                   stream=None, strides=None) -> torch.Tensor:
    """mapreducedim!: reduce the 0-based column-major dimensions ``dims``.

    ``src`` may be a non-contiguous view (a slice, a transpose): its strides
    are passed to the library, nothing is copied. Returns ``dst``: a
    contiguous tensor holding the column-major result (reduced extents 1);
    allocated when not given, with the row-major shape of the reversed
    column-major result shape.
    """
    if src is not None and (not src.is_cuda):
        raise ValueError("arrays must be CUDA tensors")
    _require_cuda(dst)
    kind = _kind(src, elem)
    acc = acc or _DEFAULT_ACC[kind]
    out = out or (kind if kind == "bf16" else acc)
    mode = mode or ("init" if init is not None else "overwrite")
    sh, st = _view_of(src, kind, shape, strides)
    mask = _mask(dims)
    out_shape = [1 if (mask >> d) & 1 else s for d, s in enumerate(sh)]
    if dst is None:
        rows = list(reversed(out_shape))
        if out == "mat2":
            rows = rows + [4]
        dst = torch.empty(rows, dtype=_TORCH_OF[out], device=src.device)
    size = ak_reduce_dims_workspace_size(sh, dims, kind, acc, opts, strides=st)
    wp, wb, _keep = _workspace(size, src.device, workspace)
    csh = (ctypes.c_int64 * len(sh))(*sh)
    cst = None if st is None else (ctypes.c_int64 * len(st))(*st)
    _check(lib().ak_reduce_dims(src.data_ptr() if src.numel() else None, len(sh), csh, cst, mask, DTYPES[kind],
                                MAPS[f],
                                OPS[op], DTYPES[acc], DTYPES[out], _value_bytes(init, acc), STORES[mode],
                                dst.data_ptr() if dst.numel() else None, wp, wb, _opts_ptr(opts),
                                _stream(stream)), "ak_reduce_dims")
    return dst


# ---------------------------------------------------------------------------
# ak_accumulate
# ---------------------------------------------------------------------------

def ak_accumulate_workspace_size(shape, dim: int, in_kind: str, acc: str, op: str = "add", opts=None) -> int:
    sh = (ctypes.c_int64 * len(shape))(*shape)
    b = ctypes.c_size_t()
    _check(lib().ak_accumulate_workspace_size(len(shape), sh, int(dim), DTYPES[in_kind], DTYPES[acc], OPS[op],
                                              _opts_ptr(opts), ctypes.byref(b)), "ak_accumulate_workspace_size")
    return b.value


def ak_accumulate(src: torch.Tensor, *, dim: int = -1, shape=None, op: str = "add", acc: str | None = None,
                  out: str | None = None, init=None, dst: torch.Tensor | None = None, elem: str | None = None,
                  workspace=None, opts=None, stream=None, exclusive: bool = False) -> torch.Tensor:
    """Inclusive scan (accumulate!): the whole array (dim=-1) or along the
    0-based column-major dimension ``dim``. ``dst`` may be ``src``. With
    ``exclusive`` element i holds the fold of init (or the neutral element)
    and the elements before it."""
    if exclusive:
        if opts is None:
            opts = make_opts(exclusive=True)
        elif isinstance(opts, dict):
            opts = make_opts(**dict(opts, exclusive=True))
        else:
            opts.exclusive = 1
    _require_cuda(src, dst)
    kind = _kind(src, elem)
    acc = acc or _DEFAULT_ACC[kind]
    out = out or acc
    sh = _colmajor_shape(src, kind, shape)
    if dst is None:
        rows = list(src.shape)
        dst = torch.empty(rows, dtype=_TORCH_OF[out], device=src.device)
    size = ak_accumulate_workspace_size(sh, dim, kind, acc, op, opts)
    wp, wb, _keep = _workspace(size, src.device, workspace)
    csh = (ctypes.c_int64 * len(sh))(*sh)
    _check(lib().ak_accumulate(src.data_ptr() if src.numel() else None, dst.data_ptr() if dst.numel() else None,
                               len(sh), csh, int(dim), DTYPES[kind], OPS[op], DTYPES[acc], DTYPES[out],
                               _value_bytes(init, acc), wp, wb, _opts_ptr(opts), _stream(stream)),
           "ak_accumulate")
    return dst


# ---------------------------------------------------------------------------
# ak_findall
# ---------------------------------------------------------------------------

def ak_findall_workspace_size(n: int, in_kind: str, opts=None) -> int:
    b = ctypes.c_size_t()
    _check(lib().ak_findall_workspace_size(int(n), DTYPES[in_kind], _opts_ptr(opts), ctypes.byref(b)),
           "ak_findall_workspace_size")
    return b.value


def ak_findall(src: torch.Tensor, *, idx: torch.Tensor | None = None, count: torch.Tensor | None = None,
               to_host: bool = True, workspace=None, opts=None, stream=None):
    """Indices (0-based, increasing, int64) of the nonzero elements of src
    (bool / uint8 flags, int32, int64, float32, float64). With ``to_host``
    returns ``idx[:count]`` (the call synchronizes); otherwise returns
    ``(idx, count)`` with the count in a one-element device tensor."""
    _require_cuda(src, idx, count)
    kind = _kind(src, None)
    if kind not in ("u8", "i32", "i64", "f32", "f64"):
        raise ValueError("findall takes bool / uint8, int32, int64, float32 or float64 arrays")
    n = src.numel()
    if idx is None:
        idx = torch.empty(max(n, 1), dtype=torch.int64, device=src.device)
    if not to_host and count is None:
        count = torch.empty(1, dtype=torch.int64, device=src.device)
    size = ak_findall_workspace_size(n, kind, opts)
    wp, wb, _keep = _workspace(size, src.device, workspace)
    hc = ctypes.c_int64(-1) if to_host else None
    _check(lib().ak_findall(src.data_ptr() if n else None, n, DTYPES[kind], idx.data_ptr(),
                            count.data_ptr() if count is not None else None,
                            ctypes.byref(hc) if hc is not None else None, wp, wb, _opts_ptr(opts),
                            _stream(stream)), "ak_findall")
    if to_host:
        return idx[: hc.value]
    return idx, count


def ak_scan_status(workspace: torch.Tensor) -> int:
    """Status of the last ak_accumulate on this workspace (0 ok, AK_ERR_TIMEOUT
    when a bounded wait ran out); call after the stream has passed the scan."""
    return int(lib().ak_scan_status(workspace.data_ptr()))


def ak_dims_select(inner: int, red_len: int, outer: int, elem_bytes: int, vec_elems: int, sm_count: int,
                   forced: str = "auto"):
    """The dims-reduction shape selector (host logic): returns
    (shape name, outputs per block, row groups, split)."""
    vals = [ctypes.c_int32() for _ in range(4)]
    _check(lib().ak_dims_select(inner, red_len, outer, elem_bytes, vec_elems, sm_count, SHAPES[forced],
                                *[ctypes.byref(v) for v in vals]), "ak_dims_select")
    names = {v: k for k, v in SHAPES.items()}
    return names[vals[0].value], vals[1].value, vals[2].value, vals[3].value
