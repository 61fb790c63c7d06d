"""Canary words around every output buffer: each entry point writes exactly
its outputs and nothing next to them.

Outputs sit in the middle of a byte buffer whose 256-byte margins hold a
fixed pattern; after the call (at sizes on either side of vector widths, rows,
tiles and super-tiles) the margins must be intact and the outputs must match
the oracle. Also: AK_LOG=1 names the path each call takes, on stderr.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mapreduce_prefix_scan_gb300 as ak
import oracle
import synth
from helpers import F32_REL, assert_close_f32, assert_exact, dev_of, gen

pytestmark = pytest.mark.gpu

MARGIN = 256
CANARY = 0xA5


def _guarded(numel: int, dtype: torch.dtype):
    """(buffer, view): `numel` elements of dtype between two canary margins."""
    nbytes = numel * torch.empty(0, dtype=dtype).element_size()
    buf = torch.full((MARGIN + nbytes + MARGIN,), CANARY, dtype=torch.uint8, device="cuda")
    return buf, buf[MARGIN:MARGIN + nbytes].view(dtype)


def _margins_intact(buf: torch.Tensor):
    torch.cuda.synchronize()
    b = buf.cpu().numpy()
    assert np.all(b[:MARGIN] == CANARY), "write before the output"
    assert np.all(b[-MARGIN:] == CANARY), "write after the output"


SIZES = [1, 2, 31, 33, 255, 257, 4095, 4097, 8193, 16385, 65537, 262145, 1_000_003]


@pytest.mark.parametrize("n", SIZES)
def test_reduce_writes_one_element(n):
    x = gen("i64", n, stream=140)
    buf, dst = _guarded(1, torch.int64)
    ak.ak_reduce(dev_of("i64", x), dst=dst)
    _margins_intact(buf)
    assert int(dst.item()) == oracle.reduce(x, "i64")
    buf2, dst2 = _guarded(1, torch.int64)
    ak.ak_reduce2(dev_of("i64", x), dev_of("i64", x[::-1].copy()), f="mul", dst=dst2)
    _margins_intact(buf2)
    assert int(dst2.item()) == oracle.reduce2(x, x[::-1].copy(), "i64", map2="mul")


@pytest.mark.parametrize("shape,dims", [((31, 33), (1,)), ((33, 31), (0,)), ((3072, 7), (1,)), ((5, 7, 9), (1,)),
                                        ((257, 3, 65), (0, 2)), ((1, 1000), (1,)), ((64, 4096, 3), (1,))])
def test_reduce_dims_writes_its_outputs(shape, dims):
    n = int(np.prod(shape))
    x = gen("i32", n, stream=141)
    want = oracle.reduce_dims(x, "i32", shape, dims)
    buf, dst = _guarded(want.size, torch.int32)
    xd = dev_of("i32", x).reshape(tuple(reversed(shape)))
    ak.ak_reduce_dims(xd, list(dims), dst=dst)
    _margins_intact(buf)
    assert_exact(dst.cpu().numpy().astype(np.int64), want)


@pytest.mark.parametrize("kind", ["f32", "f64", "i64", "mat2"])
@pytest.mark.parametrize("n", [1, 31, 33, 4097, 65537, 262145, 1_000_003])
@pytest.mark.parametrize("exclusive", [False, True])
def test_accumulate_writes_its_outputs(kind, n, exclusive):
    if kind == "mat2":
        x = synth.mat2_modp(n, stream=142)
        buf, dst = _guarded(4 * n, torch.int32)
        ak.ak_accumulate(dev_of("mat2", x), dst=dst.view(n, 4), op="matmul", elem="mat2", exclusive=exclusive)
        _margins_intact(buf)
        init = np.array([1, 0, 0, 1], np.uint32) if exclusive else None
        assert_exact(dst.cpu().numpy().view(np.uint32).reshape(-1, 4),
                     oracle.scan(x, "mat2", exclusive=exclusive, init=init))
        return
    x = gen(kind, n, stream=143, dist="normal" if kind != "i64" else "uniform")
    tdt = {"f32": torch.float32, "f64": torch.float64, "i64": torch.int64}[kind]
    buf, dst = _guarded(n, tdt)
    ak.ak_accumulate(dev_of(kind, x), dst=dst, exclusive=exclusive)
    _margins_intact(buf)
    want = oracle.scan(x, kind, exclusive=exclusive, init=0 if exclusive else None)
    if kind == "i64":
        assert_exact(dst.cpu().numpy(), want)
    else:
        a = np.abs(x.astype(np.float64))
        mass = np.concatenate([[0.0], np.cumsum(a)[:-1]]) if exclusive else np.cumsum(a)
        assert_close_f32(dst.cpu().numpy(), want, mass, rel=F32_REL if kind == "f32" else 2.0**-36)


@pytest.mark.parametrize("n", [1, 63, 65, 16383, 16385, 100_003])
def test_findall_writes_count_indices(n):
    w = synth.words(n, 0, 144)
    flags = ((w >> np.uint64(62)) == 1).astype(np.uint8)
    want = oracle.findall(flags, "u8")
    ibuf, idx = _guarded(n, torch.int64)
    cbuf, cnt = _guarded(1, torch.int64)
    ak.ak_findall(torch.from_numpy(flags).cuda(), idx=idx, count=cnt, to_host=False)
    _margins_intact(ibuf)
    _margins_intact(cbuf)
    c = int(cnt.item())
    assert c == want.size
    assert_exact(idx[:c].cpu().numpy(), want)


def test_ak_log_names_the_path(capfd, monkeypatch):
    monkeypatch.setenv("AK_LOG", "1")
    x = dev_of("f32", synth.normal_f32(10**6, stream=145))
    ak.ak_reduce(x, to_host=True)
    ak.ak_reduce_dims(x.reshape(1000, 1000), [1])
    ak.ak_accumulate(x)
    ak.ak_accumulate(x, op="max", opts=ak.make_opts(no_neutral=True))
    ak.ak_findall(torch.ones(1000, dtype=torch.uint8, device="cuda"))
    torch.cuda.synchronize()
    err = capfd.readouterr().err
    lines = [ln for ln in err.splitlines() if ln.startswith("[ak] ")]
    assert any(ln.startswith("[ak] reduce n=1000000") and "host (mapped slot, polled)" in ln for ln in lines), err
    assert any(ln.startswith("[ak] reduce_dims nout=1000 nfold=1000") and "strided kernel" in ln for ln in lines), err
    assert any(ln.startswith("[ak] accumulate") and "TMA tile ring" in ln for ln in lines), err
    assert any("optional partials" in ln and "three-launch" in ln for ln in lines), err
    assert any(ln.startswith("[ak] findall n=1000") for ln in lines), err
    monkeypatch.setenv("AK_LOG", "0")
    ak.ak_accumulate(x)
    torch.cuda.synchronize()
    assert "[ak] " not in capfd.readouterr().err
