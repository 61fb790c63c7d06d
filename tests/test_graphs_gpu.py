"""Calls captured in a CUDA graph and replayed on fresh data.

Production callers capture launch-bound sequences in CUDA graphs; every
argument of a captured call (including anything the library derives per
call on the host) is frozen at capture time. Each replay here runs on new
input data copied into the captured buffers and is checked against the
oracle, so state carried from one replay to the next (a stale tile-prefix
record, a claim counter) would show up as a wrong result.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mapreduce_prefix_scan_gb300 as ak
import oracle
import synth
from helpers import F64_REL, assert_close_f32, assert_exact, colmajor_mass, dev_of

pytestmark = pytest.mark.gpu


def _capture(fn):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()  # warm up outside the graph (lazy module loading, attributes)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_reduce_replays():
    n = 3_000_001
    x = torch.empty(n, dtype=torch.int64, device="cuda")
    r = torch.empty(1, dtype=torch.int64, device="cuda")
    ws = torch.empty(ak.ak_reduce_workspace_size(n, "i64", "i64"), dtype=torch.uint8, device="cuda")
    g = _capture(lambda: ak.ak_reduce(x, op="max", dst=r, workspace=ws))
    for rep in range(3):
        h = synth.uniform_int(n, -(2**31), 2**31 - 1, np.int64, stream=100 + rep)
        x.copy_(torch.from_numpy(h))
        g.replay()
        torch.cuda.synchronize()
        assert r.item() == oracle.reduce(h, "i64", op="max")


def test_reduce_dims_replays():
    shape = (3072, 2048)
    x = torch.empty((2048, 3072), dtype=torch.float32, device="cuda")
    dst = torch.empty((1, 3072), dtype=torch.float32, device="cuda")
    ws = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    g = _capture(lambda: ak.ak_reduce_dims(x, [1], dst=dst, workspace=ws))
    for rep in range(3):
        h = synth.normal_f32(3072 * 2048, stream=110 + rep)
        x.copy_(torch.from_numpy(h).reshape(2048, 3072))
        g.replay()
        torch.cuda.synchronize()
        want = oracle.reduce_dims(h, "f32", shape, [1])
        assert_close_f32(dst.cpu().numpy(), want, colmajor_mass(h.astype(np.float64), shape, [1]))


@pytest.mark.parametrize("kind,n,op", [("f64", 2_500_003, "add"), ("mat2", 300_001, "matmul"),
                                       ("i64", 1_000_000, "max")])
def test_accumulate_replays(kind, n, op):
    shape = (n, 4) if kind == "mat2" else (n,)
    dt = {"f64": torch.float64, "i64": torch.int64, "mat2": torch.int32}[kind]
    x = torch.empty(shape, dtype=dt, device="cuda")
    y = torch.empty_like(x)
    elem = "mat2" if kind == "mat2" else None
    ws = torch.empty(ak.ak_accumulate_workspace_size([n], -1, kind, kind, op), dtype=torch.uint8, device="cuda")
    g = _capture(lambda: ak.ak_accumulate(x, dst=y, op=op, elem=elem, workspace=ws))
    for rep in range(3):
        if kind == "f64":
            h = synth.uniform_f64_01(n, stream=120 + rep)
        elif kind == "i64":
            h = synth.uniform_int(n, -(2**20), 2**20, np.int64, stream=120 + rep)
        else:
            h = synth.mat2_modp(n, stream=120 + rep)
        x.copy_(torch.from_numpy(h))
        g.replay()
        torch.cuda.synchronize()
        got = y.cpu().numpy()
        if kind == "f64":
            assert_close_f32(got, oracle.scan(h, "f64"), np.cumsum(np.abs(h)), rel=F64_REL)
        elif kind == "i64":
            assert_exact(got, oracle.scan(h, "i64", op="max"))
        else:
            assert_exact(got.view(np.uint32).reshape(-1, 4), oracle.scan(h, "mat2"))
