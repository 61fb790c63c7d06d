"""GPU parity of ak_reduce2 (fused two-source reductions) against the oracle.

A fused (Broadcasted) source such as sum(x .* y) or sum(abs2.(x .- y)) is
reduced without materialising the elementwise array ("Finish whole-array
reductions on the device", section "What changes"; its tests cover fused
sources). Float sums within 2^-20 * sum |f(a_i, b_i)| of the f64 oracle, bf16
inputs likewise (f32 accumulate), integers and max / min bit-exact. Covered:
the 1e8 f32 dot product, ragged sizes, every map and type, co-aligned and
differently aligned sources, init / fold / host results, and Optional
partials.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mapreduce_prefix_scan_gb300 as ak
import oracle
import synth
from helpers import F32_REL, dev_of, gen

pytestmark = pytest.mark.gpu


def _mass(a, b, f):
    a64, b64 = a.astype(np.float64), b.astype(np.float64)
    if f == "mul":
        return float(np.abs(a64 * b64).sum())
    if f == "sqdiff":
        return float(((a64 - b64) ** 2).sum())
    return float(np.abs(a64 - b64).sum())


def _pair(kind, n, s1, s2):
    if kind == "bf16":
        return synth.normal_bf16_bits(n, 0, s1), synth.normal_bf16_bits(n, 0, s2)
    return gen(kind, n, stream=s1), gen(kind, n, stream=s2)


def _check(kind, a, b, f, op, got, init=None):
    want = oracle.reduce2(a, b, kind, f, op=op, init=init)
    if kind in ("i32", "i64"):
        assert got == want, (got, want)
    elif op in ("max", "min"):
        # f is applied in the f32 accumulator; rounding is monotone, so the
        # extreme of the rounded values is the rounded exact extreme
        assert got == float(np.float32(want)), (got, want)
    else:
        if kind == "bf16":
            a = synth.bf16_bits_to_f32(a)
            b = synth.bf16_bits_to_f32(b)
        tol = F32_REL * (_mass(a, b, f) + abs(init or 0))
        if kind == "f64":
            tol = 2.0**-40 * (_mass(a, b, f) + abs(init or 0))
        assert abs(got - want) <= tol, (got, want, tol)


def test_dot_1e8_f32():
    a = synth.uniform_f32_pm1(10**8, 0, 100)
    b = synth.uniform_f32_pm1(10**8, 0, 101)
    got = ak.ak_reduce2(dev_of("f32", a), dev_of("f32", b), f="mul", to_host=True)
    _check("f32", a, b, "mul", "add", got)


@pytest.mark.parametrize("n", [1, 17, 1000, 16385, 1_000_003])
@pytest.mark.parametrize("kind", ["f32", "f64", "bf16", "i32", "i64"])
@pytest.mark.parametrize("f", ["mul", "sqdiff", "absdiff"])
def test_maps_types_sizes(n, kind, f):
    a, b = _pair(kind, n, 102, 103)
    ad, bd = dev_of(kind, a), dev_of(kind, b)
    got = ak.ak_reduce2(ad, bd, f=f, to_host=True, acc="f32" if kind == "bf16" else None,
                        out="f32" if kind == "bf16" else None)
    _check(kind, a, b, f, "add", got)


@pytest.mark.parametrize("op", ["max", "min"])
@pytest.mark.parametrize("kind", ["f32", "i64"])
def test_max_min(op, kind):
    a, b = _pair(kind, 300_001, 104, 105)
    got = ak.ak_reduce2(dev_of(kind, a), dev_of(kind, b), f="sqdiff", op=op, to_host=True)
    _check(kind, a, b, "sqdiff", op, got)


@pytest.mark.parametrize("offa,offb", [(0, 0), (3, 3), (0, 5), (7, 2)])
def test_alignments(offa, offb):
    n = 1_000_000
    a, b = _pair("f32", n + 8, 106, 107)
    ad, bd = dev_of("f32", a), dev_of("f32", b)
    got = ak.ak_reduce2(ad[offa: offa + n], bd[offb: offb + n], f="mul", to_host=True)
    _check("f32", a[offa: offa + n], b[offb: offb + n], "mul", "add", got)


def test_store_modes_and_optional():
    a, b = _pair("i64", 100_003, 108, 109)
    ad, bd = dev_of("i64", a), dev_of("i64", b)
    r = torch.tensor([5], dtype=torch.int64, device="cuda")
    ak.ak_reduce2(ad, bd, f="mul", dst=r, mode="fold")
    assert int(r.item()) == oracle.reduce2(a, b, "i64", "mul", init=5)
    ak.ak_reduce2(ad, bd, f="absdiff", dst=r, init=-3)
    assert int(r.item()) == oracle.reduce2(a, b, "i64", "absdiff", init=-3)
    # Optional partials (no neutral element): same result for max
    got = ak.ak_reduce2(ad, bd, f="mul", op="max", to_host=True, opts=ak.make_opts(no_neutral=True))
    assert got == oracle.reduce2(a, b, "i64", "mul", op="max")
    # f32 sources, f64 accumulator
    fa, fb = _pair("f32", 50_000, 110, 111)
    got = ak.ak_reduce2(dev_of("f32", fa), dev_of("f32", fb), f="sqdiff", acc="f64", to_host=True)
    assert abs(got - oracle.reduce2(fa, fb, "f32", "sqdiff")) <= 2.0**-44 * _mass(fa, fb, "sqdiff")


def test_empty_and_rejections():
    e = torch.zeros(0, dtype=torch.float32, device="cuda")
    assert ak.ak_reduce2(e, e, to_host=True) == 0.0
    with pytest.raises(ak.AkError, match="empty reduction"):
        ak.ak_reduce2(e, e, op="max", to_host=True)
    m = torch.zeros(8, 4, dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        ak.ak_reduce2(torch.zeros(4, device="cuda"), torch.zeros(5, device="cuda"))
    from mapreduce_prefix_scan_gb300 import _abi
    L = ak.lib()
    assert L.ak_reduce2(m.data_ptr(), m.data_ptr(), 8, 5, 0, 4, 5, 5, None, 0, m.data_ptr(), None, None, 0, None,
                        None) == _abi.AK_ERR_UNSUPPORTED
