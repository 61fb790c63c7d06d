"""GPU parity of ak_findall (stream compaction) against the oracle.

findall returns the indices of the nonzero elements in increasing order:
index work, so the comparison is bit-exact (same indices, same count).
Covered: the Bool-flag workload at full size (1e8 flags, half of them set),
ragged sizes around the tile sizes, densities 0 to 1, every element type
(floats with -0.0 and NaN), unaligned sources, the count left on the device,
and a bounded look-back wait running out on an injected missing
publication.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import mapreduce_prefix_scan_gb300 as ak
import oracle
import synth
from helpers import assert_exact

pytestmark = pytest.mark.gpu


def _flags(n, density, stream):
    """Bool flags (uint8 0/1), each set with probability `density`."""
    if density <= 0:
        return np.zeros(n, np.uint8)
    if density >= 1:
        return np.ones(n, np.uint8)
    w = synth.words(n, seed=0, stream=stream)
    return ((w >> np.uint64(11)).astype(np.float64) * 2.0**-53 < density).astype(np.uint8)


def test_findall_1e8_flags_half_set():
    x = _flags(10**8, 0.5, 90)
    got = ak.ak_findall(torch.from_numpy(x).cuda()).cpu().numpy()
    assert_exact(got, oracle.findall(x, "u8"))


@pytest.mark.parametrize("n", [1, 63, 64, 65, 16383, 16384, 16385, 3 * 16384 + 7, 1_000_003])
@pytest.mark.parametrize("density", [0.0, 0.01, 0.5, 1.0])
def test_findall_sizes_and_densities(n, density):
    x = _flags(n, density, 91)
    got = ak.ak_findall(torch.from_numpy(x).cuda()).cpu().numpy()
    assert_exact(got, oracle.findall(x, "u8"))


@pytest.mark.parametrize("kind", ["i32", "i64", "f32", "f64"])
@pytest.mark.parametrize("n", [1000, 8192 * 3 + 5, 2_000_001])
def test_findall_element_types(kind, n):
    w = synth.uniform_int(n, 0, 2, np.int64, stream=92)   # a third zero
    dt = {"i32": np.int32, "i64": np.int64, "f32": np.float32, "f64": np.float64}[kind]
    x = (w - 1).astype(dt)                                # -1, 0, 1
    if kind in ("f32", "f64"):
        x[::7] = -0.0                                     # counts as zero
        x[3::11] = np.nan                                 # counts as nonzero
    got = ak.ak_findall(torch.from_numpy(x).cuda()).cpu().numpy()
    assert_exact(got, oracle.findall(x, kind))


def test_findall_bool_tensor_unaligned_and_device_count():
    x = _flags(500_003, 0.3, 93)
    xd = torch.from_numpy(x).cuda()
    # a bool tensor holds the same bytes
    assert_exact(ak.ak_findall(xd.bool()).cpu().numpy(), oracle.findall(x, "u8"))
    # an offset view starts off the 32-byte boundary (element-wise loads)
    assert_exact(ak.ak_findall(xd[5:]).cpu().numpy(), oracle.findall(x[5:].copy(), "u8"))
    # the count stays on the device; entries past it are untouched
    idx = torch.full((x.size,), -7, dtype=torch.int64, device="cuda")
    idx, cnt = ak.ak_findall(xd, idx=idx, to_host=False)
    want = oracle.findall(x, "u8")
    assert int(cnt.item()) == want.size
    got = idx.cpu().numpy()
    assert_exact(got[: want.size], want)
    assert np.all(got[want.size:] == -7)


def test_findall_empty_input():
    got = ak.ak_findall(torch.zeros(0, dtype=torch.uint8, device="cuda"))
    assert got.numel() == 0
    idx, cnt = ak.ak_findall(torch.zeros(0, dtype=torch.uint8, device="cuda"), to_host=False)
    assert int(cnt.item()) == 0


def test_findall_wait_runs_out_and_next_call_is_correct():
    x = _flags(16384 * 40, 0.5, 94)
    xd = torch.from_numpy(x).cuda()
    o = ak.make_opts(check=True, wait_limit_ns=20_000_000, debug_skip_publish_tile=3)
    with pytest.raises(ak.AkError, match="wait ran out"):
        ak.ak_findall(xd, opts=o)
    assert_exact(ak.ak_findall(xd, opts=ak.make_opts(check=True)).cpu().numpy(), oracle.findall(x, "u8"))
