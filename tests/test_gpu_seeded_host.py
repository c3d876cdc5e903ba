"""GPU parity of the seeded scan (device carries) and of the host-buffer
scan (chunks streamed through the GPU), against the CPU oracle.

A carry c in front of x is the oracle's scan of the array [c, x0, x1, ...]:
inclusive seeded y[i] = incl([c] + x)[i + 1], exclusive y[i] = incl([c] + x)[i],
and the carry out is incl([c] + x)[n].
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from conftest import FP32_ABS, FP32_REL
from prefix_scan_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from prefix_scan_gb300 import api  # noqa: E402

DEV = torch.device("cuda:0")
NP = {"int32": np.int32, "int64": np.int64, "float32": np.float32}
TT = {"int32": torch.int32, "int64": torch.int64, "float32": torch.float32}


def make(dtype, n, seed):
    if dtype == "int32":
        return inputs.full_range_i32(n, seed)
    if dtype == "int64":
        return inputs.hashes(n, seed).view(np.int64)
    return inputs.uniform_f32(n, seed)


def expected(x, c, exclusive):
    """(y, carry_out) from the oracle on [c, x...]."""
    cx = np.concatenate([np.array([c], dtype=x.dtype), x])
    inc = oracle.inclusive(cx)
    y = inc[:-1] if exclusive else inc[1:]
    return y, inc[-1], cx


def assert_close(got, want, cx, exclusive, dtype):
    if dtype != "float32":
        bad = np.flatnonzero(got != want)
        assert bad.size == 0, f"{bad.size} mismatches, first {bad[:5]}"
        return
    a = oracle.abs_prefix(cx, False)
    a = a[:-1] if exclusive else a[1:]
    ok = np.abs(got.astype(np.float64) - want) <= FP32_REL * a + FP32_ABS
    assert ok.all(), f"{(~ok).sum()} fp32 elements out of bound"


@pytest.mark.parametrize("dtype", list(NP))
@pytest.mark.parametrize("exclusive", [False, True], ids=["incl", "excl"])
def test_seeded_carries(dtype, exclusive):
    T = api.tile_elements(TT[dtype])
    # the last two: enough tiles for look-back units of two tiles (an odd
    # count leaves a unit with one tile past the end)
    for k, n in enumerate([1, 5, T, T + 1, 3 * T + 7, (1 << 20) + 3, 1301 * T + 5, 1302 * T]):
        x = make(dtype, n, 500 + k)
        c = make(dtype, 1, 900 + k)[0]
        y_want, tot_want, cx = expected(x, c, exclusive)
        xt = torch.from_numpy(x).to(DEV)
        cin = torch.tensor([c], dtype=TT[dtype], device=DEV)
        cout = torch.zeros(1, dtype=TT[dtype], device=DEV)
        y = api.scan_seeded(xt, cin, cout, exclusive=exclusive).cpu().numpy()
        assert_close(y, y_want, cx, exclusive, dtype)
        if dtype != "float32":
            assert cout.item() == int(tot_want)
        else:
            bound = FP32_REL * float(np.abs(cx.astype(np.float64)).sum()) + FP32_ABS
            assert abs(cout.item() - float(tot_want)) <= bound
        # carry in and out in one tensor (in place), and the scan in place too
        cio = torch.tensor([c], dtype=TT[dtype], device=DEV)
        api.scan_seeded(xt, cio, cio, exclusive=exclusive, out=xt)
        assert_close(xt.cpu().numpy(), y_want, cx, exclusive, dtype)
        if dtype != "float32":
            assert cio.item() == int(tot_want)
        else:
            bound = FP32_REL * float(np.abs(cx.astype(np.float64)).sum()) + FP32_ABS
            assert abs(cio.item() - float(tot_want)) <= bound


def test_seeded_without_carries_is_the_plain_scan():
    x = make("int32", 100_000, 7)
    y = api.scan_seeded(torch.from_numpy(x).to(DEV)).cpu().numpy()
    assert np.array_equal(y, oracle.inclusive(x))


def test_seeded_empty_copies_the_carry():
    e = torch.empty(0, dtype=torch.int64, device=DEV)
    cin = torch.tensor([1234567890123], dtype=torch.int64, device=DEV)
    cout = torch.zeros(1, dtype=torch.int64, device=DEV)
    api.scan_seeded(e, cin, cout)
    assert cout.item() == 1234567890123
    api.scan_seeded(e, None, cout)
    assert cout.item() == 0


def test_chunked_scan_with_carries_equals_whole_scan():
    # the use case of seeded scans: pieces scanned one after the other
    x = make("int64", 3_000_001, 11)
    xt = torch.from_numpy(x).to(DEV)
    carry = torch.zeros(1, dtype=torch.int64, device=DEV)
    outs = [api.scan_seeded(piece, carry, carry) for piece in torch.split(xt, 777_777)]
    got = torch.cat(outs).cpu().numpy()
    assert np.array_equal(got, oracle.inclusive(x))


@pytest.mark.parametrize("dtype", list(NP))
@pytest.mark.parametrize("exclusive", [False, True], ids=["incl", "excl"])
def test_host_scan_multi_chunk(dtype, exclusive):
    chunk = (32 << 20) // np.dtype(NP[dtype]).itemsize
    n = 4 * chunk + chunk // 2 + 3            # four and a half chunks (buffers reused), ragged tail
    x = make(dtype, n, 42)
    xt = torch.from_numpy(x).pin_memory()
    y = api.scan_host(xt, exclusive=exclusive).numpy()
    if dtype == "float32":
        from conftest import fp32_ok
        assert fp32_ok(y, x, exclusive).all()
    else:
        ref = oracle.exclusive(x) if exclusive else oracle.inclusive(x)
        assert np.array_equal(y, ref)


def test_host_scan_in_place_pageable_and_small():
    for n in (1, 1000, (32 << 20) // 4 + 1, 7 * (32 << 20) // 4 + 5):
        x = make("int32", n, 3 + n)
        xt = torch.from_numpy(x.copy())           # pageable, scanned in place
        api.scan_host(xt, out=xt)
        assert np.array_equal(xt.numpy(), oracle.inclusive(x))
    e = torch.empty(0, dtype=torch.int32)
    assert api.scan_host(e).numel() == 0


def test_host_scan_reuses_buffers():
    n = 5_000_000
    buf = api.HostScanBuffers(torch.int32, n, DEV)
    for seed in (1, 2):
        x = make("int32", n, seed)
        y = api.scan_host(torch.from_numpy(x).pin_memory(), buffers=buf).numpy()
        assert np.array_equal(y, oracle.inclusive(x))
