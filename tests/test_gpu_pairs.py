"""GPU parity of the 8-byte pair scans against the CPU oracle.

{int32, fp32} pairs: the int32 field bit for bit, the fp32 field within the
scan bound FP32_REL * sum|f| + FP32_ABS.  Affine maps (a, b) composed in
order: A within FP32_REL * |A| + FP32_ABS, B within FP32_REL * (the same
recurrence over |a|, |b|) + FP32_ABS, of the fp64 oracle.
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
T = 4096   # elements per tile of 8-byte elements
# the last: enough tiles for look-back units of two tiles, an odd count
SIZES = [1, 2, 31, 33, 1000, T - 1, T, T + 1, 3 * T + 7, 40 * T + 5, (1 << 20) + 3, 1301 * T + 5]


def pairs(n: int, seed: int):
    xi = inputs.full_range_i32(n, seed)
    xf = inputs.uniform_f32(n, seed + 1)
    packed = np.empty((n, 2), dtype=np.int32)
    packed[:, 0] = xi
    packed[:, 1] = xf.view(np.int32)
    return xi, xf, packed


def check_pairs(got: np.ndarray, xi, xf, exclusive: bool) -> None:
    yi, yf, ya = oracle.scan_pair_i32_f32(xi, xf, exclusive)
    assert np.array_equal(got[:, 0], yi), f"{np.count_nonzero(got[:, 0] != yi)} int32 mismatches"
    gf = got[:, 1].view(np.float32).astype(np.float64)
    bad = np.flatnonzero(~(np.abs(gf - yf) <= FP32_REL * ya + FP32_ABS))
    assert bad.size == 0, f"{bad.size} fp32 fields out of bound, first at {bad[:5]}"


def check_affine(got: np.ndarray, a, b, exclusive: bool) -> None:
    A, B, Aa, Ba = oracle.scan_affine_f32(a, b, exclusive)
    ga = got[:, 0].astype(np.float64)
    gb = got[:, 1].astype(np.float64)
    bad_a = np.flatnonzero(~(np.abs(ga - A) <= FP32_REL * Aa + FP32_ABS))
    bad_b = np.flatnonzero(~(np.abs(gb - B) <= FP32_REL * Ba + FP32_ABS))
    assert bad_a.size == 0, f"{bad_a.size} A out of bound, first at {bad_a[:5]}"
    assert bad_b.size == 0, f"{bad_b.size} B out of bound, first at {bad_b[:5]}"


@pytest.mark.parametrize("exclusive", [False, True], ids=["incl", "excl"])
@pytest.mark.parametrize("inplace", [False, True], ids=["oop", "inplace"])
def test_pair_sizes(exclusive, inplace):
    for k, n in enumerate(SIZES):
        xi, xf, packed = pairs(n, 40 + k)
        t = torch.from_numpy(packed).to(DEV)
        y = api.scan_pairs(t, exclusive=exclusive, inplace=inplace)
        if inplace:
            assert y.data_ptr() == t.data_ptr()
        check_pairs(y.cpu().numpy(), xi, xf, exclusive)


@pytest.mark.parametrize("exclusive", [False, True], ids=["incl", "excl"])
@pytest.mark.parametrize("inplace", [False, True], ids=["oop", "inplace"])
def test_affine_sizes(exclusive, inplace):
    for k, n in enumerate(SIZES):
        a = inputs.uniform_f32(n, 60 + k)
        b = inputs.uniform_f32(n, 80 + k)
        t = torch.from_numpy(np.stack([a, b], axis=1)).to(DEV)
        y = api.scan_affine(t, exclusive=exclusive, inplace=inplace)
        check_affine(y.cpu().numpy(), a, b, exclusive)


def test_affine_long_memory_and_closed_forms():
    n = 20 * T + 11
    # |a| close to 1: each output depends on hundreds of earlier maps
    a = (np.float32(0.95) + np.float32(0.05) * inputs.uniform_f32(n, 7)).astype(np.float32)
    b = inputs.uniform_f32(n, 8)
    y = api.scan_affine(torch.from_numpy(np.stack([a, b], axis=1)).to(DEV)).cpu().numpy()
    check_affine(y, a, b, False)
    # a = 1: B is the running sum of b; exclusive starts with the identity
    ones = np.ones(n, dtype=np.float32)
    y = api.scan_affine(torch.from_numpy(np.stack([ones, b], axis=1)).to(DEV), exclusive=True).cpu().numpy()
    assert y[0, 0] == 1.0 and y[0, 1] == 0.0 and np.all(y[:, 0] == 1.0)
    check_affine(y, ones, b, True)
    # small integers and a = 1: every association order is exact
    bi = inputs.uniform_int(n, -8, 8, 9).astype(np.float32)
    y = api.scan_affine(torch.from_numpy(np.stack([ones, bi], axis=1)).to(DEV)).cpu().numpy()
    assert np.array_equal(y[:, 1], np.cumsum(bi.astype(np.float64)).astype(np.float32))


def test_unaligned_arrays_take_the_fallback_kernel():
    # 8-byte aligned but not 16: one CTA per tile, scalar loads
    n = 9 * T + 77
    xi, xf, packed = pairs(n + 1, 5)
    buf = torch.from_numpy(packed).to(DEV)
    t = buf[1:]
    out = torch.empty((n + 2, 2), dtype=torch.int32, device=DEV)[1:n + 1]
    y = api.scan_pairs(t, out=out)
    check_pairs(y.cpu().numpy(), xi[1:], xf[1:], False)
    a = inputs.uniform_f32(n + 1, 11)
    b = inputs.uniform_f32(n + 1, 12)
    buf = torch.from_numpy(np.stack([a, b], axis=1)).to(DEV)
    for excl in (False, True):
        y = api.scan_affine(buf[1:], exclusive=excl)
        check_affine(y.cpu().numpy(), a[1:], b[1:], excl)


def test_16_byte_but_not_32_byte_aligned():
    # the bulk-copy kernel with an output off a 32-byte boundary: each lane's
    # 32 bytes of a row go out as two 16-byte stores
    n = 7 * T + 19
    xi, xf, packed = pairs(n + 2, 31)
    buf = torch.from_numpy(packed).to(DEV)
    assert buf.data_ptr() % 32 == 0
    out = torch.empty((n + 2, 2), dtype=torch.int32, device=DEV)[2:]
    for excl in (False, True):
        y = api.scan_pairs(buf[2:], exclusive=excl, out=out)
        check_pairs(y.cpu().numpy(), xi[2:], xf[2:], excl)
    a = inputs.uniform_f32(n + 2, 41)
    b = inputs.uniform_f32(n + 2, 42)
    ab = torch.from_numpy(np.stack([a, b], axis=1)).to(DEV)
    for excl in (False, True):
        y = api.scan_affine(ab[2:], exclusive=excl)
        check_affine(y.cpu().numpy(), a[2:], b[2:], excl)


def test_int64_view_and_empty():
    xi, xf, packed = pairs(5000, 21)
    t64 = torch.from_numpy(packed.view(np.int64).reshape(-1)).to(DEV)
    y = api.scan_pairs(t64)
    check_pairs(y.cpu().numpy().view(np.int32).reshape(-1, 2), xi, xf, False)
    e = torch.empty((0, 2), dtype=torch.float32, device=DEV)
    assert api.scan_affine(e).numel() == 0


@pytest.mark.parametrize("kind", ["pairs", "affine"])
def test_full_size_2p27(kind):
    # 2^27 8-byte elements (1 GiB in, 1 GiB out), every output against the
    # oracle
    n = 1 << 27
    if kind == "pairs":
        xi, xf, packed = pairs(n, 31)
        y = api.scan_pairs(torch.from_numpy(packed).to(DEV)).cpu().numpy()
        check_pairs(y, xi, xf, False)
    else:
        a = inputs.uniform_f32(n, 33)
        b = inputs.uniform_f32(n, 34)
        y = api.scan_affine(torch.from_numpy(np.stack([a, b], axis=1)).to(DEV)).cpu().numpy()
        check_affine(y, a, b, False)
    torch.cuda.empty_cache()
