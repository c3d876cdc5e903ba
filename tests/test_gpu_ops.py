"""GPU parity of the max / min scans against the CPU oracle: exact for every
dtype (a running max/min never rounds), fp32 NaN elements skipped."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
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
    x = inputs.uniform_f32(n, seed) * np.float32(1000)
    x[7::4099] = np.nan
    return x


def same(got, want):
    if got.dtype.kind == "f":
        return bool(np.all((got == want) | (np.isnan(got) & np.isnan(want))))
    return bool(np.array_equal(got, want))


@pytest.mark.parametrize("dtype", list(NP))
@pytest.mark.parametrize("op", ["max", "min"])
@pytest.mark.parametrize("exclusive", [False, True], ids=["incl", "excl"])
def test_max_min(dtype, op, exclusive):
    T = api.tile_elements(TT[dtype])
    for k, n in enumerate([1, 2, 33, 1000, T - 1, T, T + 1, 5 * T + 17, (1 << 20) + 3]):
        x = make(dtype, n, 200 + k)
        want = oracle.scan_op(x, op, exclusive)
        got = api.scan(torch.from_numpy(x).to(DEV), exclusive=exclusive, op=op).cpu().numpy()
        assert same(got, want), (n, np.flatnonzero(got != want)[:5])


@pytest.mark.parametrize("dtype", list(NP))
def test_max_min_unaligned_and_in_place(dtype):
    T = api.tile_elements(TT[dtype])
    n = 4 * T + 9
    x = make(dtype, n + 1, 300)
    for op in ("max", "min"):
        t = torch.from_numpy(x).to(DEV)[1:]          # not 16-byte aligned: the one-tile-per-CTA kernel
        got = api.scan(t, op=op).cpu().numpy()
        assert same(got, oracle.scan_op(x[1:], op))
        t = torch.from_numpy(x[:n].copy()).to(DEV)
        api.scan(t, op=op, exclusive=True, inplace=True)
        assert same(t.cpu().numpy(), oracle.scan_op(x[:n], op, True))


def test_max_min_large():
    n = (1 << 26) + 5
    x = inputs.full_range_i32(n, 301)
    t = torch.from_numpy(x).to(DEV)
    for op in ("max", "min"):
        assert same(api.scan(t, op=op).cpu().numpy(), oracle.scan_op(x, op))
    xf = make("float32", n, 302)
    tf = torch.from_numpy(xf).to(DEV)
    assert same(api.scan(tf, op="max", exclusive=True).cpu().numpy(), oracle.scan_op(xf, "max", True))


def test_max_min_all_nan_and_extremes():
    x = np.full(3 * api.tile_elements(torch.float32), np.nan, dtype=np.float32)
    got = api.scan(torch.from_numpy(x).to(DEV), op="max").cpu().numpy()
    assert np.all(got == -np.inf)
    xi = np.array([np.iinfo(np.int64).min, -1, np.iinfo(np.int64).max, 0], dtype=np.int64)
    got = api.scan(torch.from_numpy(xi).to(DEV), op="max").cpu().numpy()
    assert list(got) == [np.iinfo(np.int64).min, -1, np.iinfo(np.int64).max, np.iinfo(np.int64).max]
