"""GPU parity at the full workload sizes, through the same C-ABI call the
bench times: int32 2^20, fp32 2^24, int32 exclusive 2^28 (0/1 flags),
int64 2^29, and the in-place int32 length sweep up to 2^30.  Every output
element is compared with the oracle.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from conftest import fp32_ok
from prefix_scan_gb300 import workloads

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from prefix_scan_gb300 import api  # noqa: E402

DEV = torch.device("cuda:0")


def _run_and_check(w: workloads.Workload, n: int) -> None:
    x = w.make(n)
    t = torch.from_numpy(x).to(DEV)
    y = api.scan(t, exclusive=w.exclusive, inplace=w.inplace)
    if w.inplace:
        assert y.data_ptr() == t.data_ptr()
    got = y.cpu().numpy()
    del t, y
    if x.dtype == np.float32:
        bad = np.flatnonzero(~fp32_ok(got, x, w.exclusive))
        assert bad.size == 0, f"{w.name} n={n}: {bad.size} fp32 elements out of bound"
    else:
        ref = oracle.exclusive(x) if w.exclusive else oracle.inclusive(x)
        bad = np.flatnonzero(got != ref)
        assert bad.size == 0, f"{w.name} n={n}: {bad.size} mismatches, first at {bad[:5]}"
    if w.dist == "bern" and w.exclusive:
        # compaction offsets: non-decreasing, last + last flag = popcount
        assert np.all(np.diff(got) >= 0)
        assert int(got[-1]) + int(x[-1]) == int(x.sum())
    torch.cuda.empty_cache()


@pytest.mark.parametrize("w", [workloads.SMALL_I32, workloads.F32_2P24, workloads.I32_EXCL_2P28,
                               workloads.I64_2P29], ids=lambda w: w.name)
def test_workload_full_size(w):
    _run_and_check(w, w.n)


@pytest.mark.parametrize("n", workloads.I32_INPLACE_SWEEP.sweep)
def test_inplace_length_sweep(n):
    _run_and_check(workloads.I32_INPLACE_SWEEP, n)


def test_inclusive_scan_above_2p31_elements():
    # 2^31 + 12345 ones scanned in place: y[i] = i + 1 modulo 2^32 (as int32),
    # past the 2^31 mark where 32-bit signed indices would overflow; checked
    # on the device in chunks.
    n, step = (1 << 31) + 12345, 1 << 28
    x = torch.ones(n, dtype=torch.int32, device=DEV)
    api.scan(x, inplace=True)
    for s in range(0, n, step):
        i = torch.arange(s, min(n, s + step), dtype=torch.int64, device=DEV) + 1
        want = (i - (i >= 2 ** 31).to(torch.int64) * 2 ** 32).to(torch.int32)
        assert torch.equal(x[s:s + i.numel()], want)
    del x
    torch.cuda.empty_cache()


def test_scans_past_2p32_elements_and_int64_past_2p31():
    # 2^32 + 5 int32 ones in place (y[i] = i + 1 modulo 2^32: element and tile
    # indices past 32 bits), and 2^31 + 5 int64 ones (y[i] = i + 1 exactly);
    # each checked on the device in chunks against the closed form
    step = 1 << 28
    n = (1 << 32) + 5
    x = torch.ones(n, dtype=torch.int32, device=DEV)
    api.scan(x, inplace=True)
    for s in range(0, n, step):
        i = torch.arange(s, min(n, s + step), dtype=torch.int64, device=DEV) + 1
        want = (i % (1 << 32))
        want = (want - (want >= 2 ** 31).to(torch.int64) * 2 ** 32).to(torch.int32)
        assert torch.equal(x[s:s + i.numel()], want), s
    del x
    torch.cuda.empty_cache()
    n = (1 << 31) + 5
    x = torch.ones(n, dtype=torch.int64, device=DEV)
    y = api.scan_inclusive(x)
    del x
    for s in range(0, n, step):
        i = torch.arange(s, min(n, s + step), dtype=torch.int64, device=DEV) + 1
        assert torch.equal(y[s:s + i.numel()], i), s
    del y
    torch.cuda.empty_cache()
