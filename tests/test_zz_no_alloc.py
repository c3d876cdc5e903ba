"""The allocation-free int32 inclusive scan against the regular entry point.

ps_scan_inclusive_i32_noalloc serves callers that cannot allocate device
memory (allocator callbacks, plug-ins whose host owns all device memory,
paths that must never reach the allocator): its look-back scratch is a fixed
array inside the library instead of a caller workspace.  This file is named
so that pytest collects it last; it must pass on its own in a fresh process
and after every other test.

Both calls go through the C ABI; the result must equal the regular
ps_scan_inclusive_i32 result bit for bit (the tolerance every int32 test
here uses), on two calls in a row -- the second one shorter than the first,
so that anything the first left in the shared scratch would show -- and the
CPU oracle's running sum element by element (so a fault that both entry
points share, such as one in the fixed scratch's geometry, shows too).
After every call the device-side status in the scratch array must be PS_OK.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

import oracle
from prefix_scan_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from prefix_scan_gb300 import _lib, api  # noqa: E402

DEV = torch.device("cuda:0")


def _stream() -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)


def _noalloc(t: torch.Tensor, out: torch.Tensor) -> int:
    lib = _lib.load()
    return lib.ps_scan_inclusive_i32_noalloc(t.data_ptr(), out.data_ptr(), t.numel(), _stream())


def _scratch_status() -> int:
    """Device-side status of the last allocation-free call (waits for it)."""
    lib = _lib.load()
    ptr = ctypes.c_void_p()
    _lib.check("ps_testing_noalloc_scratch", lib.ps_testing_noalloc_scratch(ctypes.byref(ptr), _stream()))
    st = ctypes.c_int(-1)
    _lib.check("ps_get_device_status", lib.ps_get_device_status(ptr, _stream(), ctypes.byref(st)))
    return st.value


def test_noalloc_matches_regular_entry_point_and_oracle_twice_in_a_row():
    T = api.tile_elements(torch.int32)
    for n in ((1 << 22) + 4097, 5 * T + 13):     # second call shorter than the first
        host = inputs.full_range_i32(n, 424242 + n)
        x = torch.from_numpy(host).to(DEV)
        want = api.scan_inclusive(x)             # regular entry point, own workspace
        got = torch.empty_like(x)
        assert _noalloc(x, got) == _lib.PS_OK
        torch.cuda.synchronize()
        assert _scratch_status() == _lib.PS_OK
        assert torch.equal(got, want), n
        ref = oracle.inclusive(host)             # wraps modulo 2^32, bit for bit
        bad = np.flatnonzero(got.cpu().numpy() != ref)
        assert bad.size == 0, (n, bad[:5])


def test_noalloc_in_place_and_empty():
    n = 3 * api.tile_elements(torch.int32) + 5
    host = inputs.uniform_int(n, -50, 50, 77)
    x = torch.from_numpy(host).to(DEV)
    want = api.scan_inclusive(x.clone())
    assert _noalloc(x, x) == _lib.PS_OK           # in == out: in place
    torch.cuda.synchronize()
    assert _scratch_status() == _lib.PS_OK
    assert torch.equal(x, want)
    assert np.array_equal(x.cpu().numpy(), oracle.inclusive(host))
    e = torch.empty(0, dtype=torch.int32, device=DEV)
    assert _noalloc(e, e) == _lib.PS_OK


def test_noalloc_largest_accepted_size():
    # n exactly at the limit must fit the fixed scratch; full-range values
    # wrap modulo 2^32 all along
    n = _lib.PS_NOALLOC_MAX_ELEMENTS
    host = inputs.full_range_i32(n, 99)
    x = torch.from_numpy(host).to(DEV)
    want = api.scan_inclusive(x)
    assert _noalloc(x, x) == _lib.PS_OK
    torch.cuda.synchronize()
    assert _scratch_status() == _lib.PS_OK
    assert torch.equal(x, want)
    got = x.cpu().numpy()
    del x, want
    torch.cuda.empty_cache()
    ref = oracle.inclusive(host)
    bad = np.flatnonzero(got != ref)
    assert bad.size == 0, bad[:5]


def test_noalloc_rejects_sizes_beyond_its_scratch():
    n = _lib.PS_NOALLOC_MAX_ELEMENTS + 1
    # a real buffer of that length, so nothing could go out of bounds even if
    # the check were missing; the call must refuse before enqueuing anything
    x = torch.zeros(n, dtype=torch.int32, device=DEV)
    x[-1] = 7
    assert _noalloc(x, x) == _lib.PS_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert x[-1].item() == 7 and x[0].item() == 0
    del x
    torch.cuda.empty_cache()
    assert np.dtype(np.int32).itemsize == 4
