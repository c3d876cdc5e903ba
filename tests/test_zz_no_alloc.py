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
so that anything the first left in the shared scratch would show.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

from prefix_scan_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from prefix_scan_gb300 import _lib, api  # noqa: E402

DEV = torch.device("cuda:0")


def _noalloc(t: torch.Tensor, out: torch.Tensor) -> int:
    lib = _lib.load()
    s = ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)
    return lib.ps_scan_inclusive_i32_noalloc(t.data_ptr(), out.data_ptr(), t.numel(), s)


def test_noalloc_matches_regular_entry_point_twice_in_a_row():
    T = api.tile_elements(torch.int32)
    for n in ((1 << 22) + 4097, 5 * T + 13):     # second call shorter than the first
        x = torch.from_numpy(inputs.full_range_i32(n, 424242 + n)).to(DEV)
        want = api.scan_inclusive(x)             # regular entry point, own workspace
        got = torch.empty_like(x)
        assert _noalloc(x, got) == _lib.PS_OK
        torch.cuda.synchronize()
        assert torch.equal(got, want), n


def test_noalloc_in_place_and_empty():
    n = 3 * api.tile_elements(torch.int32) + 5
    host = inputs.uniform_int(n, -50, 50, 77)
    x = torch.from_numpy(host).to(DEV)
    want = api.scan_inclusive(x.clone())
    assert _noalloc(x, x) == _lib.PS_OK           # in == out: in place
    torch.cuda.synchronize()
    assert torch.equal(x, want)
    e = torch.empty(0, dtype=torch.int32, device=DEV)
    assert _noalloc(e, e) == _lib.PS_OK


def test_noalloc_largest_accepted_size():
    # n exactly at the limit must fit the fixed scratch
    n = _lib.PS_NOALLOC_MAX_ELEMENTS
    x = torch.from_numpy(inputs.uniform_int(n, -3, 3, 99)).to(DEV)
    want = api.scan_inclusive(x)
    assert _noalloc(x, x) == _lib.PS_OK
    torch.cuda.synchronize()
    assert torch.equal(x, want)
    del x, want
    torch.cuda.empty_cache()


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
