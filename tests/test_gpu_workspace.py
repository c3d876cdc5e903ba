"""The workspace across calls: zero-filled once, never reset by a call.

Descriptors carry the number (epoch) of the call that wrote them, and each
call leaves the header ready for the next: tile counter and done count back
at 0, epoch advanced (by the last CTA to take a tile id, or, in the call
before an epoch wrap, by the last CTA to finish).
These tests drive one workspace through many calls of mixed lengths,
dtypes and algorithms, a workspace that was never zero-filled, and the
epoch wrap-around, always checking the results against the oracle.
"""
from __future__ import annotations

import ctypes
import struct

import numpy as np
import pytest

import oracle
from conftest import fp32_ok
from prefix_scan_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from prefix_scan_gb300 import _lib, api  # noqa: E402

DEV = torch.device("cuda:0")
EPOCH_MASK = (1 << 30) - 1


def epoch_of(ws) -> int:
    e = ctypes.c_uint32(0)
    _lib.check("ps_testing_workspace_epoch",
               _lib.load().ps_testing_workspace_epoch(ws.data_ptr(), None, ctypes.byref(e)))
    return e.value


def set_epoch(ws, epoch: int) -> None:
    _lib.check("ps_testing_set_workspace_epoch",
               _lib.load().ps_testing_set_workspace_epoch(ws.data_ptr(), epoch, None))


def header(ws) -> dict:
    """The workspace header as the library lays it out: u64 tile counter,
    u64 status, u64 capacity, u32 done count, u32 epoch, u32 magic."""
    raw = ws[:36].cpu().numpy().tobytes()
    tc, status, cap, done, epoch, magic = struct.unpack_from("<QQQIII", raw)
    return {"tile_counter": tc, "status": status, "capacity": cap, "done": done, "epoch": epoch, "magic": magic}


def check(y, x, exclusive):
    if x.dtype == np.float32:
        assert fp32_ok(y, x, exclusive).all()
    else:
        ref = oracle.exclusive(x) if exclusive else oracle.inclusive(x)
        assert np.array_equal(y, ref)


def test_one_workspace_many_calls_mixed():
    big = 1 << 22
    ws = api.alloc_workspace(torch.int32, big, DEV)   # largest need: int32, n = 2^22
    assert epoch_of(ws) == 0
    plan = [  # (dtype, n, exclusive, algo, inplace)
        ("int32", big, False, "decoupled", False),
        ("int32", 5000, True, "decoupled", False),       # shorter: stale descriptors beyond
        ("int64", big // 2, False, "decoupled", True),   # another descriptor format
        ("float32", 123_457, False, "decoupled", False),
        ("int32", big, True, "reduce_then_scan", False),  # does not touch the descriptors
        ("int32", big, False, "decoupled", False),        # long again, over stale slots
        ("int64", 77_777, True, "chained", False),
        ("int32", 3, False, "decoupled", True),
        ("int32", big - 1, True, "decoupled", False),
    ]
    expected_epoch = 0
    for k, (dt, n, excl, algo, inplace) in enumerate(plan):
        x = (inputs.full_range_i32(n, 70 + k) if dt == "int32"
             else inputs.hashes(n, 70 + k).view(np.int64) if dt == "int64"
             else inputs.uniform_f32(n, 70 + k))
        t = torch.from_numpy(x.copy()).to(DEV)
        y = api.scan(t, exclusive=excl, algo=algo, inplace=inplace, workspace=ws)
        check(y.cpu().numpy(), x, excl)
        tdt = {"int32": torch.int32, "int64": torch.int64, "float32": torch.float32}[dt]
        small = n <= 2 * api.tile_elements(tdt)   # one CTA, no look-back: the header is left as it is
        if algo != "reduce_then_scan" and not small:
            expected_epoch += 1
        assert epoch_of(ws) == expected_epoch, (k, dt, algo)
        assert api.device_status(ws) == _lib.PS_OK


def test_workspace_never_zero_filled_refuses_to_run():
    n = 50_000
    ws = torch.full((api.workspace_size(torch.int32, n),), 0xAB, dtype=torch.uint8, device=DEV)
    x = torch.ones(n, dtype=torch.int32, device=DEV)
    out = torch.full_like(x, -7)
    api.scan_inclusive(x, out=out, workspace=ws)        # enqueued, does nothing on the device
    assert api.device_status(ws) == _lib.PS_ERR_WORKSPACE_NOT_INITIALIZED
    assert torch.all(out == -7)
    _lib.check("ps_workspace_init", _lib.load().ps_workspace_init(ws.data_ptr(), ws.numel(), None))
    api.scan_inclusive(x, out=out, workspace=ws)
    assert api.device_status(ws) == _lib.PS_OK
    assert torch.equal(out, torch.arange(1, n + 1, dtype=torch.int32, device=DEV))


def test_short_arrays_leave_the_workspace_alone_and_respect_an_unzeroed_one():
    # up to two tiles one CTA scans the array without touching the header
    ws = api.alloc_workspace(torch.int32, 1 << 20, DEV)
    for n in (1, 1000, 2 * api.tile_elements(torch.int32)):
        x = inputs.full_range_i32(n, 90 + n)
        y = api.scan_inclusive(torch.from_numpy(x).to(DEV), workspace=ws).cpu().numpy()
        assert np.array_equal(y, oracle.inclusive(x))
        assert epoch_of(ws) == 0 and api.device_status(ws) == _lib.PS_OK
    bad = torch.full((api.workspace_size(torch.int32, 1000),), 0xAB, dtype=torch.uint8, device=DEV)
    x = torch.ones(1000, dtype=torch.int32, device=DEV)
    out = torch.full_like(x, -7)
    api.scan_inclusive(x, out=out, workspace=bad)
    assert api.device_status(bad) == _lib.PS_ERR_WORKSPACE_NOT_INITIALIZED
    assert torch.all(out == -7)


def _plant_stale_descriptors(ws, code: int, epoch: int, count: int) -> None:
    """Write descriptors that claim P with a wrong value, tagged `epoch`, into
    the first `count` slots (what a call 2^30 calls earlier could have left)."""
    lib = _lib.load()
    db = lib.ps_testing_descriptor_bytes(code)
    raw = bytearray(db * count)
    v = np.array([123456789], dtype=np.int64 if code == 1 else np.int32)
    buf = (ctypes.c_char * db)()
    assert lib.ps_testing_encode_descriptor(code, 2, epoch, v.ctypes.data, buf) == 0
    for k in range(count):
        raw[k * db:(k + 1) * db] = bytes(buf)
    ws[256:256 + len(raw)].copy_(torch.frombuffer(raw, dtype=torch.uint8))


@pytest.mark.parametrize("dtype", ["int32", "int64"])
def test_epoch_wraparound_clears_stale_descriptors(dtype):
    tdt = torch.int32 if dtype == "int32" else torch.int64
    code = 0 if dtype == "int32" else 1
    n = 200 * api.tile_elements(tdt) + 17
    ws = api.alloc_workspace(tdt, n, DEV)
    x0 = torch.ones(n, dtype=tdt, device=DEV)
    api.scan_inclusive(x0, workspace=ws)                # the workspace is in use now
    torch.cuda.synchronize()
    # descriptors of epoch 0 that a look-back at epoch 0 would trust
    _plant_stale_descriptors(ws, code, 0, 200)
    set_epoch(ws, EPOCH_MASK)                           # the next call is the last before the wrap
    m = 3 * api.tile_elements(tdt) + 1                  # long enough for the look-back kernel
    ones = torch.ones(m, dtype=tdt, device=DEV)
    assert torch.equal(api.scan_inclusive(ones, workspace=ws).cpu(), torch.arange(1, m + 1, dtype=tdt))
    assert epoch_of(ws) == 0
    # epoch 0 again: a wrong value planted above would now be read unless cleared
    xs = (inputs.full_range_i32(n, 5) if dtype == "int32" else inputs.hashes(n, 5).view(np.int64))
    y = api.scan_inclusive(torch.from_numpy(xs).to(DEV), workspace=ws).cpu().numpy()
    assert np.array_equal(y, oracle.inclusive(xs))
    assert epoch_of(ws) == 1 and api.device_status(ws) == _lib.PS_OK


def test_stale_descriptors_of_other_epochs_are_ignored():
    n = 64 * api.tile_elements(torch.int32)
    ws = api.alloc_workspace(torch.int32, n, DEV)
    m = 3 * api.tile_elements(torch.int32) + 1         # long enough for the look-back kernel
    for e in (1, 2, 3):
        api.scan_inclusive(torch.ones(m, dtype=torch.int32, device=DEV), workspace=ws)
    torch.cuda.synchronize()
    assert epoch_of(ws) == 3
    _plant_stale_descriptors(ws, 0, 2, 64)             # written "two calls ago"
    x = inputs.full_range_i32(n, 6)
    y = api.scan_inclusive(torch.from_numpy(x).to(DEV), workspace=ws).cpu().numpy()
    assert np.array_equal(y, oracle.inclusive(x))


def test_every_kernel_leaves_the_header_ready_for_the_next_call():
    # The persistent scan, select, partition, reduce-by-key and run-length
    # encoding ready the header when their last CTA takes its last tile id,
    # while other CTAs may still be storing; the one-tile-per-CTA fallback
    # when its last CTA finishes.  After each: counter and done count 0,
    # epoch + 1, and the results right -- including calls that run right
    # after one another.
    n = (1 << 21) + 77
    need = max(api.workspace_size(torch.int32, n), api.reduce_by_key_workspace_size(torch.int32, n))
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    x = inputs.full_range_i32(n + 1, 31)
    xt = torch.from_numpy(x).to(DEV)
    f = inputs.bernoulli_half(n, 32).astype(np.uint8)
    ft = torch.from_numpy(f).to(DEV)
    k = inputs.run_keys(n, 16, 33)
    kt = torch.from_numpy(k).to(DEV)
    epoch = 0
    for rep in range(2):
        y = api.scan(xt[:n], workspace=ws)                          # persistent kernel
        epoch += 1
        assert header(ws) == {"tile_counter": 0, "status": 0, "capacity": need, "done": 0,
                              "epoch": epoch, "magic": 0x50534742}, rep
        assert np.array_equal(y.cpu().numpy(), oracle.inclusive(x[:n]))
        y = api.scan(xt[1:], exclusive=True, workspace=ws)         # 4-byte offset: fallback kernel
        epoch += 1
        assert np.array_equal(y.cpu().numpy(), oracle.exclusive(x[1:]))
        sel, cnt = api.select(xt[:n], ft, workspace=ws)
        epoch += 1
        want = oracle.select(x[:n], f)
        assert int(cnt.item()) == want.shape[0] and np.array_equal(sel[:want.shape[0]].cpu().numpy(), want)
        part, cnt = api.partition(xt[:n], ft, workspace=ws)
        epoch += 1
        assert int(cnt.item()) == want.shape[0] and np.array_equal(part[:want.shape[0]].cpu().numpy(), want)
        uk, agg, runs = api.reduce_by_key(kt, xt[:n], workspace=ws)
        epoch += 1
        ok_k, ok_v = oracle.reduce_by_key(k, x[:n])
        r = int(runs.item())
        assert r == ok_k.shape[0] and np.array_equal(uk[:r].cpu().numpy(), ok_k)
        assert np.array_equal(agg[:r].cpu().numpy(), ok_v)
        uk, lens, runs = api.run_length_encode(kt, workspace=ws)
        epoch += 1
        lk, lc = oracle.reduce_by_key(k, None)
        r = int(runs.item())
        assert r == lk.shape[0] and np.array_equal(uk[:r].cpu().numpy(), lk)
        assert np.array_equal(lens[:r].cpu().numpy(), lc)
        h = header(ws)
        assert (h["tile_counter"], h["done"], h["epoch"]) == (0, 0, epoch), rep
        assert api.device_status(ws) == _lib.PS_OK
    # the call before the wrap: the last CTA to finish clears and readies
    set_epoch(ws, EPOCH_MASK)
    y = api.scan(xt[:n], exclusive=True, workspace=ws)
    h = header(ws)
    assert (h["tile_counter"], h["done"], h["epoch"]) == (0, 0, 0)
    assert np.array_equal(y.cpu().numpy(), oracle.exclusive(x[:n]))
    sel, cnt = api.select(xt[:n], ft, workspace=ws)
    h = header(ws)
    assert (h["tile_counter"], h["done"], h["epoch"]) == (0, 0, 1)
    assert int(cnt.item()) == want.shape[0] and np.array_equal(sel[:want.shape[0]].cpu().numpy(), want)
    # and run-length encoding as the call before a wrap
    set_epoch(ws, EPOCH_MASK)
    for want_epoch in (0, 1):
        uk, lens, runs = api.run_length_encode(kt, workspace=ws)
        h = header(ws)
        assert (h["tile_counter"], h["done"], h["epoch"]) == (0, 0, want_epoch)
        r = int(runs.item())
        assert r == lk.shape[0] and np.array_equal(uk[:r].cpu().numpy(), lk)
        assert np.array_equal(lens[:r].cpu().numpy(), lc)
    assert api.device_status(ws) == _lib.PS_OK
