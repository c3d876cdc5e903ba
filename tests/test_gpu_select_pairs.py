"""Select and partition from a build with the paired-tile select kernel.

That kernel (a compile-time option of csrc/scan_select.cu, off in the
product build because it measured slower) runs the two CTAs of a cluster on
two consecutive tiles as one unit: one claim, one descriptor and one
look-back per unit, the partner's count and its tile's offset exchanged
through distributed shared memory.  Every result is compared with the
oracle exactly: lengths of one tile and less, odd and even tile counts (an
odd count leaves the second CTA an empty tile in the last unit), the
predicate forms, int64 and fp32 values, in place, and repeated runs over
thousands of units.
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

from prefix_scan_gb300 import _lib  # noqa: E402
from prefix_scan_gb300 import build as nvbuild  # noqa: E402

DEV = torch.device("cuda:0")
CODES = {np.dtype(np.int32): _lib.PS_INT32, np.dtype(np.int64): _lib.PS_INT64,
         np.dtype(np.float32): _lib.PS_FLOAT32}
OPS = {"flagged": _lib.PS_SELECT_FLAGGED, "nonzero": _lib.PS_SELECT_NONZERO,
       "greater": _lib.PS_SELECT_GREATER, "less": _lib.PS_SELECT_LESS}


@pytest.fixture(scope="module")
def paired():
    path = nvbuild.build_variant("select_pairs", {"PS_SEL_PAIR": 1})
    lib = ctypes.CDLL(str(path))
    for name, (res, args) in _lib.SIGNATURES.items():
        if "noalloc" in name:
            continue   # not in this build
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    return lib


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)


def _values(dt, n: int, seed: int) -> np.ndarray:
    if dt == np.float32:
        x = inputs.uniform_f32(n, seed)
        x[::97] = 0.0
        return x
    return inputs.uniform_int(n, -100, 100, seed, dt)


def _call(lib, fname: str, x: np.ndarray, op: str, f, t, inplace: bool = False):
    """(out on the host, count, device status) of one ps_select / ps_partition."""
    n = x.shape[0]
    code = CODES[x.dtype]
    xt = torch.from_numpy(x.copy()).to(DEV)
    ft = torch.from_numpy(f).to(DEV) if f is not None else None
    out = xt if inplace else torch.zeros_like(xt)
    cnt = torch.zeros(1, dtype=torch.int64, device=DEV)
    ws = torch.zeros(max(int(lib.ps_scan_workspace_size(code, n)), 16), dtype=torch.uint8, device=DEV)
    thr = np.array([t if t is not None else 0], dtype=x.dtype)
    st = getattr(lib, fname)(code, OPS[op], xt.data_ptr(), ft.data_ptr() if ft is not None else None,
                             thr.ctypes.data if op in ("greater", "less") else None, out.data_ptr(),
                             cnt.data_ptr(), n, ws.data_ptr(), ws.numel(), _stream())
    assert st == _lib.PS_OK, (fname, st)
    dst = ctypes.c_int(-1)
    assert lib.ps_get_device_status(ws.data_ptr(), _stream(), ctypes.byref(dst)) == _lib.PS_OK
    return out.cpu().numpy(), int(cnt.item()), dst.value


def _check(lib, x: np.ndarray, op: str, f, t):
    flags = f if op == "flagged" else oracle.flags(x, op, t if t is not None else 0)
    want = oracle.select(x, flags)
    got, cnt, st = _call(lib, "ps_select", x, op, f, t)
    assert st == _lib.PS_OK and cnt == want.shape[0]
    assert np.array_equal(got[:cnt], want)
    pw, pk = oracle.partition(x, flags)
    got, cnt, st = _call(lib, "ps_partition", x, op, f, t)
    assert st == _lib.PS_OK and cnt == pk
    assert np.array_equal(got, pw)


@pytest.mark.parametrize("dt", [np.int32, np.int64, np.float32])
def test_tile_counts(paired, dt):
    tile = int(paired.ps_tile_elements(CODES[np.dtype(dt)]))
    for k, n in enumerate([1, 31, tile - 1, tile, tile + 1, 2 * tile, 3 * tile - 5, 3 * tile, 5 * tile + 17,
                           (1 << 20) + 3]):
        x = _values(dt, n, 300 + k)
        f = inputs.bernoulli_half(n, 400 + k).astype(np.uint8)
        _check(paired, x, "flagged", f, None)


@pytest.mark.parametrize("op", ["nonzero", "greater", "less"])
def test_predicates(paired, op):
    n = 7 * 8192 + 123
    for dt in (np.int32, np.int64, np.float32):
        x = _values(dt, n, 500)
        _check(paired, x, op, None, 3)


def test_in_place(paired):
    n = (1 << 21) + 9
    x = inputs.uniform_int(n, -100, 100, 600, np.int32)
    f = inputs.bernoulli_half(n, 601).astype(np.uint8)
    got, cnt, st = _call(paired, "ps_select", x, "flagged", f, None, inplace=True)
    want = oracle.select(x, f)
    assert st == _lib.PS_OK and cnt == want.shape[0]
    assert np.array_equal(got[:cnt], want)


def test_repeated(paired):
    # 2^22 + 5 int32 elements: 513 tiles, 257 units (the last one half empty)
    n = (1 << 22) + 5
    x = inputs.full_range_i32(n, 700)
    f = inputs.bernoulli_half(n, 701).astype(np.uint8)
    want_sel = torch.from_numpy(oracle.select(x, f)).to(DEV)
    want_part, kept = oracle.partition(x, f)
    want_part = torch.from_numpy(want_part).to(DEV)
    xt, ft = torch.from_numpy(x).to(DEV), torch.from_numpy(f).to(DEV)
    o = torch.empty_like(xt)
    cnt = torch.zeros(1, dtype=torch.int64, device=DEV)
    ws = torch.zeros(max(int(paired.ps_scan_workspace_size(_lib.PS_INT32, n)), 16), dtype=torch.uint8, device=DEV)
    for k in range(40):
        for fname in ("ps_select", "ps_partition"):
            st = getattr(paired, fname)(_lib.PS_INT32, _lib.PS_SELECT_FLAGGED, xt.data_ptr(), ft.data_ptr(), None,
                                        o.data_ptr(), cnt.data_ptr(), n, ws.data_ptr(), ws.numel(), _stream())
            assert st == _lib.PS_OK
            assert int(cnt.item()) == kept, (fname, k)
            assert torch.equal(o[:kept], want_sel) if fname == "ps_select" else torch.equal(o, want_part), (fname, k)
    dst = ctypes.c_int(-1)
    assert paired.ps_get_device_status(ws.data_ptr(), _stream(), ctypes.byref(dst)) == _lib.PS_OK
    assert dst.value == _lib.PS_OK
