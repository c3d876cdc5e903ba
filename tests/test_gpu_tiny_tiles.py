"""Scans, pair scans, select, reduce-by-key and run-length encoding from a
tiny-tile build of the library.

A second copy of the library is built with the smallest tile geometry the
scan and select kernels accept (four elements per thread: tiles of 1024
elements instead of 8192 / 4096), so the same array makes eight times as
many tiles, and so eight times as many descriptor publishes, look-backs and
role hand-offs per byte.  That is where a wrong ordering of a descriptor's
words (or of a hand-off) would show as a rare mismatch, so each case runs
100 times over thousands of tiles, every run against the oracle: integers
bit for bit, fp32 within FP32_REL * sum|x| + FP32_ABS of the fp64 result.
The build's look-back also reads two descriptors per lane, so the affine
maps and the segmented sum of reduce-by-key (operators that are not
commutative) check that a window is folded in sequence order.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

import oracle
from conftest import FP32_ABS, FP32_REL
from prefix_scan_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from prefix_scan_gb300 import _lib  # noqa: E402
from prefix_scan_gb300 import build as nvbuild  # noqa: E402

DEV = torch.device("cuda:0")
REPEATS = 100
N = (1 << 22) + 5          # 4097 tiles of 1024 elements
CODES = {torch.int32: _lib.PS_INT32, torch.int64: _lib.PS_INT64, torch.float32: _lib.PS_FLOAT32}


@pytest.fixture(scope="module")
def tiny():
    path = nvbuild.build_variant("tiny", nvbuild.TINY_TILE_DEFINES)
    lib = ctypes.CDLL(str(path))
    for name, (res, args) in _lib.SIGNATURES.items():
        if "noalloc" in name:
            continue   # not in this build
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    for code in CODES.values():
        assert lib.ps_tile_elements(code) == 1024
    return lib


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream(DEV).cuda_stream)


def _workspace(lib, code: int, n: int) -> torch.Tensor:
    return torch.zeros(max(int(lib.ps_scan_workspace_size(code, n)), 16), dtype=torch.uint8, device=DEV)


def _status(lib, ws: torch.Tensor) -> int:
    st = ctypes.c_int(-1)
    assert lib.ps_get_device_status(ws.data_ptr(), _stream(), ctypes.byref(st)) == 0
    return st.value


def _scan(lib, x: torch.Tensor, out: torch.Tensor, ws: torch.Tensor, exclusive: bool) -> None:
    st = lib.ps_scan(_lib.PS_ALGO_DECOUPLED_LOOKBACK, CODES[x.dtype], int(exclusive), x.data_ptr(),
                     out.data_ptr(), x.numel(), ws.data_ptr(), ws.numel(), _stream())
    assert st == _lib.PS_OK, st


def _host(dtype: torch.dtype, n: int, seed: int) -> np.ndarray:
    if dtype == torch.int32:
        return inputs.full_range_i32(n, seed)
    if dtype == torch.int64:
        return inputs.hashes(n, seed).view(np.int64)
    return inputs.uniform_f32(n, seed)


@pytest.mark.parametrize("exclusive", [False, True], ids=["incl", "excl"])
@pytest.mark.parametrize("dtype", [torch.int32, torch.int64, torch.float32], ids=["i32", "i64", "f32"])
def test_scans_repeated(tiny, dtype, exclusive):
    # first a sweep of lengths across tile edges, then 100 runs at 4097 tiles
    T = 1024
    for n in (T - 1, T + 1, 3 * T, 17 * T + 3, 16384 + 1, 333 * T + 77):
        h = _host(dtype, n, 500 + n)
        x = torch.from_numpy(h).to(DEV)
        o = torch.empty_like(x)
        ws = _workspace(tiny, CODES[dtype], n)
        _scan(tiny, x, o, ws, exclusive)
        ref = oracle.exclusive(h) if exclusive else oracle.inclusive(h)
        _compare(o.cpu().numpy(), ref, h, exclusive, n)
    h = _host(dtype, N, 41)
    x = torch.from_numpy(h).to(DEV)
    o = torch.empty_like(x)
    ws = _workspace(tiny, CODES[dtype], N)
    ref = torch.from_numpy(oracle.exclusive(h) if exclusive else oracle.inclusive(h)).to(DEV)
    tol = None
    if dtype == torch.float32:
        tol = torch.from_numpy(FP32_REL * oracle.abs_prefix(h, exclusive) + FP32_ABS).to(DEV)
    for k in range(REPEATS):
        _scan(tiny, x, o, ws, exclusive)
        if tol is None:
            assert torch.equal(o, ref), k
        else:
            assert bool(((o.double() - ref).abs() <= tol).all()), k
    assert _status(tiny, ws) == _lib.PS_OK


def _compare(y: np.ndarray, ref: np.ndarray, x: np.ndarray, exclusive: bool, n: int) -> None:
    if x.dtype == np.float32:
        bound = FP32_REL * oracle.abs_prefix(x, exclusive) + FP32_ABS
        bad = np.flatnonzero(~(np.abs(y.astype(np.float64) - ref) <= bound))
    else:
        bad = np.flatnonzero(y != ref)
    assert bad.size == 0, (n, bad[:5])


def test_pair_and_affine_scans_repeated(tiny):
    xi, xf = inputs.full_range_i32(N, 42), inputs.uniform_f32(N, 43)
    packed = np.empty((N, 2), dtype=np.int32)
    packed[:, 0], packed[:, 1] = xi, xf.view(np.int32)
    a, b = inputs.uniform_f32(N, 44), inputs.uniform_f32(N, 45)
    cases = []
    yi, yf, ya = oracle.scan_pair_i32_f32(xi, xf, False)
    ri, rf = torch.from_numpy(yi).to(DEV), torch.from_numpy(yf).to(DEV)
    tf = torch.from_numpy(FP32_REL * ya + FP32_ABS).to(DEV)
    cases.append(("ps_scan_pair_i32_f32", torch.from_numpy(packed).to(DEV),
                  lambda o: torch.equal(o[:, 0], ri)
                  and bool(((o[:, 1].view(torch.float32).double() - rf).abs() <= tf).all())))
    A_, B_, Aa, Ba = oracle.scan_affine_f32(a, b, False)
    rA, rB = torch.from_numpy(A_).to(DEV), torch.from_numpy(B_).to(DEV)
    tA, tB = torch.from_numpy(FP32_REL * Aa + FP32_ABS).to(DEV), torch.from_numpy(FP32_REL * Ba + FP32_ABS).to(DEV)
    cases.append(("ps_scan_affine_f32", torch.from_numpy(np.stack([a, b], axis=1)).to(DEV),
                  lambda o: bool(((o[:, 0].double() - rA).abs() <= tA).all())
                  and bool(((o[:, 1].double() - rB).abs() <= tB).all())))
    ws = _workspace(tiny, _lib.PS_INT64, N)
    for fname, x, ok in cases:
        o = torch.empty_like(x)
        for k in range(REPEATS):
            st = getattr(tiny, fname)(0, x.data_ptr(), o.data_ptr(), N, ws.data_ptr(), ws.numel(), _stream())
            assert st == _lib.PS_OK
            assert ok(o), (fname, k)
    assert _status(tiny, ws) == _lib.PS_OK


def test_select_and_partition_repeated(tiny):
    x = inputs.full_range_i32(N, 46)
    f = inputs.bernoulli_half(N, 47).astype(np.uint8)
    want_sel = oracle.select(x, f)
    want_part, kept = oracle.partition(x, f)
    xt, ft = torch.from_numpy(x).to(DEV), torch.from_numpy(f).to(DEV)
    o = torch.empty_like(xt)
    cnt = torch.zeros(1, dtype=torch.int64, device=DEV)
    ws = _workspace(tiny, _lib.PS_INT32, N)
    rs, rp = torch.from_numpy(want_sel).to(DEV), torch.from_numpy(want_part).to(DEV)
    m = want_sel.shape[0]
    assert m == kept
    for k in range(REPEATS):
        for fname in ("ps_select", "ps_partition"):
            st = getattr(tiny, fname)(_lib.PS_INT32, _lib.PS_SELECT_FLAGGED, xt.data_ptr(), ft.data_ptr(), None,
                                      o.data_ptr(), cnt.data_ptr(), N, ws.data_ptr(), ws.numel(), _stream())
            assert st == _lib.PS_OK
            assert int(cnt.item()) == m, (fname, k)
            assert torch.equal(o[:m], rs) if fname == "ps_select" else torch.equal(o, rp), (fname, k)
    assert _status(tiny, ws) == _lib.PS_OK


def test_reduce_by_key_repeated(tiny):
    # reduce-by-key keeps its own tiles (4096 keys) but this build's
    # two-descriptor look-back window: its segmented sum is not commutative
    keys = inputs.run_keys(N, 16, 48)
    vals = inputs.full_range_i32(N, 49)
    want_keys, want_sums = oracle.reduce_by_key(keys, vals)
    m = want_keys.shape[0]
    kt, vt = torch.from_numpy(keys).to(DEV), torch.from_numpy(vals).to(DEV)
    uk, ag = torch.empty_like(kt), torch.empty_like(vt)
    nr = torch.zeros(1, dtype=torch.int64, device=DEV)
    ws = torch.zeros(max(int(tiny.ps_reduce_by_key_workspace_size(_lib.PS_INT32, N)), 16), dtype=torch.uint8,
                     device=DEV)
    rk = torch.from_numpy(want_keys.view(np.int32)).to(DEV)
    rs = torch.from_numpy(want_sums.view(np.int32)).to(DEV)
    for k in range(REPEATS):
        st = tiny.ps_reduce_by_key(_lib.PS_INT32, _lib.PS_INT32, kt.data_ptr(), vt.data_ptr(), uk.data_ptr(),
                                   ag.data_ptr(), nr.data_ptr(), N, ws.data_ptr(), ws.numel(), _stream())
        assert st == _lib.PS_OK
        assert int(nr.item()) == m, k
        assert torch.equal(uk[:m], rk) and torch.equal(ag[:m], rs), k
    assert _status(tiny, ws) == _lib.PS_OK


def test_run_length_encode_repeated(tiny):
    # this build's run-length encoding has 16 KiB tiles (four compute warps):
    # four times the tiles, look-backs and output-buffer hand-offs per byte;
    # runs of mean length 4 (dense tiles), 16 and 256, int32 and int64 keys
    for kdt, code in ((np.int32, _lib.PS_INT32), (np.int64, _lib.PS_INT64)):
        ws = torch.zeros(max(int(tiny.ps_reduce_by_key_workspace_size(code, N)), 16), dtype=torch.uint8,
                         device=DEV)
        for mean in (4, 16, 256):
            keys = inputs.run_keys(N, mean, 60 + mean, kdt)
            want_keys, want_counts = oracle.reduce_by_key(keys, None)
            m = want_keys.shape[0]
            kt = torch.from_numpy(keys).to(DEV)
            uk = torch.empty_like(kt)
            cnt = torch.empty(N, dtype=torch.int32, device=DEV)
            nr = torch.zeros(1, dtype=torch.int64, device=DEV)
            rk = torch.from_numpy(want_keys).to(DEV)
            rc = torch.from_numpy(np.asarray(want_counts).astype(np.int64)).to(DEV)
            for k in range(30):
                st = tiny.ps_run_length_encode(code, kt.data_ptr(), uk.data_ptr(), cnt.data_ptr(), nr.data_ptr(), N,
                                               ws.data_ptr(), ws.numel(), _stream())
                assert st == _lib.PS_OK
                assert int(nr.item()) == m, (kdt, mean, k)
                assert torch.equal(uk[:m], rk) and torch.equal(cnt[:m].long(), rc), (kdt, mean, k)
        assert _status(tiny, ws) == _lib.PS_OK
