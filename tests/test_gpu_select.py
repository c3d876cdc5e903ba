"""GPU parity of single-pass stream compaction (select / partition) against
the CPU oracle: exact for every dtype (elements are moved, not summed)."""
from __future__ import annotations

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
NP = {"int32": np.int32, "int64": np.int64, "float32": np.float32}


def make(dtype, n, seed):
    if dtype == "float32":
        x = inputs.uniform_f32(n, seed)
        x[::97] = 0.0            # some zeros for "nonzero"
        return x
    x = inputs.uniform_int(n, -100, 100, seed, NP[dtype])
    return x


def flags_for(n, seed, p=0.5):
    h = inputs.hashes(n, seed)
    f = ((h >> np.uint64(40)).astype(np.float64) * 2.0 ** -24 < p).astype(np.uint8)
    return f * ((h & np.uint64(0x7F)).astype(np.uint8) | np.uint8(1))   # assorted nonzero bytes


def run(dtype, x, op, f=None, t=None, partition=False, inplace=False):
    xt = torch.from_numpy(x.copy()).to(DEV)
    ft = torch.from_numpy(f).to(DEV) if f is not None else None
    fn = api.partition if partition else api.select
    kw = dict(op=op, threshold=t)
    if not partition:
        kw["inplace"] = inplace
    out, cnt = fn(xt, ft, **kw)
    return out.cpu().numpy(), int(cnt.item())


def expect(dtype, x, op, f, t):
    flags = f if op == "flagged" else oracle.flags(x, op, t if t is not None else 0)
    return flags


@pytest.mark.parametrize("dtype", list(NP))
@pytest.mark.parametrize("op", ["flagged", "nonzero", "greater", "less"])
def test_select_and_partition(dtype, op):
    T = api.tile_elements(torch.int32 if dtype != "int64" else torch.int64)
    for k, n in enumerate([1, 7, 1000, T - 1, T, T + 1, 3 * T + 11, 40 * T + 5, (1 << 20) + 3]):
        x = make(dtype, n, 10 + k)
        f = flags_for(n, 20 + k, p=(0.1, 0.5, 0.9)[k % 3]) if op == "flagged" else None
        t = None if op in ("flagged", "nonzero") else NP[dtype](3)
        flags = expect(dtype, x, op, f, t)
        want = oracle.select(x, flags)
        got, cnt = run(dtype, x, op, f, t)
        assert cnt == want.shape[0], (n, cnt, want.shape[0])
        assert np.array_equal(got[:cnt], want), n
        pw, pk = oracle.partition(x, flags)
        got, cnt = run(dtype, x, op, f, t, partition=True)
        assert cnt == pk and np.array_equal(got, pw), n


@pytest.mark.parametrize("dtype", list(NP))
def test_select_in_place(dtype):
    T = api.tile_elements(torch.int32 if dtype != "int64" else torch.int64)
    for k, n in enumerate([5, T + 3, 17 * T + 1, (1 << 22) + 7]):
        x = make(dtype, n, 40 + k)
        f = flags_for(n, 50 + k, p=0.3)
        got, cnt = run(dtype, x, "flagged", f, inplace=True)
        want = oracle.select(x, f)
        assert cnt == want.shape[0] and np.array_equal(got[:cnt], want)
        # past the count the array keeps whatever the compaction left there:
        # inputs that were not overwritten
        got, cnt = run(dtype, x, "nonzero", inplace=True)
        assert np.array_equal(got[:cnt], oracle.select(x, oracle.flags(x, "nonzero")))


def test_select_edge_cases():
    n = 3 * api.tile_elements(torch.int32) + 5
    x = make("int32", n, 60)
    for f in (np.zeros(n, np.uint8), np.ones(n, np.uint8)):
        got, cnt = run("int32", x, "flagged", f)
        assert cnt == int(f.sum()) and np.array_equal(got[:cnt], x[f != 0])
    e = torch.empty(0, dtype=torch.int32, device=DEV)
    out, cnt = api.select(e, op="nonzero")
    assert cnt.item() == 0
    xf = np.array([np.nan, -0.0, 0.0, 1.0, -np.inf, np.inf], dtype=np.float32)
    got, cnt = run("float32", xf, "nonzero")
    assert cnt == 4 and np.isnan(got[0]) and list(got[1:4]) == [1.0, -np.inf, np.inf]
    got, cnt = run("float32", xf, "greater", t=np.float32(0))
    assert cnt == 2 and list(got[:2]) == [1.0, np.inf]


@pytest.mark.parametrize("dtype", list(NP))
def test_select_unaligned_reads_from_global(dtype):
    T = api.tile_elements(torch.int32 if dtype != "int64" else torch.int64)
    n = 5 * T + 9
    x = make(dtype, n + 1, 70)
    f = flags_for(n + 1, 71)
    xt = torch.from_numpy(x).to(DEV)[1:]           # values not 16-byte aligned
    ft = torch.from_numpy(f).to(DEV)[1:]
    out, cnt = api.select(xt, ft)
    want = oracle.select(x[1:], f[1:])
    assert cnt.item() == want.shape[0] and np.array_equal(out.cpu().numpy()[:cnt.item()], want)
    with pytest.raises(_lib.PrefixScanError, match="OVERLAP"):
        api.select(xt, ft, inplace=True)           # in place needs the bulk-copy path


def test_compaction_offsets_workload_full_size():
    # the int32 0/1 flag array of the exclusive-scan workload, used for what
    # its scan is for: compacting a 2^28-element array
    n = 1 << 28
    f = inputs.bernoulli_half(n, 3).astype(np.uint8)
    x = inputs.full_range_i32(n, 8)
    xt, ft = torch.from_numpy(x).to(DEV), torch.from_numpy(f).to(DEV)
    out, cnt = api.select(xt, ft)
    k = cnt.item()
    want = oracle.select(x, f)
    assert k == want.shape[0]
    assert np.array_equal(out[:k].cpu().numpy(), want)


def _wrap_i32(idx: torch.Tensor) -> torch.Tensor:
    """int64 values as int32 modulo 2^32."""
    return (idx - (idx >= 2 ** 31).to(torch.int64) * 2 ** 32).to(torch.int32)


def test_select_and_partition_above_2p31():
    # n > 2^31: output positions and counts need unsigned 32-bit arithmetic.
    # x[i] = i (as int32, modulo 2^32), kept where i % 3 == 0; checked in
    # chunks on the device against the closed forms: kept element j is
    # x[3 j]; partition's r-th rejected element (at out[n-1-r]) is x[i] for
    # i = 3 (r // 2) + 1 + r % 2.
    n, step = (1 << 31) + 4099, 1 << 28
    x = torch.empty(n, dtype=torch.int32, device=DEV)
    f = torch.empty(n, dtype=torch.uint8, device=DEV)
    for s in range(0, n, step):
        idx = torch.arange(s, min(n, s + step), dtype=torch.int64, device=DEV)
        x[s:s + idx.numel()] = _wrap_i32(idx)
        f[s:s + idx.numel()] = (idx % 3 == 0).to(torch.uint8)
    kept = (n + 2) // 3
    out = torch.empty_like(x)
    for part in (False, True):
        _, cnt = (api.partition if part else api.select)(x, f, out=out)
        assert int(cnt.item()) == kept
        for s in range(0, kept, step):
            j = torch.arange(s, min(kept, s + step), dtype=torch.int64, device=DEV)
            assert torch.equal(out[s:s + j.numel()], _wrap_i32(3 * j))
        if part:
            rejected = n - kept
            for s in range(0, rejected, step):
                r = torch.arange(s, min(rejected, s + step), dtype=torch.int64, device=DEV)
                got = out[n - 1 - (s + r.numel() - 1): n - s].flip(0)
                assert torch.equal(got, _wrap_i32(3 * (r // 2) + 1 + r % 2))
    del x, f, out
    torch.cuda.empty_cache()
