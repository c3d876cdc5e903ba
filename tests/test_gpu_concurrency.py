"""Several calls in flight at once on different streams, each with its own
workspace.

The persistent kernels size their grid for the whole GPU, but correctness
does not depend on all their CTAs being resident: tile ids come from an
atomic counter, so a CTA only ever waits on tiles that running CTAs have
already claimed.  Kernels sharing the GPU must therefore all finish, with
correct results and no look-back timeout.
"""
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


def test_scans_on_concurrent_streams():
    n = (1 << 24) + 11
    streams = [torch.cuda.Stream(device=DEV) for _ in range(4)]
    xs = [inputs.full_range_i32(n, 900 + i) for i in range(4)]
    xt = [torch.from_numpy(x).to(DEV) for x in xs]
    ys = [torch.empty_like(t) for t in xt]
    wss = [api.alloc_workspace(torch.int32, n, DEV) for _ in range(4)]
    torch.cuda.synchronize()
    for rep in range(5):
        for i, st in enumerate(streams):
            with torch.cuda.stream(st):
                api.scan(xt[i], exclusive=bool(i & 1), out=ys[i], workspace=wss[i], stream=st)
    torch.cuda.synchronize()
    for i in range(4):
        ref = oracle.exclusive(xs[i]) if i & 1 else oracle.inclusive(xs[i])
        assert np.array_equal(ys[i].cpu().numpy(), ref), i
        assert api.device_status(wss[i]) == _lib.PS_OK


def test_different_kernels_concurrently():
    n = (1 << 23) + 5
    s1, s2, s3, s4, s5 = (torch.cuda.Stream(device=DEV) for _ in range(5))
    x = inputs.full_range_i32(n, 950)
    f = inputs.bernoulli_half(n, 951).astype(np.uint8)
    k = inputs.run_keys(n, 16, 952)
    xt, ft, kt = (torch.from_numpy(a).to(DEV) for a in (x, f, k))
    ws = [torch.zeros(max(api.workspace_size(torch.int32, n), api.reduce_by_key_workspace_size(torch.int32, n)),
                      dtype=torch.uint8, device=DEV) for _ in range(5)]
    torch.cuda.synchronize()
    for rep in range(4):
        with torch.cuda.stream(s1):
            y = api.scan(xt, workspace=ws[0], stream=s1)
        with torch.cuda.stream(s2):
            sel, cnt = api.select(xt, ft, workspace=ws[1], stream=s2)
        with torch.cuda.stream(s3):
            uk, agg, runs = api.reduce_by_key(kt, xt, workspace=ws[2], stream=s3)
        with torch.cuda.stream(s4):
            uk2, lens, runs2 = api.run_length_encode(kt, workspace=ws[3], stream=s4)
        with torch.cuda.stream(s5):
            part, pcnt = api.partition(xt, ft, workspace=ws[4], stream=s5)
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy(), oracle.inclusive(x))
    want = oracle.select(x, f)
    m = int(cnt.item())
    assert m == want.shape[0] and np.array_equal(sel[:m].cpu().numpy(), want)
    pw, pk = oracle.partition(x, f)
    assert int(pcnt.item()) == pk == m and np.array_equal(part.cpu().numpy(), pw)
    ok_k, ok_v = oracle.reduce_by_key(k, x)
    r = int(runs.item())
    assert r == ok_k.shape[0]
    assert np.array_equal(uk[:r].cpu().numpy(), ok_k) and np.array_equal(agg[:r].cpu().numpy(), ok_v)
    lk, lc = oracle.reduce_by_key(k, None)
    r = int(runs2.item())
    assert r == lk.shape[0]
    assert np.array_equal(uk2[:r].cpu().numpy(), lk) and np.array_equal(lens[:r].cpu().numpy(), lc)
    for w in ws:
        assert api.device_status(w) == _lib.PS_OK
