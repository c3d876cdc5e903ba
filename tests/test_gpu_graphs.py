"""The calls captured in a CUDA graph and replayed.

A call is one kernel launch that leaves its workspace ready for the next
(descriptors carry the epoch of the call that wrote them; no per-call reset),
so a graph captured once replays any number of times: the replays below
rewrite the captured input buffers and compare every output with the
oracle.
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


def _capture(fn):
    s = torch.cuda.Stream(device=DEV)
    s.wait_stream(torch.cuda.current_stream(DEV))
    with torch.cuda.stream(s):
        fn()                       # warm-up outside the capture (one-time attribute setup)
    torch.cuda.current_stream(DEV).wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


@pytest.mark.parametrize("n", [1000, 3 * 8192 + 5, (1 << 22) + 7])
def test_scan_graph_replays(n):
    # short arrays (one CTA) and the look-back kernel
    x = torch.empty(n, dtype=torch.int32, device=DEV)
    y = torch.empty_like(x)
    ws = api.alloc_workspace(torch.int32, n, DEV)
    g = _capture(lambda: api.scan(x, exclusive=True, out=y, workspace=ws,
                                  stream=torch.cuda.current_stream(DEV)))
    for seed in range(6):
        xs = inputs.full_range_i32(n, 700 + seed)
        x.copy_(torch.from_numpy(xs))
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(y.cpu().numpy(), oracle.exclusive(xs)), seed
    assert api.device_status(ws) == _lib.PS_OK


def test_graph_of_several_kernels_sharing_one_workspace():
    # scan, select and reduce-by-key in one graph, one workspace between them
    n = (1 << 21) + 3
    x = torch.empty(n, dtype=torch.int32, device=DEV)
    f = torch.empty(n, dtype=torch.uint8, device=DEV)
    k = torch.empty(n, dtype=torch.int32, device=DEV)
    y = torch.empty_like(x)
    sel = torch.empty_like(x)
    part = torch.empty_like(x)
    uk = torch.empty_like(k)
    agg = torch.empty_like(k)
    uk2 = torch.empty_like(k)
    lens = torch.empty_like(k)
    need = max(api.workspace_size(torch.int32, n), api.reduce_by_key_workspace_size(torch.int32, n))
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    box = {}

    def body():
        st = torch.cuda.current_stream(DEV)
        api.scan(x, out=y, workspace=ws, stream=st)
        _, box["cnt"] = api.select(x, f, out=sel, workspace=ws, stream=st)
        _, box["pcnt"] = api.partition(x, f, out=part, workspace=ws, stream=st)
        _, _, box["runs"] = api.reduce_by_key(k, x, unique_keys=uk, aggregates=agg, workspace=ws, stream=st)
        _, _, box["rle"] = api.run_length_encode(k, unique_keys=uk2, counts=lens, workspace=ws, stream=st)

    g = _capture(body)
    for seed in range(4):
        xs = inputs.full_range_i32(n, 800 + seed)
        fs = inputs.bernoulli_half(n, 810 + seed).astype(np.uint8)
        ks = inputs.run_keys(n, 16, 820 + seed)
        x.copy_(torch.from_numpy(xs))
        f.copy_(torch.from_numpy(fs))
        k.copy_(torch.from_numpy(ks))
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(y.cpu().numpy(), oracle.inclusive(xs))
        want = oracle.select(xs, fs)
        m = int(box["cnt"].item())
        assert m == want.shape[0] and np.array_equal(sel[:m].cpu().numpy(), want)
        pw, pk = oracle.partition(xs, fs)
        assert int(box["pcnt"].item()) == pk == m
        assert np.array_equal(part.cpu().numpy(), pw)
        okeys, ovals = oracle.reduce_by_key(ks, xs)
        r = int(box["runs"].item())
        assert r == okeys.shape[0]
        assert np.array_equal(uk[:r].cpu().numpy(), okeys) and np.array_equal(agg[:r].cpu().numpy(), ovals)
        lkeys, lcounts = oracle.reduce_by_key(ks, None)
        r = int(box["rle"].item())
        assert r == lkeys.shape[0]
        assert np.array_equal(uk2[:r].cpu().numpy(), lkeys) and np.array_equal(lens[:r].cpu().numpy(), lcounts)
    assert api.device_status(ws) == _lib.PS_OK
