"""Pipeline trace of the single-pass scan kernel.

Builds the library with PS_TRACE defined (``_build/trace/``, not the
product library), runs the persistent scan on a workload with the L2 flushed
before each call, reads the per-tile timestamps back through
``ps_trace_read`` (include/prefix_scan_trace.h) and prints where a tile's
time goes, as a markdown section:

  claim -> A          tile id taken until its aggregate is published
  A -> look-back      the tile waits for its CTA's look-back warp
  look-back           windows walked and re-polls until P is published
  P -> compute        the prefix reached the compute warps (negative when
                      they were still busy with earlier tiles)
  compute -> stored   the compute warps' scan-and-store after the prefix

The decoupled look-back ("Single-pass Parallel Prefix Scan with Decoupled
Look-back", summary page, sections 4.1 and 4.4) is meant to keep the
look-back off the critical path; these figures say whether it does.

    python -m prefix_scan_gb300.trace --workload i32_excl_2p28 [--runs 5]
    python -m prefix_scan_gb300.trace --kernel rle --n 33554432 [--mean-run 16]

``--define NAME=VALUE`` rebuilds the variant with other compile-time
settings of the kernel (for example the look-back's poll back-off), and
``--launch-only K`` only launches the scan K times after one warm-up call
(no trace read, no summary): the command to put under a profiler when
comparing such variants.  ``--l2-probe``, ``--read-probe`` and
``--link-probe`` build and run the measurement probes under ``probes/``
instead (one look-back window's L2 round trip; HBM read bandwidth by loads
and by bulk copies; the host link by copies and by kernels).
"""
from __future__ import annotations

import argparse
import ctypes
import sys
from pathlib import Path

import numpy as np

if __package__ in (None, ""):
    sys.path.insert(0, str(Path(__file__).resolve().parents[1]))

from prefix_scan_gb300 import _lib, workloads  # noqa: E402
from prefix_scan_gb300 import build as nvbuild  # noqa: E402

POINTS = ("claim", "data", "aggregate", "lookback_start", "prefix", "compute_start",
          "prefix_received", "stored")
C, D, AG, LS, PR, CS, RC, ST = range(8)
FLUSH_BYTES = 512 << 20


def load_trace_library(defines: dict[str, int] | None = None, trace: bool = True) -> ctypes.CDLL:
    defs = dict(defines or {})
    if trace:
        defs["PS_TRACE"] = 1
    name = "trace" if defs == {"PS_TRACE": 1} else \
        "v_" + "_".join(f"{k.lower()}{v}" for k, v in sorted(defs.items()))
    path = nvbuild.build_variant(name, defs)
    lib = ctypes.CDLL(str(path))
    for name, (res, args) in _lib.SIGNATURES.items():
        if "noalloc" in name:
            continue
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    if trace and lib.ps_trace_capacity() == 0:
        raise RuntimeError("the trace build records no trace")
    return lib


def launch_only(lib: ctypes.CDLL, w: workloads.Workload, n: int, launches: int) -> None:
    """One warm-up call, then `launches` back-to-back calls; prints one line."""
    import torch
    dev = torch.device("cuda", 0)
    code = {"int32": _lib.PS_INT32, "int64": _lib.PS_INT64, "float32": _lib.PS_FLOAT32}[w.dtype]
    x = torch.from_numpy(w.make(n)).to(dev)
    out = x if w.inplace else torch.empty_like(x)
    ws = torch.zeros(max(int(lib.ps_scan_workspace_size(code, n)), 16), dtype=torch.uint8, device=dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    for _ in range(launches + 1):
        _lib.check("ps_scan", lib.ps_scan(_lib.PS_ALGO_DECOUPLED_LOOKBACK, code, int(w.exclusive), x.data_ptr(),
                                          out.data_ptr(), n, ws.data_ptr(), ws.numel(), stream))
    st = ctypes.c_int(-1)
    _lib.check("ps_get_device_status", lib.ps_get_device_status(ws.data_ptr(), stream, ctypes.byref(st)))
    print(f"{w.name} n={n}: {launches + 1} launches, device status {st.value}", flush=True)


# Kernels the trace covers: the record each keeps (include/prefix_scan_trace.h)
# and the elements of one of its tiles (32-bit keys / elements).
KERNELS = {"scan": 0, "select": 1, "partition": 1, "rbk": 2, "rle": 3}
RBK_TILE, RLE_TILE = 4096, 16384


def make_call(lib: ctypes.CDLL, kernel: str, w: workloads.Workload | None, n: int, mean_run: int, dev):
    """(call(stream) -> status, tiles, keep-alive tensors) for one launch of
    `kernel` on seeded inputs of length n: the scan workload `w`; select and
    partition of full-range int32 values by Bernoulli(1/2) flags; reduce-by-key
    ({int32 key, fp32 value}) and run-length encoding of int32 keys in runs of
    mean length `mean_run`."""
    import torch
    from prefix_scan_gb300 import inputs
    if kernel == "scan":
        code = {"int32": _lib.PS_INT32, "int64": _lib.PS_INT64, "float32": _lib.PS_FLOAT32}[w.dtype]
        x = torch.from_numpy(w.make(n)).to(dev)
        out = x if w.inplace else torch.empty_like(x)
        ws = torch.zeros(max(int(lib.ps_scan_workspace_size(code, n)), 16), dtype=torch.uint8, device=dev)

        def call(stream):
            return lib.ps_scan(_lib.PS_ALGO_DECOUPLED_LOOKBACK, code, int(w.exclusive), x.data_ptr(),
                               out.data_ptr(), n, ws.data_ptr(), ws.numel(), stream)
        return call, -(-n // int(lib.ps_tile_elements(code))), (x, out, ws)
    if kernel in ("select", "partition"):
        x = torch.from_numpy(inputs.full_range_i32(n, 8)).to(dev)
        flags = torch.from_numpy(inputs.bernoulli_half(n, 3).astype(np.uint8)).to(dev)
        out = torch.empty_like(x)
        cnt = torch.zeros(1, dtype=torch.int64, device=dev)
        ws = torch.zeros(max(int(lib.ps_scan_workspace_size(_lib.PS_INT32, n)), 16), dtype=torch.uint8, device=dev)
        fn = lib.ps_partition if kernel == "partition" else lib.ps_select

        def call(stream):
            return fn(_lib.PS_INT32, 0, x.data_ptr(), flags.data_ptr(), None, out.data_ptr(), cnt.data_ptr(), n,
                      ws.data_ptr(), ws.numel(), stream)
        return call, -(-n // int(lib.ps_tile_elements(_lib.PS_INT32))), (x, flags, out, cnt, ws)
    keys = torch.from_numpy(inputs.run_keys(n, mean_run, 11)).to(dev)
    vals = torch.from_numpy(inputs.uniform_f32(n, 12)).to(dev)
    uk = torch.empty_like(keys)
    ag = torch.empty(n, dtype=torch.int32 if kernel == "rle" else torch.float32, device=dev)
    nr = torch.zeros(1, dtype=torch.int64, device=dev)
    ws = torch.zeros(max(int(lib.ps_reduce_by_key_workspace_size(_lib.PS_INT32, n)), 16), dtype=torch.uint8,
                     device=dev)

    def call(stream):
        if kernel == "rle":
            return lib.ps_run_length_encode(_lib.PS_INT32, keys.data_ptr(), uk.data_ptr(), ag.data_ptr(),
                                            nr.data_ptr(), n, ws.data_ptr(), ws.numel(), stream)
        return lib.ps_reduce_by_key(_lib.PS_INT32, _lib.PS_FLOAT32, keys.data_ptr(), vals.data_ptr(), uk.data_ptr(),
                                    ag.data_ptr(), nr.data_ptr(), n, ws.data_ptr(), ws.numel(), stream)
    return call, -(-n // (RLE_TILE if kernel == "rle" else RBK_TILE)), (keys, vals, uk, ag, nr, ws)


def run(lib: ctypes.CDLL, w: workloads.Workload | None, n: int, runs: int, kernel: str = "scan",
        mean_run: int = 16):
    """Traces of `runs` calls (L2 flushed before each): list of
    (timestamps[tiles, 8] in us from the first CTA's start, lookback[tiles],
    cta[tiles], per-CTA timestamps[ctas, 3] in us on the same base)."""
    import torch
    dev = torch.device("cuda", 0)
    call, tiles, keep = make_call(lib, kernel, w, n, mean_run, dev)
    which = KERNELS[kernel]
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    tiles = min(tiles, int(lib.ps_trace_capacity()))
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    traces = []
    for r in range(runs + 1):   # the first call warms up and is dropped
        flush.fill_(r & 0xFF)
        _lib.check(kernel, call(stream))
        ts = np.zeros((tiles, 8), dtype=np.uint64)
        lb = np.zeros(tiles, dtype=np.uint32)
        cta = np.zeros(tiles, dtype=np.int32)
        _lib.check("ps_trace_read", lib.ps_trace_read(which, ts.ctypes.data, lb.ctypes.data, cta.ctypes.data,
                                                      tiles))
        if r == 0:
            continue
        ctas = int(cta.max()) + 1
        cts = np.zeros((ctas, 3), dtype=np.uint64)
        _lib.check("ps_trace_read_ctas", lib.ps_trace_read_ctas(which, cts.ctypes.data, ctas))
        t0 = int(cts[:, 0].min())
        t = (ts.astype(np.int64) - t0) / 1e3
        ct = (cts.astype(np.int64) - t0) / 1e3
        traces.append((t, lb, cta, ct))
    return traces


def _dist(v: np.ndarray) -> str:
    return f"{np.median(v):.2f} ({np.percentile(v, 10):.2f} / {np.percentile(v, 90):.2f})"


def summarize(name: str, n: int, traces) -> str:
    rows = []
    spans, lasts = [], []
    gaps = {k: [] for k in ("claim_A", "A_lb", "lb", "P_compute", "compute_stored", "claim_stored",
                            "claim_data", "data_A", "interval")}
    windows, polls, lbt = [], [], []
    starts = {k: [] for k in ("first_claim", "last_entry", "header", "first_data", "last_store", "last_done")}
    for t, lb, cta, ct in traces:
        starts["first_claim"].append(t[:, C].min())
        starts["last_entry"].append(ct[:, 0].max())
        starts["header"].append(np.median(ct[:, 1] - ct[:, 0]))
        starts["first_data"].append(t[:, D].min())
        starts["last_store"].append(t[:, ST].max())
        starts["last_done"].append(ct[:, 2].max())
        spans.append(t[:, ST].max() - t[:, C].min())
        gaps["claim_data"].append(t[:, D] - t[:, C])
        gaps["data_A"].append(t[:, AG] - t[:, D])
        gaps["claim_A"].append(t[:, AG] - t[:, C])
        gaps["A_lb"].append(t[1:, LS] - t[1:, AG])
        gaps["lb"].append(t[1:, PR] - t[1:, LS])
        gaps["P_compute"].append(t[:, RC] - t[:, PR])
        gaps["compute_stored"].append(t[:, ST] - t[:, RC])
        gaps["claim_stored"].append(t[:, ST] - t[:, C])
        for c in np.unique(cta):
            cl = np.sort(t[cta == c, C])
            if cl.size > 1:
                gaps["interval"].append(np.diff(cl))
        looked = t[1:, LS] > 0   # tiles whose look-back ran and recorded
        windows.append((lb[1:][looked] >> 16).astype(np.int64))
        polls.append((lb[1:][looked] & 0xFFFF).astype(np.int64))
        lbt.append((t[1:, PR] - t[1:, LS])[looked])
        lasts.append(t[:, C].max())
    cat = {k: np.concatenate(v) if v else np.zeros(1) for k, v in gaps.items()}
    win = np.concatenate(windows)
    pol = np.concatenate(polls)
    tiles = traces[0][0].shape[0]
    rows.append(f"### {name} at n = {n} ({tiles} tiles, {len(traces)} traced calls, L2 flushed before each)")
    rows.append("")
    rows.append(f"- from the first CTA's start (medians over the calls, us): last CTA starts "
                f"{np.median(starts['last_entry']):.2f}; a CTA has the header's verdict "
                f"{np.median(starts['header']):.2f} after it starts; first claim "
                f"{np.median(starts['first_claim']):.2f}; first tile landed {np.median(starts['first_data']):.2f}; "
                f"last claim {np.median(lasts):.2f}; last store issued {np.median(starts['last_store']):.2f}; "
                f"last CTA's compute warps done {np.median(starts['last_done']):.2f}")
    rows.append(f"- span, first claim to last store: median {np.median(spans):.2f} us")
    rows.append(f"- CTAs that took tiles: {len(np.unique(traces[0][2]))}; per-CTA interval between claims: "
                f"{_dist(cat['interval'])} us")
    rows.append("")
    rows.append("| stage | median (p10 / p90), us |")
    rows.append("|---|---|")
    for key, label in (("claim_data", "claim -> data landed"), ("data_A", "data landed -> A published"),
                       ("claim_A", "claim -> A published"), ("A_lb", "A -> look-back starts (queue)"),
                       ("lb", "look-back (start -> P published)"),
                       ("P_compute", "P published -> compute warps have it"),
                       ("compute_stored", "prefix received -> stores issued"),
                       ("claim_stored", "claim -> stores issued")):
        rows.append(f"| {label} | {_dist(cat[key])} |")
    rows.append("")
    hist = [(win == k).mean() for k in (1, 2, 3, 4)] + [(win >= 5).mean()]
    rows.append(f"- look-back windows of 32 descriptors walked: 1: {hist[0]:.1%}, 2: {hist[1]:.1%}, "
                f"3: {hist[2]:.1%}, 4: {hist[3]:.1%}, 5+: {hist[4]:.1%} (mean {win.mean():.2f})")
    rows.append(f"- re-polls of unpublished descriptors per look-back: median {np.median(pol):.0f}, "
                f"p90 {np.percentile(pol, 90):.0f}, none in {(pol == 0).mean():.1%}")
    # a look-back's time against the windows it walked, among those that never
    # re-polled: the slope is the cost of one more window, the rest is fixed
    lt = np.concatenate(lbt)
    cells = []
    for k in (1, 2, 3, 4, 5):
        sel = (win == k) & (pol == 0)
        if sel.sum() >= 20:
            cells.append(f"{k}: {np.median(lt[sel]):.2f} us ({int(sel.sum())})")
    if cells:
        rows.append("- look-back time by windows walked, no re-polls (median, count): " + "; ".join(cells))
    rows.append("")
    return "\n".join(rows)


def run_l2_probe() -> None:
    """Builds (under _build/) and runs the probe of one look-back window's
    L2 round trip, idle and under a full-rate copy; prints its lines."""
    import subprocess
    src = Path(__file__).resolve().parent / "probes" / "l2_window_latency.cu"
    exe = nvbuild.BUILD_DIR / "l2_window_latency"
    exe.parent.mkdir(parents=True, exist_ok=True)
    subprocess.run([nvbuild.nvcc_path(), *nvbuild.ARCH, "-O3", "-o", str(exe), str(src)], check=True)
    subprocess.run([str(exe)], check=True)


def run_read_probe() -> None:
    """Builds (under _build/) and runs the read-bandwidth probe: 1 GiB read by
    plain loads and by bulk copies into shared-memory stages; prints its lines."""
    import subprocess
    src = Path(__file__).resolve().parent / "probes" / "read_bandwidth.cu"
    exe = nvbuild.BUILD_DIR / "read_bandwidth"
    exe.parent.mkdir(parents=True, exist_ok=True)
    subprocess.run([nvbuild.nvcc_path(), *nvbuild.ARCH, "-O3", "-std=c++17", "-o", str(exe), str(src)], check=True)
    subprocess.run([str(exe)], check=True)


def run_link_probe() -> None:
    """Builds (under _build/) and runs the host-link probe: 1 GiB each way
    between pinned host memory and the GPU by copies and by kernels."""
    import subprocess
    src = Path(__file__).resolve().parent / "probes" / "host_link.cu"
    exe = nvbuild.BUILD_DIR / "host_link"
    exe.parent.mkdir(parents=True, exist_ok=True)
    subprocess.run([nvbuild.nvcc_path(), *nvbuild.ARCH, "-O3", "-std=c++17", "-o", str(exe), str(src)], check=True)
    subprocess.run([str(exe)], check=True)


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--workload", action="append", choices=sorted(workloads.BY_NAME), default=[],
                    help="scan workload (repeatable)")
    ap.add_argument("--kernel", action="append", choices=[k for k in KERNELS if k != "scan"], default=[],
                    help="another persistent kernel, on its seeded inputs (repeatable; length from --n)")
    ap.add_argument("--mean-run", type=int, default=16, help="mean run length of the rbk / rle keys")
    ap.add_argument("--n", type=int, action="append", default=None,
                    help="length per --workload (default: the workload's own)")
    ap.add_argument("--runs", type=int, default=5)
    ap.add_argument("--define", action="append", default=[], metavar="NAME=VALUE",
                    help="compile-time setting of the variant build (repeatable)")
    ap.add_argument("--l2-probe", action="store_true",
                    help="build and run the L2 window-latency probe (probes/l2_window_latency.cu)")
    ap.add_argument("--read-probe", action="store_true",
                    help="build and run the read-bandwidth probe (probes/read_bandwidth.cu)")
    ap.add_argument("--link-probe", action="store_true",
                    help="build and run the host-link probe (probes/host_link.cu)")
    ap.add_argument("--launch-only", type=int, default=0, metavar="K",
                    help="only launch the scan K times (a build without the trace)")
    args = ap.parse_args(argv)
    if args.l2_probe:
        run_l2_probe()
        return
    if args.read_probe:
        run_read_probe()
        return
    if args.link_probe:
        run_link_probe()
        return
    defines = {}
    for d in args.define:
        k, _, v = d.partition("=")
        defines[k] = int(v)
    lib = load_trace_library(defines, trace=not args.launch_only)
    for i, name in enumerate(args.workload):
        w = workloads.BY_NAME[name]
        n = args.n[i] if args.n and i < len(args.n) else w.n
        if args.launch_only:
            launch_only(lib, w, n, args.launch_only)
        else:
            print(summarize(w.name, n, run(lib, w, n, args.runs)), flush=True)
    for j, kernel in enumerate(args.kernel):
        i = len(args.workload) + j
        n = args.n[i] if args.n and i < len(args.n) else 1 << 25
        label = kernel + (f" (int32 keys, mean run {args.mean_run})" if kernel in ("rbk", "rle")
                          else " (int32 values, flag array, Bernoulli(1/2))")
        print(summarize(label, n, run(lib, None, n, args.runs, kernel, args.mean_run)), flush=True)


if __name__ == "__main__":
    main()
