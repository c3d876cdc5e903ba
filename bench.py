#!/usr/bin/env python3
"""Benchmark of the single-pass decoupled look-back prefix sum on GB300.

One "step" is one scan call (one launch of the single-pass kernel) over
the whole input of the chosen workload, inputs resident in HBM.  Prints ONE
JSON line (rank 0).  Metric: achieved bandwidth in GB/s with the algorithmic
traffic 2 * n * sizeof(T) (read every input once, write every output once),
plus Gelem/s and the ratio to a device-to-device memcpy of the same bytes
timed in the same run.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference] [--no-configs] [--compare] [--compaction]
                  [--ops] [--rbk]

The line's ``configs`` key times every other workload the same way (the
in-place workload at each of its lengths), so one default run covers them
all; the headline stays the 2^28 int32 exclusive scan.

--impl reference times the CPU oracle (the plain sequential scan) on the
host cores on a bounded sample of the same workload.  With N > 1 (torchrun)
each rank runs an independent replica of the workload on its own GPU (the
scan has no data-parallel exchange to shard): "scaling": "weak".
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

from prefix_scan_gb300 import workloads  # noqa: E402

L2_BYTES = 129 * 1000 * 1000
FLUSH_BYTES = 512 << 20
METRIC = "scan Gelem/s and achieved HBM GB/s (2n·sizeof(T)) vs same-run memcpy, 1×GB300"
DEFAULT_WORKLOAD = workloads.I32_EXCL_2P28.name
DTYPE_TAG = {"int32": "int32", "int64": "int64", "float32": "f32"}


# ----------------------------------------------------------------- peaks ----

def hbm_peak() -> tuple[float, str]:
    p = ROOT / "MEASURED_PEAKS.json"
    try:
        d = json.loads(p.read_text())
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------- clocks ----

def nvml_handle(torch_device_index: int):
    """(NVML library, device handle) for a torch CUDA device, matched by PCI
    bus id (NVML and CUDA may number devices differently); read-only use."""
    import torch
    props = torch.cuda.get_device_properties(torch_device_index)
    bus = (f"{getattr(props, 'pci_domain_id', 0):08X}:{props.pci_bus_id:02X}:"
           f"{props.pci_device_id:02X}.0")
    nv = ctypes.CDLL("libnvidia-ml.so.1")
    if nv.nvmlInit_v2() != 0:
        raise RuntimeError("nvmlInit failed")
    h = ctypes.c_void_p()
    if nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
        raise RuntimeError("no NVML handle for " + bus)
    return nv, h


def bind_to_gpu_cpus(torch_device_index: int) -> str:
    """Runs this process on the CPUs that NVML reports as local to the GPU,
    so that pinned host buffers allocated afterwards sit on the GPU's NUMA
    node (a host-side setting of this process only).  Returns what it did."""
    try:
        nv, h = nvml_handle(torch_device_index)
        words = ((os.cpu_count() or 64) + 63) // 64
        mask = (ctypes.c_ulong * words)()
        if nv.nvmlDeviceGetCpuAffinity(h, ctypes.c_uint(words), mask) != 0:
            return "unbound (NVML reported no CPU affinity)"
        bits = 8 * ctypes.sizeof(ctypes.c_ulong)
        cpus = {w * bits + b for w in range(words) for b in range(bits) if (mask[w] >> b) & 1}
        cpus &= os.sched_getaffinity(0)
        if not cpus:
            return "unbound (no GPU-local CPU available)"
        os.sched_setaffinity(0, cpus)
        return f"bound to the {len(cpus)} CPUs local to the GPU"
    except Exception as exc:   # no NVML: run where the OS placed us
        return f"unbound ({type(exc).__name__})"

class ClockSampler:
    """Samples SM clock, power and clock-event reasons during a region.

    NVML through ctypes (read-only queries) every few milliseconds; falls
    back to ``nvidia-smi -lms`` when NVML cannot be opened.
    """

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_device_index: int = 0, period_s: float = 0.005):
        self.period = period_s
        self.samples: list[tuple[int, int, int]] = []   # (sm_mhz, reasons_mask, power_mw)
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self._smi = None
        self._smi_path = None
        self._nvml = None
        self._handle = None
        try:
            nv, h = nvml_handle(torch_device_index)
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self._nvml, self._handle = nv, h
            self._reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
        except Exception:
            self._nvml = None

    def _sample_nvml(self):
        nv, h = self._nvml, self._handle
        clk, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk))
            nv.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw))
            self._reasons_fn(h, ctypes.byref(rs))
            self.samples.append((clk.value, rs.value, pw.value))
            time.sleep(self.period)

    def __enter__(self):
        self._stop.clear()
        if self._nvml is not None:
            self._thread = threading.Thread(target=self._sample_nvml, daemon=True)
            self._thread.start()
        else:
            try:
                import tempfile
                fd, self._smi_path = tempfile.mkstemp(suffix=".csv")
                os.close(fd)
                self._smi = subprocess.Popen(
                    ["nvidia-smi", "-i", os.environ.get("LOCAL_RANK", "0"),
                     "--query-gpu=clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active",
                     "--format=csv,noheader,nounits", "-lms", "100", "-f", self._smi_path])
            except Exception:
                self._smi = None
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self._thread is not None:
            self._thread.join()
        if self._smi is not None:
            time.sleep(0.15)
            self._smi.terminate()
            self._smi.wait()
            for line in Path(self._smi_path).read_text().splitlines():
                try:
                    sm, mx, pw, act = [v.strip() for v in line.split(",")]
                    self.samples.append((int(float(sm)), int(act, 16), int(float(pw) * 1000)))
                    self.max_mhz = int(float(mx))
                except ValueError:
                    continue
            os.unlink(self._smi_path)
        return False

    def summary(self) -> dict:
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": "nvml" if self._nvml is not None else "nvidia-smi"}
        mask = 0
        for _, r, _ in self.samples:
            mask |= r
        reasons = [name for bit, name in self.REASONS.items() if mask & bit]
        return {"sm_mhz": int(statistics.median(s[0] for s in self.samples)),
                "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(self.samples),
                "power_w_max": round(max(s[2] for s in self.samples) / 1000.0, 1),
                "source": "nvml" if self._nvml is not None else "nvidia-smi"}


# -------------------------------------------------------------- helpers ----

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _reduce(v: float, world: int, op) -> float:
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=op)
    return float(t.item())


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    return _reduce(v, world, dist.ReduceOp.MAX)


def sum_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    return _reduce(v, world, dist.ReduceOp.SUM)


def replica_stats(local_seconds: float, local_units: float, world: int) -> tuple[float, float]:
    """Whole-job numbers of N independent replicas: (max time over ranks,
    units processed by all ranks).  Throughput = units / time."""
    return max_over_ranks(local_seconds, world), sum_over_ranks(local_units, world)


KERNEL_TRAFFIC_FILE = ROOT / "profiles" / "persistent_kernel_i32_excl_2p26_traffic.md"


# The headline kernel's translation unit and the headers it includes: a
# change anywhere else leaves its recorded DRAM traffic valid.
HEADLINE_KERNEL_SOURCES = ("scan_device.cuh", "scan_internal.h", "scan_persistent.cu", "scan_pipeline.cuh")


def _code_only(text: str) -> str:
    """C/C++ source without comments and with whitespace collapsed, so that
    editing a comment does not read as a kernel change."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_sources_sha256() -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = ROOT / "prefix_scan_gb300" / "csrc"
    for name in HEADLINE_KERNEL_SOURCES:
        h.update(name.encode())
        h.update(_code_only((csrc / name).read_text()).encode())
    return h.hexdigest()


def recorded_traffic(w: workloads.Workload, n: int):
    """DRAM bytes per launch for ``n`` elements of workload ``w``, from the
    committed ncu summary of a smaller launch of the same kernel instance
    (same dtype and scan kind), scaled by the elements processed; None when
    the summary is for another instance or the kernel sources changed since.
    The capture runs launches back to back with ncu's cache control off, so
    each captured launch also writes back what the previous one left dirty
    in L2 -- its traffic per element is the steady state's, which makes the
    linear scaling sound."""
    try:
        kv = {}
        for line in KERNEL_TRAFFIC_FILE.read_text().splitlines():
            if line.startswith("- ") and ":" in line:
                k, _, v = line[2:].partition(":")
                kv[k.strip()] = v.strip().strip("`")
        kind = "exclusive" if w.exclusive else "inclusive"
        if kv.get("dtype") != w.dtype or kv.get("kind") != kind:
            return None
        if kv.get("kernel_sources_sha256") != kernel_sources_sha256():
            return None
        n_cap = int(kv["n_captured"])
        per_launch = int(kv["dram_bytes_read_per_launch"]) + int(kv["dram_bytes_write_per_launch"])
        return {"bytes": int(round(per_launch * n / n_cap)), "captured_n": n_cap,
                "captured_bytes": per_launch, "source": KERNEL_TRAFFIC_FILE.name,
                "scaling": f"x {n / n_cap:g} (elements processed)"}
    except Exception:
        return None


def cpu_baseline(w: workloads.Workload, target_s: float = 10.0, sample_n: int = 1 << 26) -> dict:
    """The oracle as it stands, single-threaded, on a bounded sample."""
    import oracle
    n = min(sample_n, w.n)
    x = w.make(n)
    fn = oracle.exclusive if w.exclusive else oracle.inclusive
    fn(x[:1024])  # load/compile outside the timing
    reps, t0 = 0, time.perf_counter()
    best = float("inf")
    while True:
        t = time.perf_counter()
        fn(x)
        best = min(best, time.perf_counter() - t)
        reps += 1
        if time.perf_counter() - t0 >= target_s:
            break
    elems_s = n / best
    gbs = 2.0 * n * w.itemsize / best / 1e9
    return {"value": round(gbs, 3), "unit": "GB/s", "gelem_per_s": round(elems_s / 1e9, 4),
            "cores": 1, "kind": "oracle",
            "sample": f"first {n} elements of the {w.name} input, best of {reps} runs "
                      f"({time.perf_counter() - t0:.1f} s of single-threaded CPU work)",
            "cpu": _cpu_model()}


def cpu_oracle_rate(call, algorithmic_bytes: int, sample: str, target_s: float = 1.5) -> dict:
    """The oracle's rate for one operation, as it stands, single-threaded:
    best of as many calls as fit in ``target_s`` (at least two), in GB/s of
    the operation's algorithmic bytes on the sample."""
    call()   # load the oracle library outside the timing
    best, reps, t0 = float("inf"), 0, time.perf_counter()
    while reps < 2 or time.perf_counter() - t0 < target_s:
        t = time.perf_counter()
        call()
        best = min(best, time.perf_counter() - t)
        reps += 1
    return {"value": round(algorithmic_bytes / best / 1e9, 3), "unit": "GB/s", "cores": 1,
            "kind": "oracle", "sample": f"{sample}, best of {reps}"}


def _cpu_model() -> str:
    try:
        for line in Path("/proc/cpuinfo").read_text().splitlines():
            if line.lower().startswith(("model name", "cpu part")):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


# ------------------------------------------------------------ reference ----

def run_reference(args, rank: int, world: int) -> None:
    """--impl reference: the CPU oracle, timed on the host cores."""
    if rank != 0:
        return
    w = workloads.BY_NAME[args.workload]
    import oracle
    n_full = args.n or w.n                 # the workload our arm times
    n = min(args.ref_sample, n_full)       # each step: a bounded sample of it
    x = w.make(n)
    fn = oracle.exclusive if w.exclusive else oracle.inclusive
    fn(x[:1024])
    for _ in range(max(args.warmup, 0)):
        fn(x)
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        fn(x)
        times.append(time.perf_counter() - t)
    total = sum(times)
    gbs = 2.0 * n * w.itemsize * args.steps / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 3), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1000 * total / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_TAG[w.dtype], "data": "synthetic",
        "config": _config(w, world, n_full),
        "sample": f"each step scans the first {n} of the workload's {n_full} elements",
        "cpu_baseline": {"value": round(gbs, 3), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"first {n} of {n_full} elements per step", "cpu": _cpu_model()},
        "e2e": {"value": round(gbs, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gelem_per_s": round(n * args.steps / total / 1e9, 4),
    }
    print(json.dumps(line), flush=True)


def _config(w: workloads.Workload, world: int, n: int, note: str = "") -> dict:
    c = {"workload": w.describe() if n == w.n else w.describe().replace(f"n={w.n}", f"n={n}"),
         "name": w.name, "n": n, "elem_bytes": w.itemsize,
         "algorithmic_bytes_per_step": 2 * n * w.itemsize,
         "parallelism": f"replicas{world}" if world > 1 else "single-gpu",
         "l2": "inputs larger than L2" if n * w.itemsize > 2 * L2_BYTES else "L2 flushed between steps"}
    if note:
        c["note"] = note
    return c


# ------------------------------------------------------------------ ours ----

class Harness:
    def __init__(self, w: workloads.Workload, n: int, dev):
        import torch
        from prefix_scan_gb300 import api
        self.torch, self.api, self.w, self.n, self.dev = torch, api, w, n, dev
        tdt = {"int32": torch.int32, "int64": torch.int64, "float32": torch.float32}[w.dtype]
        self.tdt = tdt
        self.host_in = torch.empty(n, dtype=tdt, pin_memory=True)
        w.make(n, out=self.host_in.numpy())
        self.host_out = torch.empty(n, dtype=tdt, pin_memory=True)
        self.d_in = self.host_in.to(dev)
        self.pristine = None
        self.d_out = self.d_in if w.inplace else torch.empty_like(self.d_in)
        self.ws = api.alloc_workspace(tdt, n, dev)
        self.stream = torch.cuda.current_stream(dev)
        self.flush = None
        if n * w.itemsize <= 2 * L2_BYTES:
            self.flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.launches_per_step = 1

    def step(self, algo="decoupled"):
        self.api.scan(self.d_in, exclusive=self.w.exclusive, out=self.d_out,
                      workspace=self.ws, algo=algo)

    def timed(self, steps: int, fn, world: int) -> tuple[float, list[float]]:
        """Seconds for ``steps`` calls of fn, events on the launching stream."""
        torch = self.torch
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * steps)]
        barrier(world)
        torch.cuda.synchronize()
        per = []
        if self.flush is None:
            ev[0].record(self.stream)
            for _ in range(steps):
                fn()
            ev[1].record(self.stream)
            torch.cuda.synchronize()
            total = ev[0].elapsed_time(ev[1]) / 1e3
            per = [total / steps] * steps
        else:
            for k in range(steps):
                self.flush.fill_(k & 0xFF)        # evict the data from L2
                ev[2 * k].record(self.stream)
                fn()
                ev[2 * k + 1].record(self.stream)
            torch.cuda.synchronize()
            per = [ev[2 * k].elapsed_time(ev[2 * k + 1]) / 1e3 for k in range(steps)]
            total = sum(per)
        barrier(world)
        return total, per

    def memcpy(self):
        dst = self.d_out if not self.w.inplace else self._scratch()
        dst.copy_(self.d_in)

    def _scratch(self):
        if getattr(self, "_scr", None) is None:
            self._scr = self.torch.empty_like(self.d_in)
        return self._scr

    def e2e_step(self):
        """The public host-buffer call (ps_scan_host): pinned host in -> chunks
        streamed through the GPU (copies in both directions overlapped with
        the scans) -> pinned host out; completion is ordered on the stream."""
        if getattr(self, "_host_bufs", None) is None:
            self._host_bufs = self.api.HostScanBuffers(self.tdt, self.n, self.dev)
        self.api.scan_host(self.host_in, exclusive=self.w.exclusive, out=self.host_out,
                           buffers=self._host_bufs, stream=self.stream, synchronize=False)

    def property_check(self) -> bool:
        """Cheap self-check of a fresh output (no oracle): prefixes at a few
        sampled positions against running sums of the host input."""
        torch = self.torch
        src = self.d_in
        if self.w.inplace:
            src = self.d_out.copy_(self.host_in.to(self.dev))
        self.api.scan(src, exclusive=self.w.exclusive, out=self.d_out, workspace=self.ws)
        torch.cuda.synchronize()
        y = self.d_out.cpu().numpy()
        x = self.host_in.numpy()
        idx = sorted(set([0, self.n - 1] + list(np.linspace(0, self.n - 1, 9).astype(np.int64))))
        ok, pos = True, 0
        acc, acc_abs = 0, 0.0
        for i in idx:
            hi = i if self.w.exclusive else i + 1
            seg = x[pos:hi]
            if self.w.dtype == "float32":
                acc += float(np.sum(seg, dtype=np.float64))
                acc_abs += float(np.sum(np.abs(seg), dtype=np.float64))
                ok &= abs(float(y[i]) - acc) <= 1e-5 * acc_abs + 1e-6
            else:
                bits = 32 if self.w.dtype == "int32" else 64
                acc += int(np.sum(seg, dtype=np.int64)) if bits == 32 else \
                    int(np.sum(seg.view(np.uint64), dtype=np.uint64))
                ok &= (int(y[i]) - acc) % (1 << bits) == 0
            pos = hi
        return bool(ok)


def run_ours(args, rank: int, world: int, local: int) -> None:
    import torch
    from prefix_scan_gb300 import build as nvbuild
    if not nvbuild.is_fresh():
        nvbuild.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    host_binding = bind_to_gpu_cpus(local)   # before any pinned host buffer exists
    w = workloads.BY_NAME[args.workload]
    n = args.n or w.n
    h = Harness(w, n, dev)
    bytes_step = 2 * n * w.itemsize
    peak, peak_kind = hbm_peak()

    for _ in range(args.warmup):
        h.step()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    with sampler:
        t_scan, per = h.timed(args.steps, h.step, world)
    t_scan, units_total = replica_stats(t_scan, float(n * args.steps), world)
    # same-run device-to-device copy of the same bytes, same protocol
    for _ in range(max(3, args.warmup)):
        h.memcpy()
    t_copy, _ = h.timed(args.steps, h.memcpy, world)
    t_copy = max_over_ranks(t_copy, world)
    # end to end through the public API on pinned host buffers
    e2e_steps = max(3, min(args.steps, args.e2e_steps))
    for _ in range(2):
        h.e2e_step()
    torch.cuda.synchronize()
    saved = h.flush
    h.flush = None
    t_e2e, _ = h.timed(e2e_steps, h.e2e_step, world)
    h.flush = saved
    t_e2e = max_over_ranks(t_e2e, world)
    ok = h.property_check()

    gbs = 2.0 * w.itemsize * units_total / t_scan / 1e9
    per_launch = statistics.median(per)
    achieved = bytes_step / per_launch / 1e9
    copy_gbs = 2.0 * n * w.itemsize * args.steps / t_copy / 1e9
    e2e_gbs = 2.0 * w.itemsize * sum_over_ranks(float(n * e2e_steps), world) / t_e2e / 1e9

    extra = {}
    if args.compare and world == 1:
        for algo in ("reduce_then_scan", "chained"):
            k = max(3, min(args.steps, 20))
            h.step(algo)
            torch.cuda.synchronize()
            t, _ = h.timed(k, lambda: h.step(algo), 1)
            extra[algo] = {"gbs": round(bytes_step * k / t / 1e9, 2),
                           "ms_per_step": round(1000 * t / k, 4)}
    configs = []
    if not args.no_configs and world == 1:
        configs = run_configs(w)
    compaction = run_compaction(args) if args.compaction and world == 1 else None
    ops = run_ops(args) if args.ops and world == 1 else None
    rbk = run_reduce_by_key(args) if args.rbk and world == 1 else None

    if rank != 0:
        return
    if args.traffic is not None:
        traffic = {"bytes": int(args.traffic), "source": "--traffic"}
    else:
        traffic = recorded_traffic(w, n)
    tbytes = traffic["bytes"] if traffic else None
    line = {
        "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1000 * t_scan / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_TAG[w.dtype], "data": "synthetic",
        "config": _config(w, world, n),
        "gelem_per_s": round(units_total / t_scan / 1e9, 3),
        "memcpy_gbs": round(copy_gbs, 2), "vs_memcpy": round(gbs / copy_gbs, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": tbytes,
                     "dram_frac": round(tbytes / per_launch / 1e9 / peak, 4) if tbytes else None,
                     "traffic_source": traffic,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                     else "fallback 6.8 TB/s",
                     "per_launch_ms": round(per_launch * 1000, 4),
                     "note": "one kernel launch per step (no workspace reset); median CUDA-event step time; "
                             "frac counts the algorithmic 2n*sizeof(T) bytes, dram_frac the DRAM bytes ncu "
                             "counted (traffic) over the same time"},
        "e2e": {"value": round(e2e_gbs, 2), "unit": "GB/s",
                "h2d_bytes_per_step": n * w.itemsize, "d2h_bytes_per_step": n * w.itemsize,
                "steps": e2e_steps,
                "path": "ps_scan_host: pinned host buffers, 32 MiB chunks in 3 device buffers, H2D/scan/D2H overlapped",
                "host_cpus": host_binding},
        "gpu_launches": args.steps * h.launches_per_step,
        "clocks": sampler.summary(),
        "parity_spot_check": ok,
    }
    if extra:
        line["comparison_paths"] = extra
    if configs:
        line["configs"] = configs
    if compaction:
        line["compaction"] = compaction
    if ops:
        line["other_ops"] = ops
    if rbk:
        line["reduce_by_key"] = rbk
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, target_s=args.cpu_seconds)
    print(json.dumps(line), flush=True)


def run_configs(headline: workloads.Workload) -> list[dict]:
    """Every other workload (each length of the in-place sweep), timed as
    the headline is: warm-up, then median CUDA-event time of K calls (the L2
    flushed before each call where the data would fit in it), beside a
    device-to-device copy of the same bytes timed the same way, and a
    sampled self-check of the output.  Compact: one entry per length."""
    import torch
    out = []
    for w in workloads.ALL:
        if w.name == headline.name:
            continue
        for n in (w.sweep if w.sweep else (w.n,)):
            h = Harness(w, n, torch.device("cuda", 0))
            k = 40 if h.flush is not None else 20
            for _ in range(3):
                h.step()
            _, per = h.timed(k, h.step, 1)
            for _ in range(3):
                h.memcpy()
            _, per_c = h.timed(k, h.memcpy, 1)
            b = 2 * n * w.itemsize
            med, med_c = statistics.median(per), statistics.median(per_c)
            out.append({"name": w.name, "n": n, "ms": round(med * 1000, 4),
                        "gbs": round(b / med / 1e9, 2), "gelem_per_s": round(n / med / 1e9, 3),
                        "memcpy_gbs": round(b / med_c / 1e9, 2), "vs_memcpy": round(med_c / med, 4),
                        "steps": k, "l2": "flushed before each call" if h.flush is not None else "larger than L2",
                        "spot_check": h.property_check()})
            del h
            torch.cuda.empty_cache()
    return out


def run_compaction(args, n: int = 1 << 28) -> dict:
    """Single-pass select / partition of int32 values by a Bernoulli(1/2)
    flag array (the 0/1 pattern of the exclusive-scan workload), GB/s with
    the algorithmic bytes: values read + flags read + elements written."""
    import torch
    from prefix_scan_gb300 import api, inputs
    dev = torch.device("cuda", 0)
    x = torch.from_numpy(inputs.full_range_i32(n, 8)).to(dev)
    f = torch.from_numpy(inputs.bernoulli_half(n, 3).astype(np.uint8)).to(dev)
    ws = api.alloc_workspace(torch.int32, n, dev)
    out = torch.empty_like(x)
    res = {"n": n, "values": "int32 uniform", "flags": "Bernoulli(0.5) uint8"}
    stream = torch.cuda.current_stream(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for name, fn in (("select", lambda: api.select(x, f, out=out, workspace=ws)),
                     ("partition", lambda: api.partition(x, f, out=out, workspace=ws))):
        for _ in range(3):
            _, cnt = fn()
        torch.cuda.synchronize()
        k = int(cnt.item())
        reps = max(3, min(args.steps, 20))
        ev0.record(stream)
        for _ in range(reps):
            fn()
        ev1.record(stream)
        torch.cuda.synchronize()
        t = ev0.elapsed_time(ev1) / 1e3 / reps
        written = k if name == "select" else n
        b = n * 4 + n + written * 4
        res[name] = {"ms": round(t * 1000, 4), "gbs": round(b / t / 1e9, 2),
                     "gelem_per_s": round(n / t / 1e9, 3), "kept": k,
                     "algorithmic_bytes": b, "frac_of_peak": round(b / t / 1e9 / hbm_peak()[0], 4)}
    if not args.no_cpu_baseline:
        import oracle
        m = 1 << 24
        xs, fs = inputs.full_range_i32(m, 8), inputs.bernoulli_half(m, 3).astype(np.uint8)
        kept = int(np.count_nonzero(fs))
        res["select"]["cpu_baseline"] = cpu_oracle_rate(lambda: oracle.select(xs, fs), m * 5 + kept * 4,
                                                        f"first {m} elements")
        res["partition"]["cpu_baseline"] = cpu_oracle_rate(lambda: oracle.partition(xs, fs), m * 9,
                                                           f"first {m} elements")
    return res


def run_reduce_by_key(args, n: int = 1 << 25) -> dict:
    """Single-pass reduce-by-key of {int32 key, fp32 value} pairs and
    run-length encoding of the int32 keys, for several mean run lengths, GB/s
    with the algorithmic bytes: keys (and values) read + one (key, 32-bit
    aggregate) pair written per run.  The keys of 2^25 pairs are about the
    size of L2, so L2 is flushed (a 512 MiB write) before every call and
    each call is timed on its own; the leg reports the mean call time."""
    import torch
    from prefix_scan_gb300 import api, inputs
    dev = torch.device("cuda", 0)
    ws = torch.zeros(api.reduce_by_key_workspace_size(torch.int32, n), dtype=torch.uint8, device=dev)
    vt = torch.from_numpy(inputs.uniform_f32(n, 12)).to(dev)
    uk = torch.empty(n, dtype=torch.int32, device=dev)
    agg = torch.empty(n, dtype=torch.float32, device=dev)
    cnts = agg.view(torch.int32)
    nr = torch.zeros(1, dtype=torch.int64, device=dev)   # reused: no allocation or fill per call
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    res = {"n": n, "keys": "int32, runs of uniform length in [1, 2L-1]", "values": "fp32 uniform [-1, 1)",
           "l2": "flushed before each call"}
    for mean in (1, 16, 256):
        kt = torch.from_numpy(inputs.run_keys(n, mean, 11 + mean)).to(dev)
        for name, fn in (("reduce_by_key", lambda: api.reduce_by_key(kt, vt, unique_keys=uk, aggregates=agg,
                                                                     workspace=ws, num_runs=nr)),
                         ("run_length_encode", lambda: api.run_length_encode(kt, unique_keys=uk, counts=cnts,
                                                                             workspace=ws, num_runs=nr))):
            for _ in range(3):
                _, _, cnt = fn()
            torch.cuda.synchronize()
            m = int(cnt.item())
            reps = max(3, min(args.steps, 40))
            ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * reps)]
            for k in range(reps):
                flush.fill_(k & 0xFF)   # evict the keys and values from L2
                ev[2 * k].record(stream)
                fn()
                ev[2 * k + 1].record(stream)
            torch.cuda.synchronize()
            t = sum(ev[2 * k].elapsed_time(ev[2 * k + 1]) for k in range(reps)) / 1e3 / reps
            b = n * (8 if name == "reduce_by_key" else 4) + m * 8 + 8
            res[f"{name}_L{mean}"] = {"ms": round(t * 1000, 4), "gbs": round(b / t / 1e9, 2),
                                       "gpairs_per_s": round(n / t / 1e9, 3), "runs": m,
                                       "algorithmic_bytes": b,
                                       "frac_of_peak": round(b / t / 1e9 / hbm_peak()[0], 4)}
        del kt
        if not args.no_cpu_baseline:
            import oracle
            ms_ = 1 << 22
            ks = inputs.run_keys(ms_, mean, 11 + mean)
            vs = inputs.uniform_f32(ms_, 12)
            runs = int(np.count_nonzero(np.r_[True, ks[1:] != ks[:-1]]))
            res[f"reduce_by_key_L{mean}"]["cpu_baseline"] = cpu_oracle_rate(
                lambda: oracle.reduce_by_key(ks, vs), ms_ * 8 + runs * 8, f"first {ms_} pairs")
            res[f"run_length_encode_L{mean}"]["cpu_baseline"] = cpu_oracle_rate(
                lambda: oracle.reduce_by_key(ks, None), ms_ * 4 + runs * 8, f"first {ms_} keys")
    return res


PROFILE_CASES = ("scan", "rbk_f32_L16", "rle_L16", "select_flagged", "partition_flagged")


def run_profile_case(args) -> None:
    """Launch one kernel case ``args.steps`` times after one warm-up launch and
    print one short JSON line: the entry point for ncu captures of a single
    kernel (the cases are the ones the extra bench legs time)."""
    import torch
    from prefix_scan_gb300 import api, inputs
    dev = torch.device("cuda", 0)
    case = args.profile_case
    if case == "scan":
        # the scan of --workload (its kind, placement and distribution) at
        # --n elements (default 2^26)
        n = args.n or 1 << 26
        w = workloads.BY_NAME[args.workload]
        x = torch.from_numpy(w.make(n)).to(dev)
        out = x if w.inplace else torch.empty_like(x)
        ws = api.alloc_workspace(x.dtype, n, dev)
        fn = lambda: api.scan(x, exclusive=w.exclusive, out=out, workspace=ws)[-1:].view(torch.uint8)[:1]
    elif case in ("rbk_f32_L16", "rle_L16"):
        n = args.n or 1 << 25
        kt = torch.from_numpy(inputs.run_keys(n, 16, 27)).to(dev)
        vt = torch.from_numpy(inputs.uniform_f32(n, 12)).to(dev)
        ws = torch.zeros(api.reduce_by_key_workspace_size(torch.int32, n), dtype=torch.uint8, device=dev)
        uk, agg = torch.empty_like(kt), torch.empty_like(vt)
        if case == "rbk_f32_L16":
            fn = lambda: api.reduce_by_key(kt, vt, unique_keys=uk, aggregates=agg, workspace=ws)[2]
        else:
            fn = lambda: api.run_length_encode(kt, unique_keys=uk, counts=agg.view(torch.int32), workspace=ws)[2]
    else:
        n = args.n or 1 << 28
        x = torch.from_numpy(inputs.full_range_i32(n, 8)).to(dev)
        f = torch.from_numpy(inputs.bernoulli_half(n, 3).astype(np.uint8)).to(dev)
        ws = api.alloc_workspace(torch.int32, n, dev)
        out = torch.empty_like(x)
        sel = api.select if case == "select_flagged" else api.partition
        fn = lambda: sel(x, f, out=out, workspace=ws)[1]
    cnt = fn()
    for _ in range(args.steps):
        cnt = fn()
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": case, "workload": args.workload if case == "scan" else None, "n": n,
                      "launches": args.steps + 1, "count": int(cnt.item()), "status": api.device_status(ws)}),
          flush=True)


def run_ops(args, n: int = 1 << 28) -> dict:
    """Running max / min of int32 (uniform full range), the fp32 sum of the
    deterministic mode at 2^28, and the {int32, fp32} pair sum and fp32
    affine-map composition over 2^27 8-byte elements (the same bytes); GB/s
    with one read and one write of every element."""
    import torch
    from prefix_scan_gb300 import api, inputs
    dev = torch.device("cuda", 0)
    x = torch.from_numpy(inputs.full_range_i32(n, 9)).to(dev)
    xf = torch.from_numpy(inputs.uniform_f32(n, 10)).to(dev)
    out = torch.empty_like(x)
    ws = api.alloc_workspace(torch.int32, n, dev)
    stream = torch.cuda.current_stream(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    res = {"n": n}
    n8 = n // 2   # 8-byte elements: the same bytes as the int32 cases
    p8 = torch.empty((n8, 2), dtype=torch.int32, device=dev)
    p8[:, 0] = torch.from_numpy(inputs.full_range_i32(n8, 13)).to(dev)
    p8[:, 1] = torch.from_numpy(inputs.uniform_f32(n8, 14).view(np.int32)).to(dev)
    f8 = torch.from_numpy(np.stack([inputs.uniform_f32(n8, 15), inputs.uniform_f32(n8, 16)], axis=1)).to(dev)
    o8 = torch.empty_like(p8)
    ws8 = api.alloc_workspace(torch.int64, n8, dev)
    cases = (("max_int32", lambda: api.scan(x, op="max", out=out, workspace=ws)),
             ("min_int32", lambda: api.scan(x, op="min", out=out, workspace=ws)),
             ("sum_fp32_deterministic", lambda: api.scan(xf, out=out.view(torch.float32), workspace=ws,
                                                         algo="deterministic")),
             ("pair_i32_f32_sum", lambda: api.scan_pairs(p8, out=o8, workspace=ws8)),
             ("affine_f32_compose", lambda: api.scan_affine(f8, out=o8.view(torch.float32), workspace=ws8)))
    for name, fn in cases:
        for _ in range(3):
            fn()
        reps = max(3, min(args.steps, 20))
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(reps):
            fn()
        ev1.record(stream)
        torch.cuda.synchronize()
        t = ev0.elapsed_time(ev1) / 1e3 / reps
        res[name] = {"ms": round(t * 1000, 4), "gbs": round(8 * n / t / 1e9, 2),
                     "frac_of_peak": round(8 * n / t / 1e9 / hbm_peak()[0], 4)}
    if not args.no_cpu_baseline:
        import oracle
        m = 1 << 24
        xi, xf = inputs.full_range_i32(m, 9), inputs.uniform_f32(m, 10)
        a8, b8 = inputs.uniform_f32(m // 2, 15), inputs.uniform_f32(m // 2, 16)
        i8 = inputs.full_range_i32(m // 2, 13)
        smp = f"first {m} 4-byte elements ({m // 2} 8-byte ones)"
        res["max_int32"]["cpu_baseline"] = cpu_oracle_rate(lambda: oracle.scan_op(xi, "max"), 8 * m, smp)
        res["min_int32"]["cpu_baseline"] = cpu_oracle_rate(lambda: oracle.scan_op(xi, "min"), 8 * m, smp)
        res["sum_fp32_deterministic"]["cpu_baseline"] = cpu_oracle_rate(lambda: oracle.inclusive(xf), 8 * m, smp)
        res["pair_i32_f32_sum"]["cpu_baseline"] = cpu_oracle_rate(
            lambda: oracle.scan_pair_i32_f32(i8, a8), 8 * m, smp)
        res["affine_f32_compose"]["cpu_baseline"] = cpu_oracle_rate(
            lambda: oracle.scan_affine_f32(a8, b8), 8 * m, smp)
    return res


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(workloads.BY_NAME))
    ap.add_argument("--n", type=int, default=0, help="override the workload length")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--compare", action="store_true", help="also time the comparison paths")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads (the `configs` key of the default run)")
    ap.add_argument("--compaction", action="store_true", help="also time select / partition at 2^28")
    ap.add_argument("--ops", action="store_true", help="also time max / min and the deterministic mode at 2^28")
    ap.add_argument("--rbk", action="store_true", help="also time reduce-by-key / run-length encoding at 2^25")
    ap.add_argument("--profile-case", choices=PROFILE_CASES, default=None,
                    help="only launch this kernel case --steps times (for ncu captures)")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch from an ncu capture of the current kernel")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-sample", type=int, default=1 << 25)
    args = ap.parse_args()
    if args.profile_case:
        run_profile_case(args)
        return
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        if args.impl == "reference":
            if rank != 0:
                return
        else:
            import torch
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    try:
        run_ours(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            if dist.is_initialized():
                dist.destroy_process_group()


if __name__ == "__main__":
    main()
