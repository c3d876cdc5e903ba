"""The DRAM-traffic record bench.py reports for its headline kernel.

bench.py scales the ncu-counted DRAM bytes of a small capture of the
headline kernel (profiles/persistent_kernel_i32_excl_2p26_traffic.md) to the
timed workload, and reports them only while the hash of that kernel's
sources still matches the one recorded beside the capture.  These tests run
on the CPU: the record is present and current for the headline workload (so
a kernel edit that left it stale fails here, before any GPU run), the
scaling is by elements processed, and the hash ignores comments but not
code.
"""
from __future__ import annotations

import sys
from pathlib import Path

ROOT = Path(__file__).resolve().parents[1]
sys.path.insert(0, str(ROOT))

import bench  # noqa: E402
from prefix_scan_gb300 import workloads  # noqa: E402


def test_record_is_current_for_the_headline_workload():
    w = workloads.BY_NAME["i32_excl_2p28"]
    rec = bench.recorded_traffic(w, w.n)
    assert rec is not None, ("the headline kernel's sources changed since its DRAM traffic was captured: "
                             "recapture it and update the record's kernel_sources_sha256")
    # the capture's reads and writes are each close to the 4-byte elements it moved
    assert abs(rec["captured_bytes"] - 2 * 4 * rec["captured_n"]) < 0.01 * 2 * 4 * rec["captured_n"]
    assert rec["bytes"] == round(rec["captured_bytes"] * w.n / rec["captured_n"])


def test_record_is_refused_for_another_kernel_instance():
    for name in ("f32_incl_2p24", "i64_incl_2p29", "i32_incl_2p20"):
        w = workloads.BY_NAME[name]
        assert bench.recorded_traffic(w, w.n) is None, name


def test_hash_ignores_comments_but_not_code():
    a = "int f(int x) { return x + 1; } // one\n/* two */"
    b = "int f(int x) {\n    return x + 1;   // another comment\n}\n"
    c = "int f(int x) { return x + 2; }"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)
