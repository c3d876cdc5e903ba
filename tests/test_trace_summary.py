"""The pipeline-trace summary (prefix_scan_gb300/trace.py) on a hand-made trace.

The committed trace profile quotes the summary's medians, per-CTA intervals
and look-back window counts; this test feeds summarize() four tiles on two
CTAs whose every figure is worked out by hand below, so a wrong column, an
off-by-one tile or a mixed-up bit field in the look-back word fails here.
"""
from __future__ import annotations

import numpy as np

from prefix_scan_gb300 import trace


def _hand_trace():
    # per tile, us: claim, data, aggregate, look-back start, prefix,
    # compute start, prefix received, stored (tile 0 looks back at nothing)
    t = np.array([
        [1.0, 2.0, 3.0, 0.0, 0.0, 2.0, 3.5, 4.0],
        [1.5, 3.0, 4.0, 4.5, 6.0, 3.0, 6.2, 7.0],
        [3.0, 4.0, 5.0, 5.0, 7.0, 4.0, 7.1, 8.0],
        [3.5, 5.0, 6.0, 6.5, 8.5, 5.0, 8.6, 9.0],
    ])
    # look-back word: windows << 16 | re-polls
    lb = np.array([0, (1 << 16) | 0, (2 << 16) | 1, (1 << 16) | 0], dtype=np.uint32)
    cta = np.array([0, 1, 0, 1], dtype=np.int32)
    # per CTA, us: entry, header verdict, compute warps done
    ct = np.array([[0.0, 1.0, 9.5], [0.2, 1.2, 9.6]])
    return t, lb, cta, ct


def test_summary_figures():
    s = trace.summarize("hand", 4, [_hand_trace()])
    assert "(4 tiles, 1 traced calls" in s
    # starts: last CTA entry 0.2; header verdict 1.0 after entry (both CTAs);
    # first claim 1.0; first data 2.0; last claim 3.5; last store 9.0; last done 9.6
    assert ("last CTA starts 0.20; a CTA has the header's verdict 1.00 after it starts; first claim 1.00; "
            "first tile landed 2.00; last claim 3.50; last store issued 9.00; "
            "last CTA's compute warps done 9.60") in s
    assert "span, first claim to last store: median 8.00 us" in s
    # CTA 0 claims at 1.0 and 3.0, CTA 1 at 1.5 and 3.5: intervals 2.0 and 2.0
    assert "CTAs that took tiles: 2; per-CTA interval between claims: 2.00 (2.00 / 2.00) us" in s
    # claim -> data: 1.0, 1.5, 1.0, 1.5
    assert "| claim -> data landed | 1.25 (1.00 / 1.50) |" in s
    # look-backs of tiles 1-3: 1.5, 2.0, 2.0 us; queue (start - A): 0.5, 0.0, 0.5
    assert "| look-back (start -> P published) | 2.00 (1.60 / 2.00) |" in s
    assert "| A -> look-back starts (queue) | 0.50 (0.10 / 0.50) |" in s
    # windows 1, 2, 1 and re-polls 0, 1, 0
    assert "1: 66.7%, 2: 33.3%, 3: 0.0%, 4: 0.0%, 5+: 0.0% (mean 1.33)" in s
    assert "re-polls of unpublished descriptors per look-back: median 0, p90 1, none in 66.7%" in s


def test_summary_over_calls_takes_medians():
    a = _hand_trace()
    t, lb, cta, ct = _hand_trace()
    b = (t + 1.0, lb, cta, ct)   # the same call shifted by 1 us except the CTA starts
    c = (t + 2.0, lb, cta, ct)
    s = trace.summarize("hand", 4, [a, b, c])
    assert "first claim 2.00" in s            # median of 1.0, 2.0, 3.0
    assert "span, first claim to last store: median 8.00 us" in s
