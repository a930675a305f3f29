"""Host logic of bench.py --phases (CPU): summarize_phases on a constructed record of 3
launches x 4 CTAs with known timelines — global times near 1.7e18 ns (which float64 alone
would round to 256 ns), an SM clock of 2 GHz that wraps past 2^32 inside a CTA, and
phases at known offsets."""
from __future__ import annotations

import numpy as np

import bench


def make_record():
    n, grid, words = 3, 4, 16
    rec = np.zeros((n, grid, words), dtype=np.int64)
    t0 = 1_700_000_000_000_000_123
    for i in range(n):
        for c in range(grid):
            entry = t0 + i * 1000 + 10 * c
            rec[i, c, 0] = entry
            rec[i, c, 1] = entry + 900              # every CTA runs 900 ns
            rec[i, c, 2] = c                        # CTA c on SM c
            c0 = (1 << 32) - 500 + 7 * c            # entry clock: wraps during the CTA
            for word, cycles in ((3, 200), (4, 400), (5, 600), (7, 1600), (8, 1800), (9, 500)):
                rec[i, c, word] = (c0 + cycles) % (1 << 32)
            rec[i, c, 6] = c0
    return rec


def test_summarize_phases_known_timeline():
    out = bench.summarize_phases(make_record())
    assert abs(out["sm_mhz"] - 2000.0) < 1e-6
    assert out["span_ns"] == 930.0
    assert out["overlap_prev_ns"] == -70.0
    assert out["period_ns"] == 1000.0
    assert out["cta_entry_spread_ns"] == 30.0 and out["cta_exit_spread_ns"] == 30.0
    assert out["sm_handoff_ns"] == 100.0
    expect = {"copies_issued": 100.0, "wait_done": 200.0, "x_staged": 300.0, "warp0_done": 800.0,
              "cta_done": 900.0, "stage0_landed": 250.0}
    for k, v in expect.items():
        assert abs(out[k + "_ns"] - v) < 1e-6 and abs(out[k + "_ns_max"] - v) < 1e-6, (k, out[k + "_ns"])
    assert "first_stage_ns" not in out and "stage1_landed_ns" not in out   # never stamped


def test_summarize_phases_single_launch():
    out = bench.summarize_phases(make_record()[:1])
    assert "period_ns" not in out and out["sm_handoff_ns"] is None
    assert out["span_ns"] == 930.0
