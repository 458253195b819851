"""The trace summary (host logic, CPU): per-wave figures from hand-built records."""
import torch

import comm_gemm_tile_gb300 as mk
from comm_gemm_tile_gb300 import trace as T

BASE = 1_700_000_000_000_000_000        # a %globaltimer-sized origin (ns)
CLK0 = 5_000_000_000_000                # an SM clock64 origin


def _records(epoch=7, old_epoch=3):
    """Two CTAs, three items each (items 2c + j*2 ... on CTA c), at a 2 GHz clock: item j
    of CTA c starts at 20 j + c us, its inputs are ready 0.5 us later, its accumulator
    20 us after the start, its epilogue 3 us after that.  Slot 12 holds a stale record."""
    rec = torch.zeros((14, mk.TRACE_WORDS), dtype=torch.int64)
    for c in range(2):
        for j in range(3):
            i = 2 * j + c
            t = BASE + (20_000 * j + 1_000 * c)
            row = rec[2 * i]
            row[mk.TRACE_START] = t
            row[mk.TRACE_INPUTS] = t + 500
            row[mk.TRACE_ISSUED] = t + 15_000
            row[mk.TRACE_READY] = t + 20_000
            row[mk.TRACE_END] = t + 23_000
            row[mk.TRACE_CLK_START] = CLK0 + 2 * (t - BASE)
            row[mk.TRACE_CLK_READY] = CLK0 + 2 * (t + 20_000 - BASE)
            row[mk.TRACE_ID] = (epoch << 32) | (c << 1)
    rec[12, mk.TRACE_START] = BASE - 10**9
    rec[12, mk.TRACE_READY] = BASE + 10**9
    rec[12, mk.TRACE_ID] = (old_epoch << 32) | (5 << 1)
    return rec


def test_summary_of_hand_built_records():
    d = T.summarize(_records())
    assert d["items"] == 6 and d["ctas"] == 2 and d["records"] == 6     # the stale record is dropped
    assert abs(d["span_us"] - (40 + 1 + 23)) < 1e-6
    w = d["waves"]
    assert [x["n"] for x in w] == [2, 2, 2]
    assert abs(w[0]["ready_gap_us"] - 20.5) < 1e-6            # from the launch's first stamp
    for x in w[1:]:
        assert abs(x["ready_gap_us"] - 20.0) < 1e-6
        assert abs(x["ready_gap_cycles"] - 40_000) < 1e-6
    for x in w:
        assert abs(x["input_wait_us"] - 0.5) < 1e-6 and abs(x["epilogue_us"] - 3.0) < 1e-6
        assert abs(x["sm_mhz"] - 2000.0) < 1e-6
    assert "2000" in T.format_summary(d)


def test_copy_records_and_pooled_waves():
    rec = _records()
    cr = torch.zeros((mk.TRACE_COPY_RECORDS, mk.TRACE_WORDS), dtype=torch.int64)
    for wkr in range(4):
        cr[wkr, 0] = BASE + 1_000
        cr[wkr, 1] = BASE + 11_000 + 1_000 * wkr
        cr[wkr, 2] = 10
        cr[wkr, 3] = 1_000_000
        cr[wkr, mk.TRACE_ID] = (7 << 32) | wkr
    cr[9, mk.TRACE_ID] = (3 << 32) | 9                           # another call's record
    d = T.summarize(rec, cr, max_rows=2)
    c = d["copy"]
    assert c["warps"] == 4 and c["bytes"] == 4_000_000
    assert abs(c["end_max_us"] - 14.0) < 1e-6 and abs(c["start_us"] - 1.0) < 1e-6
    assert abs(c["tb_per_s"] - 4e6 / 13e-6 / 1e12) < 1e-9
    assert [x["wave"] for x in d["waves"]] == ["0-1", "2"]        # three waves in two rows
