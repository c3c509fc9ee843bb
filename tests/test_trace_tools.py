"""Host-side trace analysis (level_times, prologue_lag) on hand-made traces:
no GPU, no library call."""
import numpy as np
import pytest

import persistent_sm_decode_gb300 as amk


class FakePlan:
    """Only what the trace helpers read: n_sm and per-CTA task lists."""

    def __init__(self, per_sm):
        self.per_sm = per_sm
        self.n_sm = len(per_sm)

    def tasks(self, sm):
        return self.per_sm[sm]


def row(start, pro, last, epi, end):
    r = np.zeros(16, dtype=np.uint64)
    r[0], r[6], r[7], r[8], r[3] = start, pro, last, epi, end
    return r


def task(op, layer):
    return {"op": op, "layer": layer, "r0": 0, "r1": 1, "b": 0, "g": 0}


def make(with_merge=True):
    """Two CTAs; layer 0's down projection ends at 1000 and 1500 ns; layer 1
    runs QKV, ATT, (MRG,) OPR on both.  Rows in CTA order, as the kernel
    writes them."""
    per_sm, rows = [[], []], [[], []]

    def add(sm, op, layer, *ts):
        per_sm[sm].append(task(op, layer))
        rows[sm].append(row(*ts))

    add(0, "DWN", 0, 100, 300, 800, 1000, 1000)
    add(1, "DWN", 0, 100, 300, 1300, 1500, 1500)
    add(0, "QKV", 1, 1000, 2500, 3000, 3200, 3200)   # inputs 1.0 us after the last DWN
    add(1, "QKV", 1, 1500, 3000, 3500, 3600, 3600)   # 1.5 us
    add(0, "ATT", 1, 3200, 4600, 5000, 5200, 5200)   # 1.0 us after the last QKV (3600)
    add(1, "ATT", 1, 0, 0, 0, 0, 0)                  # never ran: skipped
    if with_merge:
        add(0, "MRG", 1, 5200, 6200, 6300, 6400, 6400)
        add(1, "OPR", 1, 3600, 7400, 8000, 8100, 8100)  # 1.0 us after MRG (6400)
    else:
        add(1, "OPR", 1, 3600, 7200, 8000, 8100, 8100)  # 2.0 us after ATT (5200)
    trace = np.stack(rows[0] + rows[1])
    return trace, FakePlan(per_sm)


def test_prologue_lag_against_hand_computed_times():
    trace, plan = make()
    got = {x["op"]: x for x in amk.prologue_lag(trace, plan, 1)}
    assert set(got) == {"QKV", "ATT", "MRG", "OPR"}
    q = got["QKV"]
    assert q["after"] == "DWN" and q["tasks"] == 2
    assert q["lag_min_us"] == pytest.approx(1.0) and q["lag_max_us"] == pytest.approx(1.5)
    assert q["lag_median_us"] == pytest.approx(1.25)
    assert q["prologue_us"] == pytest.approx(1.5)        # 1.5 and 1.5
    assert q["tiles_us"] == pytest.approx(0.5)
    assert q["epilogue_us"] == pytest.approx(0.15)       # 0.2 and 0.1
    assert got["ATT"]["tasks"] == 1 and got["ATT"]["lag_min_us"] == pytest.approx(1.0)
    assert got["MRG"]["after"] == "ATT" and got["MRG"]["lag_min_us"] == pytest.approx(1.0)
    assert got["OPR"]["after"] == "MRG" and got["OPR"]["lag_min_us"] == pytest.approx(1.0)


def test_prologue_lag_reads_attention_when_there_is_no_merge():
    trace, plan = make(with_merge=False)
    got = {x["op"]: x for x in amk.prologue_lag(trace, plan, 1)}
    assert got["OPR"]["after"] == "ATT"
    assert got["OPR"]["lag_min_us"] == pytest.approx(2.0)


def test_level_times_chain_from_level_ends():
    trace, plan = make()
    lv = [(x["layer"], x["op"], x["level_us"]) for x in amk.level_times(trace, plan)]
    assert [x[:2] for x in lv] == [(0, "DWN"), (1, "QKV"), (1, "ATT"), (1, "MRG"), (1, "OPR")]
    assert lv[0][2] == pytest.approx(1.4)     # first level: from its first start
    assert lv[1][2] == pytest.approx(2.1)     # 3600 - 1500
    assert lv[2][2] == pytest.approx(1.6)     # 5200 - 3600
    assert lv[4][2] == pytest.approx(1.7)     # 8100 - 6400
