"""Host side of the tuning trace: the Chrome trace-event export and the
per-level breakdown, on a synthetic trace laid out as amk_debug_read_trace
returns it (tasks in CTA order, sixteen entries each)."""
import json

import numpy as np
import pytest

import synth


@pytest.fixture(scope="module")
def plan():
    import persistent_sm_decode_gb300 as amk
    amk.build()
    wl = synth.workload("tiny")
    cfg = amk.make_config(wl.n_layers, wl.hidden, wl.n_heads, wl.n_kv_heads, wl.head_dim, wl.intermediate,
                          wl.vocab, wl.max_seq, 1, wl.rms_eps, wl.rope_theta)
    return amk.Plan(cfg, 1, 6)


def _synthetic(plan):
    """Task k of CTA s starts at 1 µs + 1000 k + 10 s ns: prologue 100 ns, tiles
    200 ns, epilogue 100 ns, end 50 ns later."""
    rows = []
    for sm in range(plan.n_sm):
        for k, _ in enumerate(plan.tasks(sm)):
            s = 1000 + 1000 * k + 10 * sm
            r = np.zeros(16, dtype=np.uint64)
            r[0] = r[1] = s
            r[2] = s + 100
            r[3] = s + 450
            r[4], r[5] = 20, 180
            r[6], r[7], r[8] = s + 100, s + 300, s + 400
            r[9] = 7
            rows.append(r)
    return np.array(rows)


def test_chrome_trace_has_one_track_per_cta_and_nested_phases(plan):
    import persistent_sm_decode_gb300 as amk
    tr = _synthetic(plan)
    doc = amk.chrome_trace(tr, plan)
    json.dumps(doc)  # serialisable as is
    ev = doc["traceEvents"]
    slices = [e for e in ev if e["ph"] == "X"]
    tasks = [e for e in slices if e["name"] not in ("inputs + prologue", "tiles", "epilogue")]
    n_tasks = sum(len(plan.tasks(sm)) for sm in range(plan.n_sm))
    assert len(tasks) == n_tasks and len(slices) == 4 * n_tasks
    assert {e["tid"] for e in tasks} == set(range(plan.n_sm))
    assert min(e["ts"] for e in slices) == 0.0
    first = next(e for e in tasks if e["tid"] == 2)
    assert first["ts"] == pytest.approx(0.02) and first["dur"] == pytest.approx(0.45)
    assert first["args"]["tile_us"] == pytest.approx(0.18) and first["args"]["loader_wait_us"] == pytest.approx(0.007)
    # the phases of a task lie inside it, in order
    kids = [e for e in slices if e["tid"] == 2 and e["name"] in ("inputs + prologue", "tiles", "epilogue")][:3]
    assert [k["name"] for k in kids] == ["inputs + prologue", "tiles", "epilogue"]
    assert [k["dur"] for k in kids] == pytest.approx([0.1, 0.2, 0.1])
    for k in kids:
        assert first["ts"] <= k["ts"] and k["ts"] + k["dur"] <= first["ts"] + first["dur"] + 1e-9
    names = [e["args"]["name"] for e in ev if e["ph"] == "M" and e["name"] == "thread_name"]
    assert names == ["CTA %d" % i for i in range(plan.n_sm)]


def test_tasks_that_did_not_run_are_left_out(plan):
    import persistent_sm_decode_gb300 as amk
    tr = _synthetic(plan)
    tr[0, :] = 0
    doc = amk.chrome_trace(tr, plan)
    n_tasks = sum(len(plan.tasks(sm)) for sm in range(plan.n_sm))
    assert sum(1 for e in doc["traceEvents"] if e["ph"] == "X") == 4 * (n_tasks - 1)


def test_level_times_follow_program_order_and_add_up(plan):
    import persistent_sm_decode_gb300 as amk
    tr = _synthetic(plan)
    lv = amk.level_times(tr, plan)
    ops = [(x["layer"], x["op"]) for x in lv]
    L = max(l for l, _ in ops)
    assert ops[:6] == [(0, "QKV"), (0, "ATT"), (0, "MRG"), (0, "OPR"), (0, "GUP"), (0, "DWN")]
    # the LM head, then the greedy argmax (which runs when a step asks for it)
    assert ops[-2:] == [(L, "LMH"), (L, "ARG")]
    assert all(x["level_us"] >= 0 for x in lv)
    # the levels tile the step: their times add up to last end - first start
    total = sum(x["level_us"] for x in lv)
    assert total == pytest.approx((int(tr[:, 3].max()) - int(tr[:, 0].min())) / 1e3)
