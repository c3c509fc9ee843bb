"""The measure-and-fit loop of the schedule simulation, pinned on the host:
step times made by the simulation itself under known constants must be
reproduced by the constants the fit recovers from them (the fit's residual
is the log ratio of simulated to measured time, so a wrong sign, a dropped
point or a mixed-up constant index shows up as a residual far from zero)."""
import math

import pytest

import synth


@pytest.fixture(scope="module")
def amk():
    import persistent_sm_decode_gb300 as m
    m.build()
    return m


def test_fit_recovers_step_times_made_by_known_constants(amk):
    from persistent_sm_decode_gb300 import costfit
    # a point of the search space per record: two tiny shapes, three schedules each, on few CTAs
    truth = list(costfit.FIRST_GUESS)
    truth[0] *= 1.6   # hand-off
    truth[4] *= 0.7   # batch-1 consumer rate
    truth[10] *= 1.4  # merge
    recs = []
    for B, opts in ((1, {"att_chunks": 2, "slot_bytes": 8192, "n_slots": 8, "ksplit": 1, "task_order": 1}),
                    (1, {"att_chunks": 4, "slot_bytes": 16384, "n_slots": 4, "ksplit": 1, "task_order": 1}),
                    (1, {"att_chunks": 1, "slot_bytes": 12288, "n_slots": 6, "ksplit": 1, "task_order": 2}),
                    (2, {"att_chunks": 2, "slot_bytes": 16384, "n_slots": 4, "ksplit": 1, "task_order": 1})):
        wl = synth.workload("tiny", batch=B)
        plan = amk.Plan(costfit._config(amk, wl, B), B, 16, options=opts)
        info = plan.info()
        knobs = {k: info[k] for k in costfit.KNOBS}
        recs.append({"workload": "tiny", "batch": B, "opts": opts, "us": plan.simulate(truth), "plan": knobs})
    plans = costfit._plans(recs, n_sm=16)
    fitted = costfit.fit_constants(plans, range(len(plans)), bound=1.1)
    for p, us, _ in plans:
        assert abs(math.log(p.simulate(fitted) / us)) < 0.02
    # and the untouched guess does not reproduce them: the test can fail
    assert max(abs(math.log(p.simulate(costfit.FIRST_GUESS) / us)) for p, us, _ in plans) > 0.05


def test_built_in_table_matches_the_library(amk):
    """costfit.BUILT_IN mirrors the library's COST_DEFAULT: a plan simulated
    under it and under the built-in constants takes the same time, on a shape
    where every constant enters (batch > 1, int8 at batch 1)."""
    from persistent_sm_decode_gb300 import costfit
    for name, B in (("tiny", 1), ("tiny", 4), ("tiny", 16)):
        for wd in ("bf16", "int8"):
            wl = synth.workload(name, batch=B, **({"weight_dtype": "int8"} if wd == "int8" else {}))
            plan = amk.Plan(costfit._config(amk, wl, B), B, 16)
            assert plan.simulate(costfit.BUILT_IN) == pytest.approx(plan.simulate(None), rel=1e-12)
    # and a change of any one constant moves some simulated step
    wl = synth.workload("tiny", batch=4)
    plan = amk.Plan(costfit._config(amk, wl, 4), 4, 16)
    base = plan.simulate(costfit.BUILT_IN)
    for i in (0, 1, 2, 3, 7, 9, 10, 11, 12, 14):
        c = list(costfit.BUILT_IN)
        c[i] *= 2
        assert plan.simulate(c) != pytest.approx(base, rel=1e-9), i


def test_refit_recovers_two_constants_from_a_bench_line(amk, tmp_path):
    """costfit.refit on a bench.py-shaped JSON line whose step times the
    simulation made under known values of [12] and [14]: the refit lands on
    those values, and a record whose schedule differs from the host plan is
    left out."""
    import json
    from persistent_sm_decode_gb300 import costfit
    truth = list(costfit.BUILT_IN)
    truth[12] *= 1.5
    truth[14] *= 0.8
    n_sm = 16

    def record(B):
        wl = synth.workload("tiny", batch=B)
        plan = amk.Plan(costfit._config(amk, wl, B), B, n_sm)
        info = plan.info()
        return {"config": {"workload": "tiny", "batch": B}, "ms_per_step": plan.simulate(truth) / 1e3,
                "schedule": {k: info[k] for k in ("att_chunks", "slot_bytes", "n_slots", "ksplit")}}

    line = record(1)
    line["schedule"]["n_sm"] = n_sm
    subs = {"tiny@%d" % B: record(B) for B in (2, 4, 8, 16)}
    stray = record(3)
    stray["schedule"]["slot_bytes"] += 4096  # not what the host plans: left out
    subs["tiny@3"] = stray
    line["workloads"] = subs
    path = tmp_path / "bench.json"
    path.write_text("not json, a log line\n" + json.dumps(line) + "\n")
    assert len(costfit.bench_points(str(path))) == 5
    got = costfit.refit(str(path), [12, 14])
    assert got[12] == pytest.approx(truth[12], rel=0.03)
    assert got[14] == pytest.approx(truth[14], rel=0.03)
    assert [got[i] for i in range(15) if i not in (12, 14)] == [costfit.BUILT_IN[i] for i in range(15)
                                                                if i not in (12, 14)]
