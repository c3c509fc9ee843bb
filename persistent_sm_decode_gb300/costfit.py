"""Measure-and-fit loop for the offline search's task-level simulation
(Ada-MK technical summary, Methodology, Phase I: the offline search scores
candidate execution traces; the scores are only as good as the constants).

    python -m persistent_sm_decode_gb300.costfit measure campaign.jsonl   # GPU
    python -m persistent_sm_decode_gb300.costfit fit campaign.jsonl       # CPU
    python -m persistent_sm_decode_gb300.costfit refit bench.json 12,14   # CPU

`measure` times every point of POINTS (a workload, a batch and schedule
options) with the device-filled inputs of bench.py and appends one JSON line
per point: the median of three timed runs and the plan's knobs.  `fit` finds
the simulation constants (amk_plan_simulate's fifteen) that minimise the
squared log ratio of simulated to measured step time, each constant held
within a factor e^bound of its physical first guess in FIRST_GUESS, prints
the fitted table and, for every workload, the errors of a fit made without
it.  The HBM rate stays at the measured copy rate.  `refit` takes the JSON
line of a `bench.py` run instead, whose records are the default schedules,
and refits only the listed constants, the others held at BUILT_IN (the
library's built-in table): it brings a few constants up to date after a
kernel change that leaves the schedules alone.
"""
import json
import math
import sys
from typing import List, Sequence

# (workload, batch, schedule options)
POINTS = [
    ("tinyllama_1b1", 1, {}), ("tinyllama_1b1", 1, {"task_order": 1}), ("tinyllama_1b1", 1, {"task_order": 2}),
    ("tinyllama_1b1", 1, {"slot_bytes": 32768}), ("tinyllama_1b1", 1, {"slot_bytes": 49152}),
    ("tinyllama_1b1", 1, {"att_chunks": 16}), ("tinyllama_1b1", 1, {"att_chunks": 24}),
    ("tinyllama_1b1_w8a16", 1, {}), ("tinyllama_1b1_w8a16", 1, {"task_order": 1}),
    ("smollm2_135m", 1, {"slot_bytes": 32768, "n_slots": 6}), ("smollm2_135m", 1, {"slot_bytes": 65536, "n_slots": 3}),
    ("llama2_7b", 1, {}), ("llama2_7b", 1, {"task_order": 1}), ("llama2_7b", 1, {"att_chunks": 8}),
    ("llama2_7b_b8", 8, {"att_chunks": 4}), ("llama2_7b_b8", 8, {"att_chunks": 7}),
    ("llama2_7b_b8", 8, {"att_chunks": 8}),
    ("tinyllama_1b1_short", 1, {}), ("tinyllama_1b1_short", 2, {"slot_bytes": 49152, "n_slots": 3}),
    ("tinyllama_1b1_short", 2, {"slot_bytes": 61440, "n_slots": 3}), ("tinyllama_1b1_short", 4, {}),
    ("tinyllama_1b1_short", 8, {"slot_bytes": 49152, "n_slots": 2}),
    ("tinyllama_1b1_short", 8, {"slot_bytes": 61440, "n_slots": 2}), ("tinyllama_1b1_short", 16, {}),
    ("smollm2_135m", 1, {"slot_bytes": 40960, "n_slots": 5}),
]

FIRST_GUESS = [1.5e-6, 0.5e-6, 0.4e-6, 0.6e-6, 7.5e10, 5.0e10, 6.5e12, 0.5e-6, 2.0e-12, 0.8e-6, 0.5e-6, 0.1e-6,
               0.6e-6, 1.5e11, 2.5e10]
FITTED = [0, 1, 2, 3, 4, 5, 7, 8, 9, 10, 11, 12, 13, 14]  # [6], the HBM rate, is measured, not fitted

# The library's built-in constants (COST_DEFAULT in amk_plan.cpp), in the
# same order; a test checks that the two agree.
BUILT_IN = [1.73e-6, 0.166e-6, 0.133e-6, 0.211e-6, 6.87e10, 2.67e10, 6.5e12, 1.5e-6, 6.01e-12, 1.93e-6, 1.5e-6,
            0.247e-6, 0.339e-6, 3.55e11, 2.69e10]

KNOBS = ("att_chunks", "slot_bytes", "n_slots", "ksplit", "task_order")


def _config(amk, wl, batch):
    return amk.make_config(wl.n_layers, wl.hidden, wl.n_heads, wl.n_kv_heads, wl.head_dim, wl.intermediate,
                           wl.vocab, wl.max_seq, batch, wl.rms_eps, wl.rope_theta, int8=wl.weight_dtype == "int8",
                           tied=wl.tied, int4=wl.weight_dtype == "int4", group_size=wl.group_size)


def measure(path: str, points=POINTS) -> None:
    import torch
    import bench
    import synth
    import persistent_sm_decode_gb300 as amk
    amk.build()
    out = open(path, "a")
    cache = {}
    for name, B, opts in points:
        wl = synth.workload(name, batch=B)
        if (name, B) not in cache:
            cache.clear()
            torch.cuda.empty_cache()
            cache[(name, B)] = (bench.device_model(wl, seed=1), bench.device_kv(wl, seed=2, batch=B))
        dev, kv = cache[(name, B)]
        eng = bench.make_engine(amk, wl, dev, opts)
        steps = 256 if wl.n_layers * B < 100 else 64
        ts = [bench.Timed(amk, eng, wl, kv, steps=steps, warmup=8, local=0).ms_per_step * 1e3 for _ in range(3)]
        info = eng.plan_info()
        rec = {"workload": name, "batch": B, "opts": opts, "us": sorted(ts)[1],
               "plan": {k: info[k] for k in KNOBS + ("simulated_us",)}}
        print(json.dumps(rec), flush=True)
        out.write(json.dumps(rec) + "\n")
        eng.close()


def _constants(x: Sequence[float]) -> List[float]:
    c = list(FIRST_GUESS)
    for i, v in zip(FITTED, x):
        c[i] = FIRST_GUESS[i] * math.exp(v)
    return c


def _plans(recs, n_sm: int = 152):
    import synth
    import persistent_sm_decode_gb300 as amk
    plans = []
    for r in recs:
        wl = synth.workload(r["workload"], batch=r["batch"])
        opts = {k: r["plan"][k] for k in KNOBS}
        plans.append((amk.Plan(_config(amk, wl, r["batch"]), r["batch"], n_sm, options=opts), r["us"], r))
    return plans


def fit_constants(plans, sel, bound: float = 1.1) -> List[float]:
    """The fitted constants for the points `sel` of `plans` [(plan, measured
    µs, record)]."""
    import numpy as np
    from scipy.optimize import least_squares
    res = lambda x: [np.log(plans[i][0].simulate(_constants(x)) / plans[i][1]) for i in sel]
    return _constants(least_squares(res, np.zeros(len(FITTED)), bounds=(-bound, bound), diff_step=0.05).x)


def fit(path: str, bound: float = 1.1) -> List[float]:
    recs = [json.loads(ln) for ln in open(path) if ln.strip()]
    plans = _plans(recs)
    solve = lambda sel: fit_constants(plans, sel, bound)

    c = solve(range(len(plans)))
    print("constants:", ", ".join("%.3g" % v for v in c))
    print("| workload | batch | options | measured µs | simulated µs | error |")
    print("|---|---|---|---|---|---|")
    for p, us, r in plans:
        s = p.simulate(c)
        print("| %s | %d | %s | %.1f | %.1f | %+.1f %% |" % (r["workload"], r["batch"], json.dumps(r["opts"]) or "-",
                                                        us, s, 100 * (s / us - 1)))
    print()
    print("| held-out workload | batch | errors of a fit without it |")
    print("|---|---|---|")
    for key in sorted({(r["workload"], r["batch"]) for _, _, r in plans}):
        train = [i for i, (_, _, r) in enumerate(plans) if (r["workload"], r["batch"]) != key]
        test = [i for i, (_, _, r) in enumerate(plans) if (r["workload"], r["batch"]) == key]
        cx = solve(train)
        print("| %s | %d | %s |" % (key[0], key[1], " ".join("%+.1f %%" % (100 * (plans[i][0].simulate(cx) /
                                                                                 plans[i][1] - 1)) for i in test)))
    return c


def bench_points(path: str):
    """[(plan, measured µs, name)] of a bench.py JSON line (the last line of
    the file): the headline and every sub-record that carries a schedule,
    each planned on the host with the default search.  A record whose host
    plan differs from the schedule it ran is left out, with a note."""
    import synth
    import persistent_sm_decode_gb300 as amk
    d = json.loads([ln for ln in open(path) if ln.strip()][-1])
    n_sm = d["schedule"]["n_sm"]
    recs = [(d["config"]["workload"], d)] + [(k, v) for k, v in (d.get("workloads") or {}).items()
                                             if "schedule" in v]
    out = []
    for key, r in recs:
        name, B = r["config"]["workload"], int(r["config"]["batch"])
        wl = synth.workload(name, batch=B)
        plan = amk.Plan(_config(amk, wl, B), B, n_sm)
        info = plan.info()
        ran = r["schedule"]
        if any(info[k] != ran[k] for k in ("att_chunks", "slot_bytes", "n_slots", "ksplit")):
            print("left out %s: the host plan differs from the schedule it ran" % key)
            continue
        out.append((plan, r["ms_per_step"] * 1e3, "%s@%d" % (name, B)))
    return out


def refit(path: str, idx: Sequence[int], bound: float = 1.1) -> List[float]:
    """Refit the constants `idx` to a bench.py line, the others held at
    BUILT_IN; each fitted constant within a factor e^bound of its built-in
    value.  Prints the errors before and after."""
    import numpy as np
    from scipy.optimize import least_squares
    pts = bench_points(path)
    idx = list(idx)

    def consts(x):
        c = list(BUILT_IN)
        for i, v in zip(idx, x):
            c[i] = BUILT_IN[i] * math.exp(v)
        return c

    res = lambda x: [math.log(p.simulate(consts(x)) / us) for p, us, _ in pts]
    c = consts(least_squares(res, np.zeros(len(idx)), bounds=(-bound, bound), diff_step=0.05).x)
    print("refitted:", ", ".join("[%d] %.3g -> %.3g" % (i, BUILT_IN[i], c[i]) for i in idx))
    print("| workload | measured µs | built-in | refitted |")
    print("|---|---|---|---|")
    for p, us, name in pts:
        a, b = p.simulate(BUILT_IN), p.simulate(c)
        print("| %s | %.1f | %.1f (%+.1f %%) | %.1f (%+.1f %%) |" % (name, us, a, 100 * (a / us - 1), b,
                                                                   100 * (b / us - 1)))
    return c


if __name__ == "__main__":
    if len(sys.argv) < 3 or sys.argv[1] not in ("measure", "fit", "refit"):
        sys.exit(__doc__)
    if sys.argv[1] == "measure":
        measure(sys.argv[2])
    elif sys.argv[1] == "refit":
        refit(sys.argv[2], [int(v) for v in sys.argv[3].split(",")] if len(sys.argv) > 3 else [12, 14])
    else:
        fit(sys.argv[2], float(sys.argv[3]) if len(sys.argv) > 3 else 1.1)
