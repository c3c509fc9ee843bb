"""CPU tests of the C ABI library and the offline planner (no GPU needed).

* libamk.so loads on a machine without a GPU and exports every function that
  include/*.h declares.
* Plans build and pass the validator for every workload and many CTA counts.
* Solidified tables cover every output row exactly once per layer.
* Adversarial schedules: plans mutated in six ways are judged by the C++
  validator and, independently, by a brute-force checker written here from
  the task semantics (transitive closure of program order and counter edges,
  then every conflicting access pair).  The validator must never accept a
  schedule the checker finds unsafe.
"""
import os
import re

import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def amk():
    import persistent_sm_decode_gb300 as m
    m.build()
    return m


def _cfg(amk, wl, batch=None):
    return amk.make_config(wl.n_layers, wl.hidden, wl.n_heads, wl.n_kv_heads, wl.head_dim, wl.intermediate,
                           wl.vocab, wl.max_seq, batch or wl.batch, wl.rms_eps, wl.rope_theta,
                           int8=wl.weight_dtype == "int8", tied=wl.tied,
                          int4=wl.weight_dtype == "int4", group_size=wl.group_size)


def test_library_exports_every_declared_symbol(amk):
    lib = amk.lib()
    names = set()
    for h in ("amk.h", "amk_plan.h", "amk_unfused.h"):
        src = open(os.path.join(ROOT, "include", h)).read()
        names |= set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]*?\b(amk_\w+)\s*\(", src, re.M))
    assert len(names) == 24 and {"amk_create", "amk_decode_step", "amk_decode_step_greedy", "amk_destroy",
                                 "amk_plan_build"} <= names, names
    for n in sorted(names):
        assert hasattr(lib, n), "libamk.so does not export %s" % n


def test_status_strings(amk):
    for s in range(8):
        assert amk.lib().amk_status_string(s)


@pytest.mark.parametrize("name", sorted(synth.WORKLOADS))
def test_plans_validate_for_every_workload(amk, name):
    wl = synth.workload(name)
    p = amk.Plan(_cfg(amk, wl), wl.batch, 152)
    info = p.info()
    assert info["n_levels"] == 6 * wl.n_layers + 2  # six per layer, the LM head, the greedy argmax
    assert info["smem_bytes"] <= 232448
    assert p.validate()[0] == amk.OK
    assert info["weight_bytes"] == wl.weight_bytes() - (2 * wl.n_layers + 1) * wl.hidden * 2


@pytest.mark.parametrize("n_sm", [1, 2, 7, 33, 148, 152])
def test_plans_for_any_cta_count(amk, n_sm):
    wl = synth.workload("tiny", batch=2)
    p = amk.Plan(_cfg(amk, wl), 2, n_sm)
    assert p.validate()[0] == amk.OK
    _coverage(wl, p, 2)


def test_schedule_options_reach_the_planner(amk):
    # the last options field and the last plan-info field: a layout mismatch
    # between the binding's structures and include/amk.h shows up here
    wl = synth.workload("tiny")
    assert amk.Plan(_cfg(amk, wl), 1, 152).info()["l2_evict_first"] == 1
    off = amk.Plan(_cfg(amk, wl), 1, 152, options={"l2_evict_first": -1, "wait_timeout_ns": 5})
    assert off.info()["l2_evict_first"] == 0
    on = amk.Plan(_cfg(amk, wl), 1, 152, options={"l2_evict_first": 1, "att_chunks": 3})
    assert on.info()["l2_evict_first"] == 1 and on.info()["att_chunks"] == 3


def test_default_build_refuses_the_trace_option(amk):
    # the default library carries no per-task timing code; amk_create says so
    # before it touches the device (AMK_TRACE=1 builds the tuning variant)
    import ctypes
    import os
    if os.environ.get("AMK_TRACE", "0") not in ("", "0"):
        pytest.skip("timing build")
    wl = synth.workload("tiny")
    h = ctypes.c_void_p()
    opts = amk.ScheduleOptions(trace=1)
    st = amk.lib().amk_create(ctypes.byref(_cfg(amk, wl)), None, ctypes.byref(opts), ctypes.byref(h))
    assert st == amk.ERR_UNSUPPORTED and not h.value


def test_headline_schedule_is_the_measured_best_point(amk):
    # the 1.1B bf16 shape on 152 CTAs: the point the slot and chunk sweeps
    # measured fastest on GB300; a cost-model change that moves it needs a
    # new measurement
    wl = synth.workload("tinyllama_1b1")
    info = amk.Plan(_cfg(amk, wl), 1, 152).info()
    assert (info["slot_bytes"], info["n_slots"], info["att_chunks"], info["ksplit"]) == (65536, 3, 32, 1)
    assert info["l2_evict_first"] == 1 and info["smem_bytes"] <= 232448


def test_schedule_simulation_entry_point(amk):
    # amk_plan_simulate takes exactly fifteen constants (or none, for the
    # built-in fit) and its step time moves the way the model says: a slower
    # hand-off, a slower HBM or a slower consumer never makes a step faster
    wl = synth.workload("tinyllama_1b1")
    plan = amk.Plan(_cfg(amk, wl), 1, 152)
    base = [1.8e-6, 0.17e-6, 0.13e-6, 0.48e-6, 6.75e10, 2.63e10, 6.5e12, 1.5e-6, 6e-12, 0.27e-6, 1.5e-6,
            0.23e-6, 0.38e-6, 1.67e11, 1.77e10]
    t0 = plan.simulate(base)
    assert t0 > 0 and abs(plan.simulate(base) - t0) == 0.0
    assert abs(plan.simulate() - plan.info()["simulated_us"]) < 1e-6
    with pytest.raises(Exception):
        plan.simulate(base[:14])
    for i, f in ((0, 2.0), (6, 0.5), (4, 0.5), (10, 2.0)):
        c = list(base)
        c[i] *= f
        assert plan.simulate(c) > t0, i
    # the batched consumer rate only matters above batch 1
    c = list(base)
    c[14] *= 0.5
    assert plan.simulate(c) == t0
    plan8 = amk.Plan(_cfg(amk, synth.workload("llama2_7b_b8")), 8, 152)
    assert plan8.simulate(c) > plan8.simulate(base)


def _coverage(wl, plan, B):
    d, nq, nkv = wl.head_dim, wl.n_heads, wl.n_kv_heads
    rows = {"QKV": (nq + 2 * nkv) * d, "OPR": wl.hidden, "GUP": wl.intermediate, "DWN": wl.hidden, "LMH": wl.vocab}
    seen = {}
    C = plan.info()["att_chunks"]
    att = set()
    for sm in range(plan.n_sm):
        for t in plan.tasks(sm):
            if t["op"] == "ATT":
                key = (t["layer"], t["b"], t["g"], t["r0"])
                assert key not in att
                att.add(key)
                continue
            if t["op"] == "MRG":
                key = ("MRG", t["layer"], t["b"], t["g"])
                assert key not in seen
                seen[key] = 1
                continue
            base = 0
            if t["op"] == "QKV":
                base = [0, nq * d, (nq + nkv) * d][t["mat"]]
            for r in range(t["r0"] + base, t["r1"] + base):
                k = (t["op"], t["layer"], r)
                assert k not in seen, "row covered twice: %r" % (k,)
                seen[k] = 1
    for op, n in rows.items():
        layers = [wl.n_layers - 1] if op == "LMH" else range(wl.n_layers)
        for l in layers:
            for r in range(n):
                assert (op, l, r) in seen, "row not covered: %s layer %d row %d" % (op, l, r)
    assert len(att) == wl.n_layers * B * nkv * C
    assert all(("MRG", l, b, h) in seen for l in range(wl.n_layers) for b in range(B) for h in range(nq))


def test_rejects_bad_configs(amk):
    wl = synth.workload("tiny")
    for bad in ({"head_dim": 96}, {"n_kv_heads": 3}, {"max_batch": 17}, {"hidden": 250}):
        c = _cfg(amk, wl)
        for k, v in bad.items():
            setattr(c, k, v)
        with pytest.raises(amk.AmkError):
            amk.Plan(c, min(c.max_batch, 16), 16)


# ------------------------------------------------------- independent checker

def brute_force_unsafe(wl, plan, B, depth):
    """Returns a reason string if the schedule can deadlock or race, else ''."""
    d, nq, nkv, G = wl.head_dim, wl.n_heads, wl.n_kv_heads, wl.group
    H, I, L = wl.hidden, wl.intermediate, wl.n_layers
    C = plan.info()["att_chunks"]
    tasks = []
    for sm in range(plan.n_sm):
        for i, t in enumerate(plan.tasks(sm)):
            tasks.append((sm, i, t))
    idx = {(sm, i): k for k, (sm, i, _) in enumerate(tasks)}
    n = len(tasks)
    prod = {}
    for k, (_, _, t) in enumerate(tasks):
        for c in t["sig"]:
            prod.setdefault(c, []).append(k)
    preds = [set() for _ in range(n)]
    for k, (sm, i, t) in enumerate(tasks):
        if i > 0:
            preds[k].add(idx[(sm, i - 1)])
        if t["wait"] >= 0:
            p = prod.get(t["wait"], [])
            if t["wait_count"] > len(p):
                return "wait can never be met"
            if t["wait_count"] == len(p):
                preds[k] |= set(p)
            # fewer than all producers: no particular producer is guaranteed
    # deadlock: cycle in preds
    state = [0] * n
    order = []
    for s in range(n):
        if state[s]:
            continue
        stack = [(s, iter(preds[s]))]
        state[s] = 1
        while stack:
            v, it = stack[-1]
            nxt = next(it, None)
            if nxt is None:
                state[v] = 2
                order.append(v)
                stack.pop()
            elif state[nxt] == 1:
                return "cycle"
            elif state[nxt] == 0:
                state[nxt] = 1
                stack.append((nxt, iter(preds[nxt])))
    anc = [None] * n
    for v in order:  # predecessors first
        a = set()
        for p in preds[v]:
            a.add(p)
            a |= anc[p]
        anc[v] = a

    def hb(x, y):
        return x in anc[y]

    qd, kd = nq * d, nkv * d
    acc = []  # (task, buf, version, write, b0, b1, e0, e1)
    for k, (_, _, t) in enumerate(tasks):
        l, op = t["layer"], t["op"]
        if op == "QKV":
            base = [0, qd, qd + kd][t["mat"]]
            if l > 0:
                acc.append((k, "xin", l, 0, 0, B, 0, H))
            acc.append((k, "qkv", l, 1, 0, B, base + t["r0"], base + t["r1"]))
        elif op == "ATT":
            b, g, c = t["b"], t["g"], t["r0"]
            for lo in (g * G * d, qd + g * d, qd + kd + g * d):
                hi = lo + (G * d if lo == g * G * d else d)
                acc.append((k, "qkv", l, 0, b, b + 1, lo, hi))
            # partials are head-major: [kv head][q head of the group][chunk]
            for hh in range(G):
                e = (g * G + hh) * C + c
                acc.append((k, "part", l, 1, b, b + 1, e, e + 1))
        elif op == "MRG":
            # one merge per query head h of sequence b
            b, h = t["b"], t["g"]
            acc.append((k, "part", l, 0, b, b + 1, h * C, (h + 1) * C))
            acc.append((k, "aout", l, 1, b, b + 1, h * d, (h + 1) * d))
        elif op == "OPR":
            acc.append((k, "aout", l, 0, 0, B, 0, nq * d))
            if l > 0:
                acc.append((k, "xin", l, 0, 0, B, t["r0"], t["r1"]))
            acc.append((k, "xmid", l, 1, 0, B, t["r0"], t["r1"]))
        elif op == "GUP":
            acc.append((k, "xmid", l, 0, 0, B, 0, H))
            acc.append((k, "act", l, 1, 0, B, t["r0"], t["r1"]))
        elif op == "DWN":
            acc.append((k, "act", l, 0, 0, B, 0, I))
            acc.append((k, "xmid", l, 0, 0, B, t["r0"], t["r1"]))
            acc.append((k, "xin", l + 1, 1, 0, B, t["r0"], t["r1"]))
        elif op == "LMH":
            acc.append((k, "xin", L, 0, 0, B, 0, H))
    by = {}
    for a in acc:
        by.setdefault((a[1], a[2] % depth), []).append(a)
    for (buf, _), lst in by.items():
        writes = [a for a in lst if a[3]]
        for a in lst:
            for w in writes:
                if a is w or a[0] == w[0]:
                    continue
                if not (a[4] < w[5] and w[4] < a[5] and a[6] < w[7] and w[6] < a[7]):
                    continue
                va, vw = a[2], w[2]
                if a[3]:  # write/write
                    if va == vw:
                        return "double write"
                    older, newer = (a, w) if va < vw else (w, a)
                    if not hb(older[0], newer[0]):
                        return "WAW"
                elif vw == va:
                    if not hb(w[0], a[0]):
                        return "RAW on %s" % buf
                elif vw > va:
                    if not hb(a[0], w[0]):
                        return "WAR on %s" % buf
                else:
                    if not hb(w[0], a[0]):
                        return "stale read on %s" % buf
        # coverage of reads
        for a in lst:
            if a[3]:
                continue
            for b in range(a[4], a[5]):
                iv = sorted((w[6], w[7]) for w in writes if w[2] == a[2] and w[4] <= b < w[5])
                cur = a[6]
                for lo, hi in iv:
                    if lo <= cur:
                        cur = max(cur, hi)
                if cur < a[7]:
                    return "uncovered read on %s" % buf
    return ""


@pytest.mark.parametrize("n_sm,B,depth", [(3, 1, 2), (6, 2, 1), (8, 1, 3)])
def test_real_plans_are_safe_by_brute_force(amk, n_sm, B, depth):
    wl = synth.workload("tiny", batch=B)
    p = amk.Plan(_cfg(amk, wl), B, n_sm, options={"scratch_depth": depth})
    assert brute_force_unsafe(wl, p, B, depth) == ""


def test_adversarial_schedules_have_no_false_accepts(amk):
    stats = {"total": 0, "unsafe": 0, "rejected": 0, "false_accepts": 0, "false_rejects": 0}
    for n_sm, B, depth in ((3, 1, 2), (5, 2, 1), (8, 1, 2)):
        wl = synth.workload("tiny", batch=B)
        for kind in range(6):
            for seed in range(12):
                p = amk.Plan(_cfg(amk, wl), B, n_sm, options={"scratch_depth": depth, "att_chunks": 2})
                if p.mutate(kind, seed) != amk.OK:
                    p.close()
                    continue
                verdict, why = p.validate()
                truth = brute_force_unsafe(wl, p, B, depth)
                stats["total"] += 1
                stats["unsafe"] += bool(truth)
                stats["rejected"] += verdict != amk.OK
                if truth and verdict == amk.OK:
                    stats["false_accepts"] += 1
                if not truth and verdict != amk.OK:
                    stats["false_rejects"] += 1
                if kind in (0, 1, 5):
                    assert verdict != amk.OK, (kind, seed)  # counts no longer match producers
                p.close()
    assert stats["total"] > 150, stats
    assert stats["unsafe"] > 100, stats
    assert stats["false_accepts"] == 0, stats
