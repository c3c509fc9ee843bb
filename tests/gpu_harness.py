"""Shared GPU-test machinery: build an engine from a synth workload and run
teacher-forced decode against the CPU oracle.

Acceptance: at every step and every checked sequence,
    max |logit_gpu - logit_oracle| <= 1e-2 * max |logit_oracle| + 1e-3,
and wherever the oracle's top-1 minus top-2 margin exceeds 1e-2 the GPU's
argmax equals the oracle's.  Both sides consume the oracle's token at every
step (teacher forcing), so one near-tie cannot derail the rest of a sequence.
"""
from __future__ import annotations

import numpy as np

import oracle
import synth
from synth.device import kv_from_device, kv_rows_from_device, kv_to_device, model_to_device

REL_TOL = 1e-2
ABS_TOL = 1e-3
MARGIN = 1e-2


def log_parity(kind: str, record: dict) -> None:
    """Append one test's measured parity figures to the JSON-lines file named
    by AMK_PARITY_LOG (nothing without it).  tests/parity_report.py turns the
    file into the committed per-configuration table."""
    import json
    import os
    path = os.environ.get("AMK_PARITY_LOG")
    if not path:
        return
    rec = {"test": os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0], "kind": kind}
    rec.update(record)
    with open(path, "a") as f:
        f.write(json.dumps(rec) + "\n")


def engine_config(wl, max_batch=None):
    import persistent_sm_decode_gb300 as amk
    return amk.make_config(wl.n_layers, wl.hidden, wl.n_heads, wl.n_kv_heads, wl.head_dim, wl.intermediate,
                           wl.vocab, wl.max_seq, max_batch or wl.batch, wl.rms_eps, wl.rope_theta,
                           int8=wl.weight_dtype == "int8", tied=wl.tied,
                          int4=wl.weight_dtype == "int4", group_size=wl.group_size)


def make_engine(wl, dev, options=None, max_batch=None):
    import persistent_sm_decode_gb300 as amk
    return amk.DecodeEngine(engine_config(wl, max_batch), dev["embed"], dev["final_norm"], dev["layers"],
                            dev["lm_head"], dev["s_lm"], options)


class Result:
    def __init__(self):
        self.worst = 0.0          # max over steps/rows of max|d| / (REL*max|ref| + ABS)
        self.max_abs = 0.0
        self.checked_argmax = 0
        self.argmax_agree = 0
        self.floor = 0.0          # same ratio for the fp32-accumulation build of the definition
        self.steps = 0
        self.records = []         # (step, row, margin, gpu agrees, fp32-build max|dlogit| or None)

    @property
    def free_running(self) -> int:
        """Steps over which the GPU's own greedy stream equals the oracle's for
        every checked sequence: up to the first step where an argmax differs.
        Until then teacher forcing feeds both sides the tokens a free-running
        decode would, so no second run is needed."""
        first = [s for (s, _b, _m, agree, _f) in self.records if not agree]
        return min(first) if first else self.steps

    def relaxed_misses(self):
        """Argmax disagreements that the deep-stack rule still counts: margin
        above both 1e-2 and twice what fp32 rounding alone moved the logits."""
        return [r for r in self.records if not r[3] and r[2] > max(MARGIN, 2.0 * (r[4] or 0.0))]

    def summary(self) -> dict:
        rows = sorted({r[1] for r in self.records})
        return {"steps": int(self.steps), "rows": [int(r) for r in rows], "worst": float(self.worst),
                "floor": float(self.floor), "max_abs": float(self.max_abs), "strict_logits_ok": bool(self.worst <= 1.0),
                "argmax_checked": int(self.checked_argmax), "argmax_agree": int(self.argmax_agree),
                "strict_argmax_ok": bool(self.argmax_agree == self.checked_argmax),
                "relaxed_misses": len(self.relaxed_misses()), "free_running": int(self.free_running),
                "min_margin": float(min((r[2] for r in self.records), default=float("nan")))}

    def __repr__(self):
        return ("Result(worst=%.3g, floor=%.3g, max_abs=%.3g, argmax %d/%d, steps=%d, free-running %d)"
                % (self.worst, self.floor, self.max_abs, self.argmax_agree, self.checked_argmax, self.steps,
                   self.free_running))


def teacher_forced(wl, model=None, kv=None, steps=None, options=None, batch=None, positions0=None,
                   check_rows=None, dev=None, engine=None, check_cache=True, floor=False):
    """Run `steps` decode steps on the GPU and the oracle; return a Result.
    With floor=True the fp32-accumulation build of the definition runs beside
    the oracle on the same tokens, and res.floor records how far it lands."""
    import torch
    B = batch or wl.batch
    steps = wl.steps if steps is None else steps
    model = model or synth.make_model(wl, seed=1)
    kc, vc = kv if kv is not None else synth.make_kv(wl, seed=2, batch=B)
    rows = list(range(B)) if check_rows is None else list(check_rows)
    dev = dev or model_to_device(model)
    eng = engine or make_engine(wl, dev, options, max_batch=B)
    kv_dev = kv_to_device(kc, vc)
    orc = oracle.Oracle(model, np.ascontiguousarray(kc[:, rows]), np.ascontiguousarray(vc[:, rows]))
    o32 = (oracle.Oracle(model, np.ascontiguousarray(kc[:, rows]), np.ascontiguousarray(vc[:, rows]),
                         oracle.lib_fp32_accumulation()) if floor else None)
    tokens = synth.initial_tokens(wl, B).copy()
    pos = np.full(B, wl.ctx, dtype=np.int32) if positions0 is None else np.array(positions0, dtype=np.int32)
    pos0 = pos.copy()
    logits = torch.empty((B, wl.vocab), dtype=torch.float32, device="cuda")
    res = Result()
    for s in range(steps):
        t_dev = torch.from_numpy(tokens).cuda()
        p_dev = torch.from_numpy(pos).cuda()
        eng.step(t_dev, p_dev, kv_dev, logits)
        st = eng.sync()
        assert st == 0, "device error %d: %s" % (st, eng.last_error())
        got = logits.cpu().numpy().astype(np.float64)
        ref = orc.step(tokens[rows], pos[rows])
        for i, b in enumerate(rows):
            d = np.abs(got[b] - ref[i])
            bound = REL_TOL * np.abs(ref[i]).max() + ABS_TOL
            res.worst = max(res.worst, float(d.max() / bound))
            res.max_abs = max(res.max_abs, float(d.max()))
        fdev = [None] * len(rows)
        if o32 is not None:
            f = o32.step(tokens[rows], pos[rows])
            for i in range(len(rows)):
                bound = REL_TOL * np.abs(ref[i]).max() + ABS_TOL
                fdev[i] = float(np.abs(f[i] - ref[i]).max())
                res.floor = max(res.floor, fdev[i] / bound)
        ref_tok, margin = oracle.greedy(ref)
        gpu_tok = np.argmax(got, axis=1).astype(np.int32)
        for i, b in enumerate(rows):
            agree = bool(gpu_tok[b] == ref_tok[i])
            res.records.append((s, b, float(margin[i]), agree, fdev[i]))
            if margin[i] > MARGIN:
                res.checked_argmax += 1
                res.argmax_agree += int(agree)
        nxt = gpu_tok.copy()
        for i, b in enumerate(rows):
            nxt[b] = ref_tok[i]
        tokens = nxt
        pos = pos + 1
        res.steps += 1
    if check_cache:
        # the slots this run wrote hold bf16(rope(k)) and bf16(v) of values that
        # carry the same error bound as the logits; rounding them to bf16 adds
        # at most one bf16 ulp (2^-7 of the magnitude) on top.  The seeded
        # prefix must be untouched, bit for bit.
        # With floor=True (deep stacks) a slot may also differ by up to twice
        # what the fp32-accumulation build's cache differs from the oracle's.
        gk, gv = kv_from_device(kv_dev)
        for i, b in enumerate(rows):
            for (ga, oa, fa) in ((gk, orc.kc, o32.kc if o32 else None), (gv, orc.vc, o32.vc if o32 else None)):
                for p in range(int(pos0[b]), int(pos[b])):
                    x = synth.bf16_bits_to_f32(ga[:, b, :, p]).astype(np.float64)
                    y = synth.bf16_bits_to_f32(oa[:, i, :, p]).astype(np.float64)
                    bound = (REL_TOL + 2.0 ** -7) * np.abs(y).max() + ABS_TOL
                    if fa is not None:
                        f = synth.bf16_bits_to_f32(fa[:, i, :, p]).astype(np.float64)
                        bound = max(bound, 2.0 * np.abs(f - y).max())
                    assert np.abs(x - y).max() <= bound, \
                        "KV slot %d of sequence %d: max diff %.3g > %.3g" % (p, b, np.abs(x - y).max(), bound)
                x0 = ga[:, b, :, : int(pos0[b])]
                y0 = oa[:, i, :, : int(pos0[b])]
                assert np.array_equal(x0, y0), "cached prefix of sequence %d changed" % b
    eng.close()
    return res


def assert_ok(res: Result):
    """The flat acceptance: max|d logit| <= 1e-2 max|logit| + 1e-3 at every step
    and row, and the GPU's argmax equals the oracle's wherever the oracle's
    top-2 margin exceeds 1e-2."""
    log_parity("end_to_end_strict", res.summary())
    assert res.worst <= 1.0, res
    assert res.argmax_agree == res.checked_argmax, res


def assert_end_to_end(res: Result):
    """Deep random-init stacks amplify single bf16 rounding flips (a plain fp32
    implementation of the definition already exceeds the logit bound): the
    GPU must meet the bound, or stay within twice the fp32-accumulation
    build's deviation on the same run.  Its greedy token must equal the
    oracle's wherever the oracle's top-2 margin exceeds both 1e-2 and twice
    what fp32 rounding alone moved the logits at that step.  The record
    logged beside it also says whether the flat bound and the flat 1e-2
    margin rule held as written."""
    log_parity("end_to_end_relaxed", res.summary())
    assert res.worst <= max(1.0, 2.0 * res.floor), res
    bad = res.relaxed_misses()
    assert not bad, (res, bad[:5])


class LayerResult:
    def __init__(self):
        self.worst = {"x_mid": 0.0, "x_out": 0.0, "logits": 0.0, "kv_slot": 0.0}
        self.where = {}
        self.layers_checked = 0
        self.steps = 0

    def note(self, key, got, ref, where, extra_rel=0.0):
        bound = (REL_TOL + extra_rel) * np.abs(ref).max() + ABS_TOL
        r = float(np.abs(np.asarray(got, dtype=np.float64) - ref).max() / bound)
        if r > self.worst[key]:
            self.worst[key] = r
            self.where[key] = where

    def __repr__(self):
        return "LayerResult(%s, at %s, layers=%d, steps=%d)" % (
            {k: round(v, 3) for k, v in self.worst.items()}, self.where, self.layers_checked, self.steps)


def layerwise(wl, steps=2, options=None, batch=None, positions0=None, check_rows=None, model=None, kv=None):
    """Per-layer parity from a shared state.  After each GPU step the oracle
    re-runs every layer l from the GPU's own input residual of that layer and
    the GPU's KV cache as it was before the step, and the final norm + LM head
    from the GPU's final residual; every layer output (residual after
    attention, residual after the MLP), the K/V slot written and the logits
    are held to max|d| <= 1e-2 max|ref| + 1e-3 (the K/V slot gets one more bf16
    ulp, 2^-7 of its magnitude, for its own rounding)."""
    import torch
    B = batch or wl.batch
    rows = list(range(B)) if check_rows is None else list(check_rows)
    model = model or synth.make_model(wl, seed=1)
    kc, vc = kv if kv is not None else synth.make_kv(wl, seed=2, batch=B)
    opts = dict(options or {})
    opts["scratch_depth"] = wl.n_layers + 1
    dev = model_to_device(model)
    eng = make_engine(wl, dev, opts, max_batch=B)
    kv_dev = kv_to_device(kc, vc)
    del kc, vc
    tokens = synth.initial_tokens(wl, B).copy()
    pos = np.full(B, wl.ctx, dtype=np.int32) if positions0 is None else np.array(positions0, dtype=np.int32)
    logits = torch.empty((B, wl.vocab), dtype=torch.float32, device="cuda")
    embed = synth.bf16_bits_to_f32(model.embed)
    res = LayerResult()
    L = wl.n_layers
    for s in range(steps):
        k_before, v_before = kv_rows_from_device(kv_dev, rows)
        eng.step(torch.from_numpy(tokens).cuda(), torch.from_numpy(pos).cuda(), kv_dev, logits)
        st = eng.sync()
        assert st == 0, "device error %d: %s" % (st, eng.last_error())
        xi, xm = eng.read_residuals()
        got_logits = logits.cpu().numpy()
        k_after, v_after = kv_rows_from_device(kv_dev, rows)
        for i, b in enumerate(rows):
            orc = oracle.Oracle(model, np.ascontiguousarray(k_before[:, i:i + 1]),
                                np.ascontiguousarray(v_before[:, i:i + 1]))
            p = int(pos[b])
            for l in range(L):
                x = embed[tokens[b]].astype(np.float64) if l == 0 else xi[l, b].astype(np.float64)
                ref_mid, ref_out = orc.layer(l, 0, p, x)
                res.note("x_mid", xm[l, b], ref_mid, (s, b, l))
                res.note("x_out", xi[l + 1, b], ref_out, (s, b, l))
                for ga, oa in ((k_after, orc.kc), (v_after, orc.vc)):
                    res.note("kv_slot", synth.bf16_bits_to_f32(ga[l, i, :, p]),
                             synth.bf16_bits_to_f32(oa[l, 0, :, p]).astype(np.float64), (s, b, l), 2.0 ** -7)
                res.layers_checked += 1
            res.note("logits", got_logits[b], orc.lm_head(xi[L, b].astype(np.float64)), (s, b))
        tokens = np.argmax(got_logits, axis=1).astype(np.int32)
        pos = pos + 1
        res.steps += 1
    eng.close()
    return res


def assert_layers_ok(res: LayerResult):
    log_parity("per_layer", {"steps": int(res.steps), "layers_checked": int(res.layers_checked),
                             "worst": {k: float(v) for k, v in res.worst.items()},
                             "where": {k: [int(x) for x in v] for k, v in res.where.items()}})
    assert all(v <= 1.0 for v in res.worst.values()), res
