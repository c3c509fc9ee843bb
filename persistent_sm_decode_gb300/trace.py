"""One traced decode step of a synthetic workload, for tuning:

    python -m persistent_sm_decode_gb300.trace WORKLOAD [--batch B] [--layer L] [--out DIR]

Builds the tuning library (the kernel with its per-task timing code, as
AMK_TRACE=1 does; the next plain build() puts the default library back),
runs a few decode steps of WORKLOAD (a name from synth.workload) with
weights and KV filled on the device, and reads the last step's task
timestamps.  Prints the step's span, the per-level critical-path times of
layer L and, per operator of that layer, when its tasks got their inputs
(prologue_lag); writes the per-level times and a Chrome trace (one track
per CTA) to DIR.  Needs a GPU; the timing code itself adds about a tenth to
the step.
"""
import argparse
import json
import os
import sys


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("workload")
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--layer", type=int, default=10)
    ap.add_argument("--steps", type=int, default=6)
    ap.add_argument("--out", default=".")
    a = ap.parse_args(argv)
    os.environ["AMK_TRACE"] = "1"
    import torch
    import bench
    import synth
    import persistent_sm_decode_gb300 as amk
    amk.build()
    wl = synth.workload(a.workload, **({"batch": a.batch} if a.batch else {}))
    layer = min(max(1, a.layer), wl.n_layers - 1)
    dev = bench.device_model(wl, seed=1)
    kv = bench.device_kv(wl, seed=2, batch=wl.batch)
    opts = {"trace": 1}
    eng = bench.make_engine(amk, wl, dev, opts)
    logits = torch.empty((wl.batch, wl.vocab), dtype=torch.float32, device="cuda")
    tok = torch.ones(wl.batch, dtype=torch.int32, device="cuda")
    for s in range(a.steps):
        pos = torch.full((wl.batch,), wl.ctx + s, dtype=torch.int32, device="cuda")
        eng.step(tok, pos, kv, logits)
        if eng.sync() != amk.OK:
            sys.exit("decode step failed: %s" % eng.last_error())
    tr = eng.read_trace()
    info = eng.plan_info()
    plan = amk.Plan(eng.cfg, wl.batch, info["n_sm"], options=opts)
    assert plan.info()["n_tasks"] == info["n_tasks"], "the host plan differs from the handle's"
    eng.close()
    tag = a.workload + ("_b%d" % wl.batch if a.batch else "")
    os.makedirs(a.out, exist_ok=True)
    lv = amk.level_times(tr, plan)
    json.dump(lv, open(os.path.join(a.out, "levels_%s.json" % tag), "w"), indent=0)
    json.dump(amk.chrome_trace(tr, plan), open(os.path.join(a.out, "trace_%s.json" % tag), "w"))
    started = [int(r[0]) for r in tr if int(r[0]) > 0]
    print("%s, batch %d: step span (first task start to last task end) %.1f us" %
          (a.workload, wl.batch, (int(tr[:, 3].max()) - min(started)) / 1e3))
    print("layer %d, per level: %s" % (layer, ", ".join("%s %.2f us" % (x["op"], x["level_us"])
                                                      for x in lv if x["layer"] == layer)))
    print("| op | after | tasks | inputs ready: min / median / max us after the last producer | "
          "prologue | tiles | epilogue (median us) |")
    print("|---|---|---|---|---|---|---|")
    for x in amk.prologue_lag(tr, plan, layer):
        print("| %s | %s | %d | %.2f / %.2f / %.2f | %.2f | %.2f | %.2f |" % (
            x["op"], x["after"], x["tasks"], x["lag_min_us"], x["lag_median_us"], x["lag_max_us"],
            x["prologue_us"], x["tiles_us"], x["epilogue_us"]))
    return 0


if __name__ == "__main__":
    sys.exit(main())
