"""Writes the oracle regression fixtures in this folder.

The pages this project follows print no numeric values for the decode step
(no logits, tokens or intermediate tensors), so nothing here is quoted from
them.  These fixtures record what the pinned oracle computes on the tiny
workload, so that a later change to the oracle, or a platform difference in
the seeded generator, shows up as a diff.  Only ``synth`` and ``oracle`` are
called.

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import synth  # noqa: E402


def tiny_greedy(steps=8):
    wl = synth.workload("tiny")
    model = synth.make_model(wl, seed=1)
    kc, vc = synth.make_kv(wl, seed=2)
    orc = oracle.Oracle(model, kc, vc)
    tok = synth.initial_tokens(wl)
    rows = []
    for s in range(steps):
        lg = orc.step(tok, [wl.ctx + s])[0]
        nxt, margin = oracle.greedy(lg[None, :])
        rows.append({"step": s, "position": wl.ctx + s, "token_in": int(tok[0]), "argmax": int(nxt[0]),
                     "margin": float(margin[0]), "logits_head": [float(v) for v in lg[:8]],
                     "logits_sum": float(lg.sum()), "logits_absmax": float(np.abs(lg).max())})
        tok = nxt
    return rows


if __name__ == "__main__":
    with open(os.path.join(HERE, "tiny_oracle_greedy.json"), "w") as f:
        json.dump({"workload": "tiny", "weights_seed": 1, "kv_seed": 2, "steps": tiny_greedy()}, f, indent=1)
    print("wrote tiny_oracle_greedy.json")
