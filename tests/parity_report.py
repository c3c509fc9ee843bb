"""Turns the JSON lines that the GPU parity tests append to $AMK_PARITY_LOG
into a Markdown table: per test, the worst logit deviation against the flat
bound (max|d| / (1e-2 max|logit| + 1e-3)), how far the fp32-accumulation
build of the definition lands (the floor), the argmax checks at the flat
1e-2 margin, the misses under the deep-stack rule and the free-running
agreement length.

    python tests/parity_report.py parity.jsonl > table.md
"""
import json
import sys


def main(path):
    recs = [json.loads(ln) for ln in open(path) if ln.strip()]
    print("| test | steps | rows | worst / flat bound | floor | flat bound met | argmax agree at 1e-2 margin "
          "| misses, deep-stack rule | free-running steps |")
    print("|---|---|---|---|---|---|---|---|---|")
    for r in recs:
        if r["kind"] == "per_layer":
            continue
        name = r["test"].split("::")[-1]
        print("| %s | %d | %s | %.3f | %.3f | %s | %d / %d | %d | %d |" % (
            name, r["steps"], ",".join(str(x) for x in r["rows"]), r["worst"], r["floor"],
            "yes" if r["strict_logits_ok"] else "no", r["argmax_agree"], r["argmax_checked"],
            r["relaxed_misses"], r["free_running"]))
    print()
    print("| per-layer test | steps | layer checks | worst x_mid | worst x_out | worst K/V slot | worst logits |")
    print("|---|---|---|---|---|---|---|")
    for r in recs:
        if r["kind"] != "per_layer":
            continue
        w = r["worst"]
        print("| %s | %d | %d | %.3f | %.3f | %.3f | %.3f |" % (
            r["test"].split("::")[-1], r["steps"], r["layers_checked"], w["x_mid"], w["x_out"], w["kv_slot"],
            w["logits"]))


if __name__ == "__main__":
    main(sys.argv[1])
