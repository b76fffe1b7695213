"""Summarise the attention error statistics that the GPU parity tests append
to the file named by PA_PARITY_LOG (one JSON line per check_attention /
check_lse call) into a markdown table, one row per test and dtype, worst
case over its checks:

    PA_PARITY_LOG=/tmp/parity.jsonl python -m pytest tests -m gpu -q
    python tests/parity_report.py /tmp/parity.jsonl
"""
from __future__ import annotations

import json
import sys
from collections import defaultdict


def summarise(lines):
    rows = defaultdict(lambda: {"checks": 0, "n": 0, "max_abs": 0.0, "max_rel": 0.0,
                                "excess": float("-inf")})
    lse = defaultdict(float)
    for rec in lines:
        test = rec.get("test", "").replace("tests/", "")
        if rec["what"].endswith("[lse]"):
            lse[test] = max(lse[test], rec["max_abs"])
            continue
        r = rows[(test, rec["dtype"])]
        r["checks"] += 1
        r["n"] += rec["n"]
        r["max_abs"] = max(r["max_abs"], rec["max_abs"])
        r["max_rel"] = max(r["max_rel"], rec["max_rel_ge_1e-2"])
        r["excess"] = max(r["excess"], rec["max_abs_beyond_rounding"])
    return rows, lse


def main(path):
    with open(path) as f:
        lines = [json.loads(x) for x in f if x.strip()]
    rows, lse = summarise(lines)
    print("| test | out dtype | checks | elements | max abs | max rel (\\|ref\\| >= 1e-2) "
          "| max abs beyond output rounding |")
    print("|---|---|---|---|---|---|---|")
    for (test, dt), r in sorted(rows.items()):
        print(f"| `{test}` | {dt} | {r['checks']} | {r['n']} | {r['max_abs']:.2e} | "
              f"{r['max_rel']:.2e} | {r['excess']:.2e} |")
    if lse:
        worst_t = max(lse, key=lse.get)
        print()
        print(f"Log-sum-exp outputs: {len(lse)} tests, max abs error {lse[worst_t]:.2e} "
              f"(`{worst_t}`).")
    worst = {}
    for (test, dt), r in rows.items():
        w = worst.setdefault(dt, [0.0, 0.0, float("-inf")])
        w[0] = max(w[0], r["max_abs"])
        w[1] = max(w[1], r["max_rel"])
        w[2] = max(w[2], r["excess"])
    print()
    for dt, (a, rel, exc) in sorted(worst.items()):
        print(f"- {dt}: max abs {a:.2e}, max rel {rel:.2e}, max beyond rounding {exc:.2e}")


if __name__ == "__main__":
    main(sys.argv[1])
