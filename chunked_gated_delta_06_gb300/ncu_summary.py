"""Summarise an ncu launch list (--metrics gpu__time_duration.sum --csv) per kernel.

    python -m chunked_gated_delta_06_gb300.ncu_summary launches.csv [--skip-first N]

Prints, per kernel name, the number of launches, the total and mean device time
and the share of the total, largest first.
"""
import csv
import re
import sys
from collections import defaultdict


def summarise(path, skip_first=0):
    rows = []
    with open(path) as f:
        lines = [ln for ln in f if ln.startswith('"')]
    for r in csv.DictReader(lines):
        if r.get("Metric Name") != "gpu__time_duration.sum":
            continue
        rows.append(r)
    rows = rows[skip_first:]
    agg = defaultdict(lambda: [0, 0.0])
    for r in rows:
        name = r["Kernel Name"].replace("(anonymous namespace)", "anon")
        name = re.sub(r"\(.*", "", name).split("::")[-1].strip()
        scale = {"ns": 1e-6, "us": 1e-3, "usecond": 1e-3, "nsecond": 1e-6, "ms": 1.0,
                 "msecond": 1.0}.get(r["Metric Unit"], 1e-6)
        agg[name][0] += 1
        agg[name][1] += float(r["Metric Value"].replace(",", "")) * scale
    total = sum(v[1] for v in agg.values())
    out = ["%-28s %8s %12s %10s %7s" % ("kernel", "launches", "total ms", "mean ms", "share")]
    for name, (n, ms) in sorted(agg.items(), key=lambda kv: -kv[1][1]):
        out.append("%-28s %8d %12.3f %10.4f %6.1f%%" % (name, n, ms, ms / n, 100 * ms / total))
    out.append("%-28s %8d %12.3f" % ("total", sum(v[0] for v in agg.values()), total))
    return "\n".join(out)


if __name__ == "__main__":
    skip = 0
    if "--skip-first" in sys.argv:
        skip = int(sys.argv[sys.argv.index("--skip-first") + 1])
    print(summarise(sys.argv[1], skip))
