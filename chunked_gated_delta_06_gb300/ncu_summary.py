"""Summaries of ncu output.

    python -m chunked_gated_delta_06_gb300.ncu_summary launches.csv [--skip-first N]
        per kernel of a launch list (--metrics gpu__time_duration.sum --csv):
        launches, total and mean device time, share of the total;
    python -m chunked_gated_delta_06_gb300.ncu_summary --traffic prof.ncu-rep UNITS [prof2 UNITS2 ...]
        JSON record of DRAM bytes per work unit (UNITS = chunk x value-head units,
        or active decode rows x value heads, of the captured launches) with the
        hash of each kernel's source file at capture time (bench.py reports the
        traffic only while the source is unchanged);
    python -m chunked_gated_delta_06_gb300.ncu_summary --report prof.ncu-rep
        per captured launch of a --set full report: duration, DRAM bytes read and
        written, DRAM throughput, tensor-pipe activity, achieved occupancy,
        registers, and the largest warp-stall reasons (cycles per issued
        instruction).
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


def report(path):
    import subprocess
    out = subprocess.run(["ncu", "-i", path, "--page", "raw", "--csv"], capture_output=True,
                         text=True, check=True).stdout
    rows = list(csv.reader(out.splitlines()))
    hdr, units, data = rows[0], rows[1], rows[2:]

    def get(r, m):
        return r[hdr.index(m)] if m in hdr else ""

    def unit(r, m):
        return units[hdr.index(m)] if m in hdr else ""

    stall = [c for c in hdr if c.startswith("smsp__average_warps_issue_stalled_")
             and c.endswith("_per_issue_active.ratio")]
    lines = []
    for r in data:
        name = re.sub(r"\(.*", "", r[hdr.index("Kernel Name")].replace("(anonymous namespace)", "anon"))
        name = name.split("::")[-1].strip()
        tops = sorted(((float(get(r, c) or 0), c[len("smsp__average_warps_issue_stalled_"):-len(
            "_per_issue_active.ratio")]) for c in stall), reverse=True)[:4]
        lines.append(
            "%s: %s %s; DRAM read %s %s, write %s %s (%s %% of peak); tensor pipe %s %% of active; "
            "warps active %s %%; %s regs/thread; grid %s block %s; stalls (cycles/issue): %s" % (
                name, get(r, "gpu__time_duration.sum"), unit(r, "gpu__time_duration.sum"),
                get(r, "dram__bytes_read.sum"), unit(r, "dram__bytes_read.sum"),
                get(r, "dram__bytes_write.sum"), unit(r, "dram__bytes_write.sum"),
                get(r, "gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed"),
                get(r, "sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_active"),
                get(r, "sm__warps_active.avg.pct_of_peak_sustained_active"),
                get(r, "launch__registers_per_thread"), get(r, "launch__grid_size"),
                get(r, "launch__block_size"),
                ", ".join("%s %.2f" % (n, v) for v, n in tops)))
    return "\n".join(lines)


KERNELS = {  # ncu kernel name -> (bench kernel name, source file)
    "k_intra_tc": ("intra", "gdn_intra_tc.cu"), "k_state_tc": ("state", "gdn_state_tc.cu"),
    "k_out_tc<1>": ("out", "gdn_out_tc.cu"), "k_out_tc<0>": ("dvloc", "gdn_out_tc.cu"),
    "k_out_tc<true>": ("out", "gdn_out_tc.cu"), "k_out_tc<false>": ("dvloc", "gdn_out_tc.cu"),
    "k_bstate_tc": ("bstate", "gdn_bstate_tc.cu"), "k_bintra_a_tc": ("bintra_a", "gdn_bintra_tc.cu"),
    "k_state_tc<0>": ("state", "gdn_state_tc.cu"), "k_bstate_tc<0>": ("bstate", "gdn_bstate_tc.cu"),
    "k_bintra_b_tc": ("bintra_b", "gdn_bintra_b_tc.cu"), "k_decode": ("decode", "gdn_decode.cu"),
    "k_bnorm": ("bnorm", "gdn_chunk.cu"), "k_prep": ("prep", "gdn_chunk.cu"),
    "k_bnorm<1>": ("bnorm", "gdn_chunk.cu"), "k_bnorm<2>": ("bnorm", "gdn_chunk.cu"),
    "k_bnorm<4>": ("bnorm", "gdn_chunk.cu"), "k_bnorm<0>": ("bnorm", "gdn_chunk.cu"),
}


def traffic(path, units):
    import hashlib
    import json
    import os
    import subprocess
    out = subprocess.run(["ncu", "-i", path, "--page", "raw", "--csv"], capture_output=True,
                         text=True, check=True).stdout
    rows = list(csv.reader(out.splitlines()))
    hdr, data = rows[0], rows[2:]
    units_row = rows[1]
    scale = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "csrc")
    rec = {}
    for r in data:
        name = re.sub(r"\(.*", "", r[hdr.index("Kernel Name")].replace("(anonymous namespace)", "anon"))
        name = name.split("::")[-1].strip()
        if name not in KERNELS:
            continue
        kname, src = KERNELS[name]
        rd = float(r[hdr.index("dram__bytes_read.sum")]) * scale[units_row[hdr.index("dram__bytes_read.sum")]]
        wr = float(r[hdr.index("dram__bytes_write.sum")]) * scale[units_row[hdr.index("dram__bytes_write.sum")]]
        with open(os.path.join(csrc, src), "rb") as fh:
            sha = hashlib.sha256(fh.read()).hexdigest()[:16]
        rec[kname] = {"bytes_per_unit": (rd + wr) / units, "captured_units": units,
                      "capture": os.path.basename(path), "source_sha256_16": sha}
    return json.dumps(rec, indent=1, sort_keys=True)


if __name__ == "__main__":
    if "--traffic" in sys.argv:
        # --traffic REPORT UNITS [REPORT UNITS ...]: one merged record
        import json
        i = sys.argv.index("--traffic")
        args, rec = sys.argv[i + 1:], {}
        for r, u in zip(args[0::2], args[1::2]):
            rec.update(json.loads(traffic(r, float(u))))
        print(json.dumps(rec, indent=1, sort_keys=True))
        sys.exit(0)
    if "--report" in sys.argv:
        print(report(sys.argv[sys.argv.index("--report") + 1]))
        sys.exit(0)
    skip = 0
    if "--skip-first" in sys.argv:
        skip = int(sys.argv[sys.argv.index("--skip-first") + 1])
    print(summarise(sys.argv[1], skip))
