"""Summarise Nsight Compute output for the step's kernels.

  python -m step_gpt_train_gb300.ncu_summary launches <launches.csv>
      per kernel: launches, total device time, share of the captured time
      (input: `ncu --metrics gpu__time_duration.sum --csv --log-file ...`)
  python -m step_gpt_train_gb300.ncu_summary raw <report.ncu-rep> [kernel-regex]
      the headline counters of each captured launch (needs the ncu CLI)
"""
from __future__ import annotations

import collections
import csv
import io
import re
import subprocess
import sys

RAW_METRICS = [
    ("gpu__time_duration.sum", "duration"),
    ("dram__bytes_read.sum", "DRAM read"),
    ("dram__bytes_write.sum", "DRAM write"),
    ("gpu__dram_throughput.avg.pct_of_peak_sustained_elapsed", "DRAM throughput % of peak"),
    ("sm__pipe_tensor_cycles_active.avg.pct_of_peak_sustained_elapsed", "tensor pipe active %"),
    ("lts__throughput.avg.pct_of_peak_sustained_elapsed", "L2 throughput %"),
    ("lts__t_sector_hit_rate.pct", "L2 hit rate %"),
    ("sm__throughput.avg.pct_of_peak_sustained_elapsed", "SM throughput %"),
    ("sm__warps_active.avg.pct_of_peak_sustained_active", "warps active %"),
    ("launch__registers_per_thread", "registers/thread"),
    ("smsp__average_warps_issue_stalled_long_scoreboard_per_issue_active.ratio", "stall long scoreboard"),
    ("smsp__average_warps_issue_stalled_wait_per_issue_active.ratio", "stall wait"),
    ("smsp__average_warps_issue_stalled_barrier_per_issue_active.ratio", "stall barrier"),
    ("smsp__average_warps_issue_stalled_short_scoreboard_per_issue_active.ratio", "stall short scoreboard"),
    ("smsp__average_warps_issue_stalled_math_pipe_throttle_per_issue_active.ratio", "stall math pipe"),
    ("smsp__average_warps_issue_stalled_mio_throttle_per_issue_active.ratio", "stall MIO throttle"),
]


def short_name(name: str) -> str:
    name = re.sub(r"\(.*$", "", name)  # drop the argument list
    name = name.replace("void ", "").replace("<unnamed>::", "")
    return name.strip()


def launches(path: str) -> str:
    text = "".join(l for l in open(path) if not l.startswith("=="))
    rows = [r for r in csv.DictReader(io.StringIO(text)) if r.get("Metric Name") == "gpu__time_duration.sum"]
    per = collections.OrderedDict()
    for r in rows:
        k = short_name(r["Kernel Name"])
        unit = r["Metric Unit"]
        v = float(r["Metric Value"].replace(",", ""))
        ns = v * {"ns": 1, "us": 1e3, "usecond": 1e3, "ms": 1e6, "msecond": 1e6, "nsecond": 1}.get(unit, 1)
        c, t = per.get(k, (0, 0.0))
        per[k] = (c + 1, t + ns)
    total = sum(t for _, t in per.values())
    out = [f"captured launches: {len(rows)}; total device time {total / 1e6:.3f} ms (serialised, cold cache)",
           "", f"{'kernel':70s} {'launches':>8s} {'total ms':>10s} {'share':>7s}"]
    for k, (c, t) in sorted(per.items(), key=lambda kv: -kv[1][1]):
        out.append(f"{k[:70]:70s} {c:8d} {t / 1e6:10.3f} {100 * t / total:6.2f}%")
    return "\n".join(out)


def raw(path: str, pattern: str = ".*") -> str:
    csv_text = subprocess.run(["ncu", "-i", path, "--page", "raw", "--csv"], capture_output=True,
                              text=True).stdout
    rows = list(csv.reader(io.StringIO(csv_text)))
    hdr, units, data = rows[0], rows[1], rows[2:]
    idx = {h: i for i, h in enumerate(hdr)}
    out = []
    for n, d in enumerate(data):
        name = d[idx["Kernel Name"]]
        if not re.search(pattern, name):
            continue
        out.append(f"launch {n}: {short_name(name)}  grid {d[idx['Grid Size']]} block {d[idx['Block Size']]}")
        for m, label in RAW_METRICS:
            if m in idx:
                out.append(f"  {label:32s} {d[idx[m]]} {units[idx[m]]}")
    return "\n".join(out)


if __name__ == "__main__":
    if sys.argv[1] == "launches":
        print(launches(sys.argv[2]))
    else:
        print(raw(sys.argv[2], sys.argv[3] if len(sys.argv) > 3 else ".*"))
