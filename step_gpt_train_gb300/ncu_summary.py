"""Summarise Nsight Compute output for the step's kernels.

  python -m step_gpt_train_gb300.ncu_summary launches <launches.csv> [marker-regex n]
      per kernel: launches, total device time, share of the captured time,
      and DRAM bytes per launch when the capture has them
      (input: `ncu --metrics gpu__time_duration.sum[,dram__bytes_read.sum,
      dram__bytes_write.sum] --csv --log-file ...`); with a marker, only the
      launches from the n-th launch (1-based) of a kernel matching the marker
      up to the next one: one training step when the marker is its first kernel
  python -m step_gpt_train_gb300.ncu_summary raw <report.ncu-rep> [kernel-regex]
      the headline counters of each captured launch (needs the ncu CLI)
  python -m step_gpt_train_gb300.ncu_summary step_traffic <launches.csv>
      DRAM bytes of the matmul family over one training step, from a capture
      (gpu__time_duration.sum, dram__bytes_read.sum, dram__bytes_write.sum)
      of `opbench --ops step_gemms --warmup 0 --iters 1`: every gemm_tc_kernel
      or gemm_pair_kernel launch starts the next of the step's matmuls (in
      opbench.STEP_GEMMS order), a split_reduce_kernel after it belongs to it,
      and each matmul's bytes count as often as the step runs it
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


def _ns(value: str, unit: str) -> float:
    v = float(value.replace(",", ""))
    return v * {"ns": 1, "us": 1e3, "usecond": 1e3, "ms": 1e6, "msecond": 1e6, "nsecond": 1}.get(unit, 1)


def _bytes(value: str, unit: str) -> float:
    v = float(value.replace(",", ""))
    return v * {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "KB": 1e3, "MB": 1e6, "GB": 1e9}.get(unit, 1)


def launches(path: str, marker: str | None = None, nth: int = 1) -> str:
    text = "".join(l for l in open(path) if not l.startswith("=="))
    per_launch = collections.OrderedDict()  # launch id -> {name, ns, read, write}
    for r in csv.DictReader(io.StringIO(text)):
        lid = r.get("ID")
        d = per_launch.setdefault(lid, {"name": short_name(r["Kernel Name"])})
        m, unit, val = r.get("Metric Name"), r.get("Metric Unit"), r.get("Metric Value")
        if m == "gpu__time_duration.sum":
            d["ns"] = _ns(val, unit)
        elif m == "dram__bytes_read.sum":
            d["read"] = _bytes(val, unit)
        elif m == "dram__bytes_write.sum":
            d["write"] = _bytes(val, unit)
    rows = [d for d in per_launch.values() if "ns" in d]
    window = ""
    if marker:
        starts = [i for i, d in enumerate(rows) if re.search(marker, d["name"])]
        if len(starts) < nth:
            raise SystemExit(f"marker {marker!r} occurs {len(starts)} times, fewer than {nth}")
        lo = starts[nth - 1]
        hi = starts[nth] if len(starts) > nth else len(rows)
        rows = rows[lo:hi]
        window = f"; window: launch {nth} of {marker!r} to the next ({len(rows)} launches)"
    has_dram = all("read" in d and "write" in d for d in rows) and rows
    per = collections.OrderedDict()
    for d in rows:
        c, t, by = per.get(d["name"], (0, 0.0, 0.0))
        per[d["name"]] = (c + 1, t + d["ns"], by + (d["read"] + d["write"] if has_dram else 0.0))
    total = sum(t for _, t, _ in per.values())
    out = [f"captured launches: {len(rows)}; total device time {total / 1e6:.3f} ms (serialised, cold cache){window}",
           "", f"{'kernel':64s} {'launches':>8s} {'total ms':>10s} {'share':>7s}" +
           (f" {'DRAM MB/launch':>15s}" if has_dram else "")]
    for k, (c, t, by) in sorted(per.items(), key=lambda kv: -kv[1][1]):
        line = f"{k[:64]:64s} {c:8d} {t / 1e6:10.3f} {100 * t / total:6.2f}%"
        if has_dram:
            line += f" {by / c / 1e6:15.1f}"
        out.append(line)
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


def step_traffic(path: str) -> str:
    from step_gpt_train_gb300.opbench import STEP_GEMMS
    text = "".join(l for l in open(path) if not l.startswith("=="))
    per_launch = collections.OrderedDict()
    for r in csv.DictReader(io.StringIO(text)):
        d = per_launch.setdefault(r.get("ID"), {"name": short_name(r["Kernel Name"])})
        m, unit, val = r.get("Metric Name"), r.get("Metric Unit"), r.get("Metric Value")
        if m == "dram__bytes_read.sum":
            d["read"] = _bytes(val, unit)
        elif m == "dram__bytes_write.sum":
            d["write"] = _bytes(val, unit)
    ops, cur = [], None
    for d in per_launch.values():
        if d["name"].startswith(("gemm_tc_kernel", "gemm_pair_kernel")):
            cur = {"launches": 0, "bytes": 0.0}
            ops.append(cur)
        elif not d["name"].startswith("split_reduce_kernel") or cur is None:
            continue
        cur["launches"] += 1
        cur["bytes"] += d["read"] + d["write"]
    names = list(STEP_GEMMS)
    if len(ops) != len(names):
        raise SystemExit(f"{len(ops)} matmuls captured, {len(names)} expected")
    total_b = sum(STEP_GEMMS[n] * o["bytes"] for n, o in zip(names, ops))
    total_l = sum(STEP_GEMMS[n] * o["launches"] for n, o in zip(names, ops))
    out = [f"{'matmul':24s} {'per step':>8s} {'launches':>8s} {'DRAM MB':>10s}"]
    for n, o in zip(names, ops):
        out.append(f"{n:24s} {STEP_GEMMS[n]:8d} {o['launches']:8d} {o['bytes'] / 1e6:10.1f}")
    out += ["", f"launches_per_step: {total_l}", f"traffic_bytes_per_step: {total_b:.0f}",
            f"traffic_bytes_per_launch_full_step_avg: {total_b / total_l:.1f}"]
    return "\n".join(out)


if __name__ == "__main__":
    if sys.argv[1] == "step_traffic":
        print(step_traffic(sys.argv[2]))
    elif sys.argv[1] == "launches":
        print(launches(sys.argv[2], sys.argv[3] if len(sys.argv) > 3 else None,
                       int(sys.argv[4]) if len(sys.argv) > 4 else 1))
    else:
        print(raw(sys.argv[2], sys.argv[3] if len(sys.argv) > 3 else ".*"))
