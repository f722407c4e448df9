"""Host logic of the ncu summaries that the committed profiles are made with:
per-kernel aggregation of a launch list, the one-step window, and the matmul
family's traffic over a step (each capture launch attributed to the step's
matmuls in order, the split-K reduce to the matmul before it). Synthetic CSV in
ncu's --csv layout; no GPU."""
import csv
import io

import pytest

from step_gpt_train_gb300 import ncu_summary as NS
from step_gpt_train_gb300.opbench import STEP_GEMMS

HEADER = ["ID", "Process ID", "Process Name", "Host Name", "Kernel Name", "Context", "Stream", "Block Size",
          "Grid Size", "Device", "CC", "Section Name", "Metric Name", "Metric Unit", "Metric Value"]


def _write(tmp_path, launches):
    """launches: [(kernel name, {metric: (unit, value)})] -> an ncu --csv log file."""
    buf = io.StringIO()
    buf.write("==PROF== Connected to process 1\n")
    w = csv.writer(buf, quoting=csv.QUOTE_ALL)
    w.writerow(HEADER)
    for i, (name, metrics) in enumerate(launches):
        for m, (unit, val) in metrics.items():
            w.writerow([str(i), "1", "python3", "127.0.0.1", f"void <unnamed>::{name}(CUtensorMap_st, int)", "1", "7",
                        "(320, 1, 1)", "(152, 1, 1)", "0", "10.3", "Command line profiler metrics", m, unit, val])
    p = tmp_path / "launches.csv"
    p.write_text(buf.getvalue())
    return str(p)


def test_short_name_drops_arguments_and_namespace():
    assert NS.short_name("void <unnamed>::gemm_pair_kernel<0, 0, 0, 192>(CUtensorMap_st, int)") == \
        "gemm_pair_kernel<0, 0, 0, 192>"


def test_launches_aggregates_and_windows(tmp_path):
    t = lambda us: {"gpu__time_duration.sum": ("usecond", str(us))}
    seq = [("encoder_fwd_kernel", t(10)), ("gemm_tc_kernel<256, 0, 0, 0, 0>", t(100)),
           ("gemm_pair_kernel<0, 0, 0, 256>", t(50)), ("gemm_tc_kernel<256, 0, 0, 0, 0>", t(100)),
           ("encoder_fwd_kernel", t(12)), ("gemm_pair_kernel<0, 0, 0, 256>", t(30)),
           ("encoder_fwd_kernel", t(11))]
    out = NS.launches(_write(tmp_path, seq))
    assert "captured launches: 7; total device time 0.313 ms" in out
    rows = {l.split()[0]: l for l in out.splitlines()[3:]}
    assert rows["gemm_tc_kernel<256,"].split()[-3:] == ["2", "0.200", "63.90%"]
    # the second step only: from the second encoder launch to the third
    out2 = NS.launches(_write(tmp_path, seq), "encoder_fwd", 2)
    assert "captured launches: 2; total device time 0.042 ms" in out2
    assert "window: launch 2 of 'encoder_fwd' to the next (2 launches)" in out2
    with pytest.raises(SystemExit):
        NS.launches(_write(tmp_path, seq), "encoder_fwd", 4)


def test_step_traffic_attributes_launches_in_step_order(tmp_path):
    names = list(STEP_GEMMS)
    seq, expect = [], 0.0
    for i, n in enumerate(names):
        kernel = "gemm_pair_kernel<0, 0, 0, 256>" if i % 3 == 0 else "gemm_tc_kernel<192, 0, 1, 0, 0>"
        rd, wr = 1e6 * (i + 1), 2e5 * (i + 1)
        seq.append((kernel, {"gpu__time_duration.sum": ("usecond", "10"), "dram__bytes_read.sum": ("byte", str(rd)),
                             "dram__bytes_write.sum": ("byte", str(wr))}))
        b = rd + wr
        if n.endswith("_dw"):  # a split-K reduce after it, in Mbyte units
            seq.append(("split_reduce_kernel", {"gpu__time_duration.sum": ("usecond", "2"),
                                                "dram__bytes_read.sum": ("Mbyte", "3"),
                                                "dram__bytes_write.sum": ("Mbyte", "1")}))
            b += 4e6
        expect += STEP_GEMMS[n] * b
    out = NS.step_traffic(_write(tmp_path, seq))
    fields = dict(l.split(": ") for l in out.splitlines() if ": " in l)
    assert float(fields["traffic_bytes_per_step"]) == pytest.approx(expect)
    launches = sum(STEP_GEMMS[n] * (2 if n.endswith("_dw") else 1) for n in names)
    assert int(fields["launches_per_step"]) == launches
    assert float(fields["traffic_bytes_per_launch_full_step_avg"]) == pytest.approx(expect / launches, rel=1e-6)
    # one matmul short of the step: refused
    with pytest.raises(SystemExit):
        NS.step_traffic(_write(tmp_path, seq[1:]))
