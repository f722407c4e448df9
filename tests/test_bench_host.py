"""Host-side logic of bench.py that needs no GPU: the clock sampler's window
(a fake nvidia-smi prints numbered samples) and the parsing of its lines."""
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

# prints one sample every 20 ms with the time it was taken: the SM clock field
# is the sample's number
FAKE = ("import datetime, signal, sys, time\n"
        "signal.signal(signal.SIGTERM, lambda *a: sys.exit(0))\n"  # exits through Python: stdout is flushed
        "for k in range(1000):\n"
        "    r = 'Active' if k % 2 else 'Not Active'\n"
        "    ts = {stamp}\n"
        "    print(f'{{ts}}, 0, {{k}}, 2070, 900.0, 0x4, Not Active, Not Active, Not Active, {{r}}', flush={flush})\n"
        "    time.sleep(0.02)\n")
NOW = "datetime.datetime.now().strftime('%Y/%m/%d %H:%M:%S.%f')[:-3]"


def sampler(stamp=NOW, flush=True):
    return bench.ClockSampler(0, cmd=[sys.executable, "-c", FAKE.format(stamp=stamp, flush=flush)])


def clock_of(line):
    return int(line.split(",")[2])


def test_only_samples_inside_the_window_count():
    s = sampler()
    assert s.wait_first(10.0)
    time.sleep(0.2)
    s.mark_start()
    time.sleep(0.4)
    s.mark_stop()
    time.sleep(0.2)
    total_before_stop = len(s.lines)
    out = s.stop()
    assert out is not None and "note" not in out
    # about 20 samples in 0.4 s; none of the ~10 before the window nor the ~10 after it
    assert 5 <= out["samples"] <= 30
    assert out["samples"] < total_before_stop
    first_inside = min(clock_of(line) for t, line in s.lines if s.t_start[0] <= t <= s.t_stop[0])
    assert first_inside >= 3  # the samples before mark_start were left out
    assert out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]  # every other sample reports it


def test_region_shorter_than_the_interval_takes_the_next_sample():
    s = sampler()
    assert s.wait_first(10.0)
    time.sleep(0.05)
    s.mark_start()
    s.mark_stop()  # an empty window
    time.sleep(0.1)
    out = s.stop()
    assert out["samples"] == 1 and "note" in out


def test_missing_tool_gives_none():
    s = bench.ClockSampler(0, cmd=["/nonexistent/nvidia-smi-missing"])
    assert not s.wait_first(0.1)
    assert s.stop() is None


def test_model_flops_per_token_matches_the_published_count():
    # 6 N + 12 L T C with N = 124,439,808 (GPT-2 124M with the real vocabulary)
    n = 124_439_808
    assert bench.model_flops_per_token(12, 768, 50257, 1024) == 6.0 * n + 12.0 * 12 * 1024 * 768


def test_buffered_output_is_placed_by_its_timestamp():
    # a sampler whose output reaches the pipe only at exit: arrival times say
    # nothing, the samples' own timestamps still place them in the window
    s = sampler(flush=False)
    time.sleep(0.2)
    s.mark_start()
    time.sleep(0.4)
    s.mark_stop()
    time.sleep(0.2)
    out = s.stop()
    assert out is not None and "note" not in out
    assert 5 <= out["samples"] <= 30


def test_without_timestamps_arrival_time_decides():
    s = sampler(stamp="'n/a'")
    assert s.wait_first(10.0)
    time.sleep(0.2)
    s.mark_start()
    time.sleep(0.4)
    s.mark_stop()
    time.sleep(0.2)
    out = s.stop()
    assert out is not None and 5 <= out["samples"] <= 30


def test_strip_code_drops_comments_only():
    src = ('int a = 1; // a comment\n/* a block\n comment */ const char* s = "x // y /* z */";\n'
           "char q = '\\''; asm(\"mov.b32 %0, %1;\" : \"=r\"(a));\n")
    out = bench.strip_code(src)
    assert "comment" not in out
    assert '"x // y /* z */"' in out and "'\\''" in out and '"mov.b32 %0, %1;"' in out
    # a changed comment or re-indented code leaves the digest input unchanged; a changed token does not
    assert bench.strip_code(src.replace("a comment", "another note").replace("int a", "int   a")) == out
    assert bench.strip_code(src.replace("int a = 1", "int a = 2")) != out


def test_gemm_traffic_is_read_only_for_the_captured_code():
    # the committed summary carries the digest of the code it measured; the
    # bench reports its traffic only while the digest matches the sources
    text = open(os.path.join(ROOT, "profiles", "gemm_tc_kernel_124m_b32.txt")).read()
    fields = dict(l.split(":", 1) for l in text.splitlines() if ":" in l)
    got = bench.gemm_traffic_from_profile()
    if fields["code_sha256_16"].strip() == bench.gemm_code_digest():
        assert got == float(fields["traffic_bytes_per_launch_full_step_avg"])
    else:
        assert got is None


def run_bench(args, env_extra=None):
    import json
    import subprocess
    env = dict(os.environ, **(env_extra or {}))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                       timeout=300, env=env, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    return [json.loads(l) for l in lines]


def test_reference_arm_line_has_the_contract_keys():
    # the oracle arm needs no GPU: the tiny workload keeps it to seconds
    (line,) = run_bench(["--impl", "reference", "--config", "tiny", "--steps", "2", "--warmup", "3", "--ref-T", "64"])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in line, k
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 3 and line["n_gpus"] == 1
    assert line["unit"] == "tokens/s" and line["higher_is_better"] is True and line["value"] > 0
    assert line["vs_baseline"] is None and "workload" in line["config"]
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1 and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert abs(line["ms_per_step"] - 64 * 1000.0 / line["value"]) < 1e-6 * line["ms_per_step"]


def test_reference_arm_runs_on_rank_zero_only():
    assert run_bench(["--impl", "reference", "--config", "tiny", "--steps", "1", "--ref-T", "8", "--gpus", "2"],
                     {"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}) == []


def test_warmup_floor_is_three():
    (line,) = run_bench(["--impl", "reference", "--config", "tiny", "--steps", "1", "--warmup", "0", "--ref-T", "8"])
    assert line["warmup"] == 3
