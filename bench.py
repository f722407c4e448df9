"""Benchmark: GPT-2 training steps (forward, backward, AdamW) through the C ABI.

Default workload: GPT-2 124M shape, bf16 activations with fp32 master weights,
B=32, T=1024, Zipf(1.1) token ids with an EoS id every ~Poisson(700) tokens
(the pages' batch-32 peak-memory workload; synthetic data, random init).

One JSON line on rank 0:
  value      training tokens/s of the whole job (inputs resident in HBM),
             timed with CUDA events over exactly --steps steps after --warmup
             untimed steps, max over ranks;
  e2e        the same metric through the public API with the token batches
             copied from pinned host memory every step and the loss read back;
  roofline   the matmul kernel (the dominant one): algorithmic FLOPs / its
             CUDA-event time in an instrumented pass, against the measured
             sustained bf16 peak;
  cpu_baseline  the CPU oracle timed on this host (rank 0, N=1 only).
With --gpus N > 1 (under torchrun) every rank trains its own replica on its
own GPU and data; there is no exchange (replicas only).
--impl reference times the CPU oracle instead (the reference arm).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GPT-2 124M train tokens/sec on 1 GB300 (fwd+bwd+AdamW); MFU; kernel HBM GB/s"
SPEC_BF16_DENSE_TFLOPS = 2250.0  # NVIDIA's dense bf16 figure for one GB300
HP = dict(beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)


def lr_at(step: int) -> float:
    return 3e-4 * min(1.0, step / 5.0)  # linear warmup over 5 steps, then constant


def measured_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except Exception:
        return {}


def model_flops_per_token(L, C, V, T) -> float:
    """6 N + 12 L T C, N counted with the real vocabulary."""
    n = V * C + T * C + L * (12 * C * C + 13 * C) + 2 * C
    return 6.0 * n + 12.0 * L * T * C


def workload_cfg(name: str, B: int | None):
    from step_gpt_train_gb300 import data
    w = data.WORKLOADS[name]
    cfg = {k: w[k] for k in ("n_layer", "n_embd", "n_head", "vocab", "vocab_padded", "max_T", "mode")}
    cfg["max_B"] = B or w["B"]
    return w, cfg


def workload_label(name: str, w: dict, B: int, T: int) -> str:
    eos = " + EoS every ~Poisson(700)" if w["eos_every"] else ""
    model = {"124m-b32": "GPT-2 124M", "124m-b8": "GPT-2 124M", "350m-b16": "GPT-2 350M", "1p5b-b8": "GPT-2 1.5B",
             "tiny": "tiny GPT-2"}[name]
    prec = "bf16 activations, fp32 master" if w["mode"] == 1 else "fp32"
    return f"{model} training step, B={B}, T={T}, {prec}, {w['stream']} ids{eos}, random init"


class ClockSampler:
    """nvidia-smi clock and throttle samples, kept only where they fall inside
    the timed region. Each sample carries the time nvidia-smi took it (its
    timestamp field, local time); mark_start() / mark_stop() record the
    region's bounds on the host clock, and a sample counts when its timestamp
    lies between them (its arrival time when the timestamp does not parse).
    wait_first() returns once the first sample has arrived, so that the
    sampler's start-up does not eat into a short region."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 100

    def __init__(self, gpu_index: int, cmd: list[str] | None = None):
        import threading
        self.proc = None
        self.lines: list[tuple[float, str]] = []  # (arrival time, line)
        self.t_start = self.t_stop = None  # (monotonic, wall clock) pairs
        self._first = threading.Event()
        if cmd is None:
            cmd = ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                   "-lms", str(self.INTERVAL_MS)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self._reader = threading.Thread(target=self._read, daemon=True)
        self._reader.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line))
            self._first.set()

    def wait_first(self, timeout: float = 2.0) -> bool:
        return self.proc is not None and self._first.wait(timeout)

    @staticmethod
    def _now():
        import datetime
        return time.monotonic(), datetime.datetime.now()

    def mark_start(self):
        self.t_start = self._now()

    def mark_stop(self):
        self.t_stop = self._now()

    @staticmethod
    def _stamp(field: str):
        import datetime
        try:
            return datetime.datetime.strptime(field.strip(), "%Y/%m/%d %H:%M:%S.%f")
        except ValueError:
            return None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
            self.proc.wait()
        self._reader.join(timeout=5)
        inside, after = [], []
        for arrival, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            ts = self._stamp(parts[0])
            k = 1 if ts is not None else 0  # bound index: wall clock, else arrival time
            t = ts if ts is not None else arrival
            lo = self.t_start[k] if self.t_start else None
            hi = self.t_stop[k] if self.t_stop else None
            if (lo is None or t >= lo) and (hi is None or t <= hi):
                inside.append(parts)
            elif hi is not None and t > hi:
                after.append(parts)
        note = None
        if not inside and after:  # a region shorter than the interval: the first sample after it
            inside, note = after[:1], "no sample inside the timed region; the first one after it"
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for parts in inside:
            try:
                sm.append(float(parts[2]))
                mx.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[6:10]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
               "samples": len(sm)}
        if note:
            out["note"] = note
        return out


GEMM_SOURCES = ("gemm_tc.cu", "tc_common.cuh", "common.cuh")  # the matmul kernel and the headers it includes


def strip_code(text: str) -> str:
    """C/C++/CUDA source without its comments, whitespace runs collapsed to one
    space; string and character literals are kept as written."""
    out, i, n = [], 0, len(text)
    while i < n:
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif text[i] in "\"'":
            q, j = text[i], i + 1
            while j < n and text[j] != q:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(text[i])
            i += 1
    return " ".join("".join(out).split())


def gemm_code_digest() -> str:
    """sha256 (first 16 hex digits) of the matmul kernel's code: its source and
    the headers it includes, comments and whitespace aside, so that a change
    of a comment does not invalidate a measurement of the same code."""
    h = hashlib.sha256()
    for name in GEMM_SOURCES:
        with open(os.path.join(ROOT, "step_gpt_train_gb300", "csrc", name)) as f:
            h.update(strip_code(f.read()).encode())
        h.update(b"\0")
    return h.hexdigest()[:16]


def gemm_traffic_from_profile():
    """DRAM bytes per matmul launch from the committed ncu summary, if it was taken
    on the current matmul code; else None."""
    path = os.path.join(ROOT, "profiles", "gemm_tc_kernel_124m_b32.txt")
    try:
        text = open(path).read()
        digest = gemm_code_digest()
    except OSError:
        return None
    fields = dict(l.split(":", 1) for l in text.splitlines() if ":" in l)
    if fields.get("code_sha256_16", "").strip() != digest:
        return None
    try:
        return float(fields["traffic_bytes_per_launch_full_step_avg"].strip())
    except (KeyError, ValueError):
        return None


# Families bound by HBM bandwidth; the library counts their algorithmic
# bytes (each tensor read or written once) as their work. grad_colsum's bytes
# are the partial column sums it reads (scratch of the backward, not tensors
# of the model).
HBM_FAMILIES = ("encoder_forward", "layernorm_forward", "classifier", "loss_mean", "layernorm_backward",
                "bias_backward", "encoder_backward", "adamw", "residual_forward", "residual_backward",
                "gelu_forward", "gelu_backward", "grad_colsum", "fp8_quant")


def hbm_fractions(fam_ms: dict, stats: dict, steps: int, peaks: dict) -> dict:
    """Per HBM-bound family: algorithmic GB per step, CUDA-event ms per step,
    GB/s and the fraction of the measured copy bandwidth."""
    peak = peaks.get("hbm_gbs") or 6800.0
    out = {"peak_gbs": peak, "peak_source": "measured (MEASURED_PEAKS.json)" if peaks.get("hbm_gbs") else "fallback"}
    for f in HBM_FAMILIES:
        ms, work = fam_ms.get(f, 0.0), stats.get(f, {}).get("work", 0.0)
        if ms > 0 and work > 0:
            gbs = work / (ms / 1000.0) / 1e9
            out[f] = {"gb_per_step": work / steps / 1e9, "ms_per_step": ms / steps, "gbs": gbs,
                      "frac": gbs / peak}
    return out


def oracle_threads() -> int:
    """Threads the oracle's numpy BLAS runs on: threadpoolctl's report where it
    is installed, else the cores this process may run on."""
    try:
        from threadpoolctl import threadpool_info
        n = [p["num_threads"] for p in threadpool_info() if p.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def cpu_baseline(w_name: str):
    """The oracle, as it stands, on one bounded sample of the workload."""
    from oracle import gpt2_ref as R
    from step_gpt_train_gb300 import data
    w = data.WORKLOADS[w_name]
    cfg = R.Config(w["n_layer"], w["n_embd"], w["n_head"], w["vocab"], w["vocab_padded"], w["max_T"])
    T = 1024
    tok, tgt = data.workload_batches(w_name, 1, B=1, T=T)
    params = R.init_params(cfg, 1234)
    t0 = time.perf_counter()
    R.train_step(cfg, params, tok[0], tgt[0], None, lr_at(1), HP["beta1"], HP["beta2"], HP["eps"],
                 HP["weight_decay"], 1)
    dt = time.perf_counter() - t0
    return {"value": T / dt, "unit": "tokens/s", "cores": oracle_threads(), "kind": "oracle",
            "sample": f"one oracle train step (forward, backward, AdamW over all parameters), float64 numpy, "
                      f"GPT-2 {w_name.split('-')[0].upper()} shape, B=1, T={T}, first window of the same "
                      f"token stream; init excluded; {dt:.1f} s"}


def run_reference(args, rank: int):
    """Reference arm: the CPU oracle timed as it stands, on a bounded sample per step."""
    if rank != 0:
        return
    from oracle import gpt2_ref as R
    from step_gpt_train_gb300 import data
    w, _ = workload_cfg(args.config, None)
    cfg = R.Config(w["n_layer"], w["n_embd"], w["n_head"], w["vocab"], w["vocab_padded"], w["max_T"])
    B, T = 1, args.ref_T
    tok, tgt = data.workload_batches(args.config, args.warmup + args.steps, B=B, T=T)
    params = R.init_params(cfg, 1234)
    state = None
    times = []
    for s in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        _, _, params, state = R.train_step(cfg, params, tok[s], tgt[s], state, lr_at(s + 1), HP["beta1"],
                                           HP["beta2"], HP["eps"], HP["weight_decay"], s + 1)
        if s >= args.warmup:
            times.append(time.perf_counter() - t0)
    total = sum(times)
    value = B * T * len(times) / total
    sample = (f"each step one oracle train step (float64 numpy) at B={B}, T={T} of the {args.config} "
              f"stream; GPT-2 {args.config.split('-')[0].upper()} shape")
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1000 * total / len(times), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": workload_label(args.config, w, B, T), "sample_per_step": f"B={B}, T={T}"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="124m-b32")
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true",
                    help="separate gpt2_forward / gpt2_backward / gpt2_adamw_step calls instead of gpt2_step")
    ap.add_argument("--ref-T", type=int, default=256)
    ap.add_argument("--fp8", default="",
                    help="comma-separated FP8 linear layers (qkv, mlp, head): the FP8 variant of the step, "
                         "not the bf16 headline")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, rank)
        return

    import torch
    import torch.distributed as dist
    from step_gpt_train_gb300 import data
    from step_gpt_train_gb300.gpt2 import GPT2, load_library

    load_library(build=True)
    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    w, cfg = workload_cfg(args.config, args.batch)
    B, T = cfg["max_B"], w["T"]
    K, W = args.steps, args.warmup
    model = GPT2(cfg, seed=1234)
    fp8_names = [n for n in args.fp8.split(",") if n]
    fp8_bits = {"qkv": 1, "mlp": 2, "head": 4}
    if fp8_names:
        model.set_fp8(sum(fp8_bits[n] for n in fp8_names))
    stream = model.stream
    tok, tgt = data.workload_batches(args.config, W + K, seed=1234 + rank, B=B, T=T)
    d_tok = torch.from_numpy(tok).cuda()
    d_tgt = torch.from_numpy(tgt).cuda()

    def step(s, tk, tg):
        if not args.eager:  # one captured graph per step (gpt2_step)
            return model.step(tk, tg, lr_at(s + 1), t=s + 1, **HP)
        loss = model.forward(tk, tg)
        model.backward()
        model.adamw_step(lr_at(s + 1), t=s + 1, **HP)
        return loss

    def barrier():
        if world > 1:
            dist.barrier()

    # ---------------------------------------------------------------- device-resident timing
    for s in range(W):
        step(s, d_tok[s], d_tgt[s])
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank)
    sampler.wait_first()
    barrier()
    launches0 = model.launch_count()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler.mark_start()
    ev0.record(stream)
    losses = []
    for s in range(W, W + K):
        losses.append(step(s, d_tok[s], d_tgt[s]))
    ev1.record(stream)
    torch.cuda.synchronize()
    sampler.mark_stop()
    barrier()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    launches = model.launch_count() - launches0
    ms = ev0.elapsed_time(ev1) / K
    if world > 1:
        t = torch.tensor([ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    tokens_per_step = B * T * world
    value = tokens_per_step / (ms / 1000.0)

    # ---------------------------------------------------------------- end to end through the API
    pin_tok = torch.from_numpy(tok).pin_memory()
    pin_tgt = torch.from_numpy(tgt).pin_memory()
    buf_tok = torch.empty(B, T, dtype=torch.int32, device="cuda")
    buf_tgt = torch.empty(B, T, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    for k in range(K):
        s, t = W + k, W + K + k
        if not args.eager:
            # the library's host-buffer entry point copies the batch in itself
            model.step_host(pin_tok[s], pin_tgt[s], lr_at(t + 1), t=t + 1, **HP)
            continue
        with torch.cuda.stream(stream):
            buf_tok.copy_(pin_tok[s], non_blocking=True)
            buf_tgt.copy_(pin_tgt[s], non_blocking=True)
        step(t, buf_tok, buf_tgt)  # the loss comes back to the host inside forward
    torch.cuda.synchronize()
    e2e_s = (time.perf_counter() - t0) / K
    if world > 1:
        t = torch.tensor([e2e_s], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_s = float(t.item())
    e2e = {"value": tokens_per_step / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": 2 * B * T * 4,
           "d2h_bytes_per_step": 8,  # the loss and the status word
           "api": "gpt2_step_host: pinned host token/target buffers, copied to the device inside the call, "
                  "loss read back" if not args.eager else
                  "torch copies from pinned host memory, then gpt2_forward / gpt2_backward / gpt2_adamw_step"}

    # ---------------------------------------------------------------- instrumented pass: per-kernel times
    model.reset_stats()
    model.set_timing(True)
    for k in range(K):
        s = W + k
        step(2 * (W + K) + k, d_tok[s], d_tgt[s])
    fam_ms = model.family_times_ms()
    stats = model.family_stats()
    model.set_timing(False)
    peaks = measured_peaks()
    mm_ms = fam_ms["matmul"]
    mm_flops = stats["matmul"]["work"]
    mm_launches = stats["matmul"]["launches"]
    achieved = mm_flops / (mm_ms / 1000.0) / 1e12 if mm_ms > 0 else None
    peak = peaks.get("bf16_tflops_sustained")
    peak_src = "measured sustained (MEASURED_PEAKS.json)"
    if not peak:
        peak, peak_src = 1700.0, "fallback"
    # the committed traffic capture is of the 124M B=32 step's matmuls (bf16): other
    # workloads have none
    traffic = gemm_traffic_from_profile() if not fp8_names and args.config == "124m-b32" and B == 32 else None
    if fp8_names:
        # the family mixes FP8 and bf16 products: reported against the bf16 peak
        peak_src += "; the FP8 products' own peak is twice it (the nominal e4m3 : bf16 ratio)"
    roofline = {"kernel": "gemm_tc_kernel and gemm_pair_kernel (every matmul of the step)", "bound": "tensor",
                "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": (achieved / peak) if achieved else None, "peak_source": peak_src,
                "traffic": traffic, "launches_per_step": mm_launches / K,
                "flops_per_step": mm_flops / K}
    kernel_ms = {f: v / K for f, v in fam_ms.items() if v > 0}
    hbm = hbm_fractions(fam_ms, stats, K, peaks)

    fpt = model_flops_per_token(cfg["n_layer"], cfg["n_embd"], cfg["vocab"], T)
    tflops = value * fpt / 1e12
    mfu = {"model_flops_per_token": fpt, "tflops": tflops / world,
           "vs_spec_2250": tflops / world / SPEC_BF16_DENSE_TFLOPS,
           "vs_measured_burst": (tflops / world / peaks["bf16_tflops"]) if peaks.get("bf16_tflops") else None}

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if not fp8_names else "bf16 + fp8 (e4m3 activations/weights, e5m2 gradients) in "
                                                   + "/".join(fp8_names),
            "data": "synthetic",
            "config": {"workload": workload_label(args.config, w, B, T),
                       "parallelism": f"replicas x{world} (no exchange)" if world > 1 else "single GPU",
                       "l2": "inputs larger than L2: each step touches ~15 GB of weights, activations and state",
                       "api": "gpt2_forward, gpt2_backward, gpt2_adamw_step" if args.eager
                       else "gpt2_step (the step replayed as one CUDA graph)",
                       "roofline_pass": "per-kernel times from a separate instrumented pass of the same steps",
                       **({"fp8_linears": fp8_names} if fp8_names else {})},
            "e2e": e2e, "gpu_launches": launches, "clocks": clocks, "roofline": roofline, "mfu": mfu,
            "kernel_ms_per_step": kernel_ms, "hbm": hbm, "loss_first_last": [losses[0], losses[-1]],
            "workspace_bytes": model.bytes + getattr(model, "fp8_bytes", 0),
            "peak_device_bytes": torch.cuda.max_memory_allocated()}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.config)
    if rank == 0:
        print(json.dumps(line), flush=True)
    model.close()
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
