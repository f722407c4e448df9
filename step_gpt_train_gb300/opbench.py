"""Per-kernel micro-benchmark of the GPT-2 step's ops at a model's shapes.

Each op runs through its C entry point (gpt2_ops.h) on device buffers,
timed with CUDA events on the launching stream after warm-up, and is
reported against its roofline: algorithmic FLOPs against the measured bf16
peak for the matmuls and attention, algorithmic bytes against the measured
HBM bandwidth for the rest. Also the small, self-contained program for ncu
captures of one kernel.

  python -m step_gpt_train_gb300.opbench [--ops a,b|all|step_gemms|cublas_step_gemms] [--iters N] [--B 32 --T 1024 --C 768 --H 12]

cublas_step_gemms times torch.matmul (cuBLAS) on the plain matmul shapes of the
step, a reference point for the hand-written kernels (not part of the step).
"""
from __future__ import annotations

import argparse
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


# The matmuls of one bf16 training step and how often each runs (per layer
# the forward QKV, attention projection, MLP up-projection with its GELU and
# MLP down-projection, their input and weight gradients, and the tied LM
# head's three): `--ops step_gemms` runs each once, in this order.
def step_gemm_counts(L: int = 12) -> dict:
    per_layer = ["gemm_qkv_fwd", "gemm_proj_fwd", "gemm_fc_fwd_gelu", "gemm_fcproj_fwd", "gemm_fcproj_dw",
                 "gemm_fcproj_dx_gelu_bias", "gemm_fc_dw", "gemm_fc_dx", "gemm_proj_dw", "gemm_proj_dx", "gemm_qkv_dw",
                 "gemm_qkv_dx"]
    counts = {n: L for n in per_layer}
    counts.update({"gemm_lmhead_fwd": 1, "gemm_lmhead_dx": 1, "gemm_lmhead_dw": 1})
    return counts


STEP_GEMMS = step_gemm_counts()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p["hbm_gbs"], p["bf16_tflops"], "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--ops", default="all")
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--B", type=int, default=32)
    ap.add_argument("--T", type=int, default=1024)
    ap.add_argument("--C", type=int, default=768)
    ap.add_argument("--H", type=int, default=12)
    ap.add_argument("--V", type=int, default=50257)
    ap.add_argument("--Vp", type=int, default=50304)
    ap.add_argument("--pair", type=int, default=None,
                    help="route the wide matmuls to the CTA-pair kernel (1) or to the one-CTA kernel (0)")
    args = ap.parse_args(argv)

    import torch
    from step_gpt_train_gb300 import gpt2 as g

    g.load_library(build=True)
    torch.cuda.set_device(0)
    if args.pair is not None:
        g.load_library().gpt2_debug_matmul_pair(args.pair)
    hbm, tc, src = peaks()
    B, T, C, H, V, Vp = args.B, args.T, args.C, args.H, args.V, args.Vp
    N = B * T
    bf = torch.bfloat16
    dev = "cuda"

    def rnd(*shape, dtype=bf, std=1.0):
        return (torch.randn(*shape, device=dev) * std).to(dtype)

    ops = {}

    def gemm_op(M, Nn, K, a_mn, b_mn, fp32_out, bias):
        def setup():
            A = rnd(M * K)
            Bm = rnd(Nn * K, std=0.02)
            D = torch.empty(M, Nn, device=dev, dtype=torch.float32 if fp32_out else bf)
            b = rnd(Nn) if bias else None
            sc = torch.empty(max(256, g.load_library().gpt2_op_matmul_scratch(1, M, Nn, K, int(fp32_out))),
                             dtype=torch.uint8, device=dev)
            lib = g.load_library()

            def run():
                g.check(lib.gpt2_op_matmul(1, D.data_ptr(), int(fp32_out), A.data_ptr(), a_mn, Bm.data_ptr(),
                                           b_mn, b.data_ptr() if b is not None else None, M, Nn, K,
                                           sc.data_ptr(), sc.numel(), None, torch.cuda.current_stream().cuda_stream))
            return run
        return setup, 2.0 * M * Nn * K, "flop"

    def cublas_op(M, Nn, K, a_mn, b_mn):
        # the same product through torch.matmul (cuBLAS), bf16 output, for
        # comparison only: D[M, N] = A(m, k) B(n, k), A stored [M][K] or [K][M]
        # (a_mn), B stored [N][K] or [K][N] (b_mn)
        def setup():
            A = rnd(M * K)
            Bm = rnd(Nn * K, std=0.02)
            a = A.view(K, M).t() if a_mn else A.view(M, K)
            b = Bm.view(K, Nn) if b_mn else Bm.view(Nn, K).t()
            D = torch.empty(M, Nn, device=dev, dtype=bf)
            return lambda: torch.matmul(a, b, out=D)
        return setup, 2.0 * M * Nn * K, "flop"

    shapes = {"qkv": (3 * C, C), "proj": (C, C), "fc": (4 * C, C), "fcproj": (C, 4 * C), "lmhead": (Vp, C)}
    for name, (out, inp) in shapes.items():
        ops[f"gemm_{name}_fwd"] = gemm_op(N, out, inp, 0, 0, False, name != "lmhead")
        ops[f"gemm_{name}_dx"] = gemm_op(N, inp, out, 0, 1, False, False)
        ops[f"gemm_{name}_dw"] = gemm_op(out, inp, N, 1, 1, True, False)
        ops[f"cublas_{name}_fwd"] = cublas_op(N, out, inp, 0, 0)
        ops[f"cublas_{name}_dx"] = cublas_op(N, inp, out, 0, 1)
        ops[f"cublas_{name}_dw"] = cublas_op(out, inp, N, 1, 1)


    def gemm_gelu_op():  # the MLP's first linear with its GELU in the epilogue
        def setup():
            A, W, b = rnd(N, C), rnd(4 * C, C, std=0.02), rnd(4 * C)
            pre, out = torch.empty(N, 4 * C, device=dev, dtype=bf), torch.empty(N, 4 * C, device=dev, dtype=bf)
            return lambda: g.gpt2_op_matmul_gelu(pre, out, A, W, b, stream=torch.cuda.current_stream())
        return setup, 2.0 * N * 4 * C * C, "flop"

    def gemm_gelu_bwd_op():  # the MLP projection's input gradient through the GELU
        def setup():
            dY, W, u = rnd(N, C), rnd(C, 4 * C, std=0.02), rnd(N, 4 * C)
            du = torch.empty(N, 4 * C, device=dev, dtype=bf)
            return lambda: g.gpt2_op_matmul_gelu_backward(du, dY, W, u, stream=torch.cuda.current_stream())
        return setup, 2.0 * N * 4 * C * C, "flop"

    def gemm_fp8_op(Nn, K, a_fmt=g.FP8_E4M3, use_bias=True):
        # FP8 linear layer (codes quantized once; the GEMM is timed): A [N, K] in a_fmt
        # (e4m3 activations, or an e5m2 gradient for an input gradient), W [Nn, K] e4m3
        def setup():
            A, W, b = rnd(N, K), rnd(Nn, K, std=0.02), rnd(Nn)
            qa = torch.empty(N, K, device=dev, dtype=torch.uint8)
            qw = torch.empty(Nn, K, device=dev, dtype=torch.uint8)
            sa = torch.empty(2, device=dev, dtype=torch.float32)
            sw = torch.empty(2, device=dev, dtype=torch.float32)
            g.gpt2_op_quantize_fp8(qa, sa, A, a_fmt)
            g.gpt2_op_quantize_fp8(qw, sw, W)
            D = torch.empty(N, Nn, device=dev, dtype=bf)
            return lambda: g.gpt2_op_matmul_fp8(D, qa, sa, qw, sw, bias=b if use_bias else None, a_fmt=a_fmt,
                                                stream=torch.cuda.current_stream())
        return setup, 2.0 * N * Nn * K, "flop8"

    def quantize_op():  # per-tensor e4m3 quantization of the MLP's hidden activations
        def setup():
            x = rnd(N, 4 * C)
            q = torch.empty(N, 4 * C, device=dev, dtype=torch.uint8)
            sc = torch.empty(2, device=dev, dtype=torch.float32)
            return lambda: g.gpt2_op_quantize_fp8(q, sc, x, stream=torch.cuda.current_stream())
        return setup, N * 4.0 * C * (2 * 2 + 1), "byte"  # amax pass reads x, quantize reads x, writes q

    ops["gemm_fc_fwd_fp8"] = gemm_fp8_op(4 * C, C)
    ops["gemm_fcproj_fwd_fp8"] = gemm_fp8_op(C, 4 * C)
    # input gradient of the MLP down-projection: dY [N, C] (e5m2) times W^T stored [4C, C] (e4m3)
    ops["gemm_fcproj_dx_fp8_e5m2"] = gemm_fp8_op(4 * C, C, a_fmt=g.FP8_E5M2, use_bias=False)
    ops["quantize_fp8"] = quantize_op()

    def quantize_t_op():  # both layouts of the MLP's hidden activations' codes (the FP8 step's forward)
        def setup():
            x = rnd(N, 4 * C)
            q = torch.empty(N, 4 * C, device=dev, dtype=torch.uint8)
            qt = torch.empty(4 * C, N, device=dev, dtype=torch.uint8)
            sc = torch.empty(2, device=dev, dtype=torch.float32)
            g.gpt2_op_quantize_fp8(q, sc, x)
            return lambda: g.gpt2_op_quantize_fp8_transpose(qt, sc, x, q=q, stream=torch.cuda.current_stream())
        return setup, N * 4.0 * C * (2 + 1 + 1), "byte"  # reads x, writes q and qt

    ops["quantize_fp8_transpose"] = quantize_t_op()
    def gemm_gelu_bwd_bias_op():  # the same, with the MLP's first bias gradient from its epilogue
        def setup():
            dY, W, u = rnd(N, C), rnd(C, 4 * C, std=0.02), rnd(N, 4 * C)
            du = torch.empty(N, 4 * C, device=dev, dtype=bf)
            db = torch.empty(4 * C, device=dev)
            sc = torch.empty(g.load_library().gpt2_op_matmul_gelu_backward_bias_scratch(N, 4 * C), device=dev,
                             dtype=torch.uint8)
            lib = g.load_library()
            return lambda: g.check(lib.gpt2_op_matmul_gelu_backward_bias(
                1, du.data_ptr(), db.data_ptr(), dY.data_ptr(), W.data_ptr(), u.data_ptr(), N, 4 * C, C,
                sc.data_ptr(), sc.numel(), None, torch.cuda.current_stream().cuda_stream))
        return setup, 2.0 * N * 4 * C * C, "flop"

    ops["gemm_fc_fwd_gelu"] = gemm_gelu_op()
    ops["gemm_fcproj_dx_gelu"] = gemm_gelu_bwd_op()
    ops["gemm_fcproj_dx_gelu_bias"] = gemm_gelu_bwd_bias_op()

    def attn_fwd():
        qkv = rnd(N, 3 * C)
        o = torch.empty(N, C, device=dev, dtype=bf)
        lse = torch.empty(B * H * T, device=dev)
        return lambda: g.gpt2_op_attention_forward(o, lse, qkv, B, T, H)

    def attn_bwd():
        qkv = rnd(N, 3 * C)
        o = torch.empty(N, C, device=dev, dtype=bf)
        lse = torch.empty(B * H * T, device=dev)
        g.gpt2_op_attention_forward(o, lse, qkv, B, T, H)
        do = rnd(N, C)
        dq = torch.empty_like(qkv)
        sc = torch.empty(B * H * T * 4, dtype=torch.uint8, device=dev)
        lib = g.load_library()
        return lambda: g.check(lib.gpt2_op_attention_backward(1, dq.data_ptr(), do.data_ptr(), qkv.data_ptr(),
                                                              o.data_ptr(), lse.data_ptr(), B, T, C, H,
                                                              sc.data_ptr(), sc.numel(),
                                                              torch.cuda.current_stream().cuda_stream))

    att_flops = 4.0 * B * C * T * (T + 1) / 2
    ops["attention_fwd"] = (attn_fwd, att_flops, "flop")
    ops["attention_bwd"] = (attn_bwd, 2.5 * att_flops, "flop")

    def ln_fwd():
        x, gm, bt = rnd(N, C), rnd(C), rnd(C)
        y = torch.empty_like(x)
        mean, rstd = torch.empty(N, device=dev), torch.empty(N, device=dev)
        return lambda: g.gpt2_op_layernorm_forward(y, mean, rstd, x, gm, bt)

    def ln_bwd():
        x, gm, bt, dy = rnd(N, C), rnd(C), rnd(C), rnd(N, C)
        y = torch.empty_like(x)
        mean, rstd = torch.empty(N, device=dev), torch.empty(N, device=dev)
        g.gpt2_op_layernorm_forward(y, mean, rstd, x, gm, bt)
        dx = torch.empty_like(x)
        dgm, dbt = torch.empty(C, device=dev), torch.empty(C, device=dev)
        lib = g.load_library()
        sc = torch.empty(lib.gpt2_op_layernorm_backward_scratch(N, C), dtype=torch.uint8, device=dev)
        return lambda: g.check(lib.gpt2_op_layernorm_backward(1, dx.data_ptr(), dgm.data_ptr(), dbt.data_ptr(),
                                                              dy.data_ptr(), x.data_ptr(), gm.data_ptr(),
                                                              mean.data_ptr(), rstd.data_ptr(), N, C,
                                                              sc.data_ptr(), sc.numel(),
                                                              torch.cuda.current_stream().cuda_stream))

    def ln_fwd_res():  # the step's form: residual join then LayerNorm
        x, r, gm, bt = rnd(N, C), rnd(N, C), rnd(C), rnd(C)
        y, xs = torch.empty_like(x), torch.empty_like(x)
        mean, rstd = torch.empty(N, device=dev), torch.empty(N, device=dev)
        return lambda: g.gpt2_op_residual_layernorm_forward(y, mean, rstd, xs, x, r, gm, bt)

    def ln_bwd_res():  # the step's form: into the residual gradient, with the bias column sums
        x, gm, bt, dy, dres = rnd(N, C), rnd(C), rnd(C), rnd(N, C), rnd(N, C)
        y = torch.empty_like(x)
        mean, rstd = torch.empty(N, device=dev), torch.empty(N, device=dev)
        g.gpt2_op_layernorm_forward(y, mean, rstd, x, gm, bt)
        dgm, dbt, dbias = (torch.empty(C, device=dev) for _ in range(3))
        return lambda: g.gpt2_op_layernorm_backward_residual(dres, 1, dgm, dbt, dbias, dy, x, gm, mean, rstd)

    ops["layernorm_fwd"] = (ln_fwd, N * (2.0 * C * 2 + 8), "byte")
    ops["layernorm_bwd"] = (ln_bwd, N * (3.0 * C * 2 + 8), "byte")
    ops["layernorm_fwd_res"] = (ln_fwd_res, N * (4.0 * C * 2 + 8), "byte")
    ops["layernorm_bwd_res"] = (ln_bwd_res, N * (4.0 * C * 2 + 8), "byte")

    def gelu_fwd():
        u = rnd(N * 4 * C)
        out = torch.empty_like(u)
        return lambda: g.gpt2_op_gelu_forward(out, u)

    def gelu_bwd():
        u, dgr = rnd(N * 4 * C), rnd(N * 4 * C)
        return lambda: g.gpt2_op_gelu_backward(dgr, u, dgr)

    ops["gelu_fwd"] = (gelu_fwd, N * 4.0 * C * 4, "byte")
    ops["gelu_bwd"] = (gelu_bwd, N * 4.0 * C * 6, "byte")

    def residual():
        a, b_ = rnd(N * C), rnd(N * C)
        out = torch.empty_like(a)
        return lambda: g.gpt2_op_residual_forward(out, a, b_)

    ops["residual_fwd"] = (residual, N * C * 6.0, "byte")

    def bias_bwd(cols):
        def setup():
            dy = rnd(N, cols)
            db = torch.empty(cols, device=dev)
            lib = g.load_library()
            sc = torch.empty(lib.gpt2_op_bias_backward_scratch(N, cols), dtype=torch.uint8, device=dev)
            return lambda: g.check(lib.gpt2_op_bias_backward(1, db.data_ptr(), dy.data_ptr(), N, cols,
                                                             sc.data_ptr(), sc.numel(),
                                                             torch.cuda.current_stream().cuda_stream))
        return setup

    ops["bias_bwd_fc"] = (bias_bwd(4 * C), N * 4.0 * C * 2, "byte")
    ops["bias_bwd_qkv"] = (bias_bwd(3 * C), N * 3.0 * C * 2, "byte")
    ops["bias_bwd_proj"] = (bias_bwd(C), N * C * 2.0, "byte")

    def classifier():
        z = rnd(N, Vp, std=2.0)
        z0 = z.clone()
        losses = torch.empty(N, device=dev)
        tgt = torch.randint(0, V, (N,), device=dev, dtype=torch.int32)

        def run():
            g.gpt2_op_classifier(z, losses, tgt, V, 1.0 / N)
        return run

    ops["classifier"] = (classifier, N * (2.0 * Vp * 2 + 8), "byte")

    def adamw():
        n = 124_475_904
        th, gr, m, v = (torch.randn(n, device=dev) for _ in range(4))
        v.abs_()
        pb = torch.empty(n, dtype=bf, device=dev)
        return lambda: g.gpt2_op_adamw(th, pb, gr, m, v, 1e-9, 0.9, 0.95, 1e-8, 0.0, 1)

    ops["adamw"] = (adamw, 124_475_904 * 30.0, "byte")

    def enc_fwd():
        tok = torch.randint(0, V, (B, T), device=dev, dtype=torch.int32)
        wte, wpe = rnd(Vp, C), rnd(T, C)
        x0 = torch.empty(N, C, device=dev, dtype=bf)
        return lambda: g.gpt2_op_encoder_forward(x0, tok, wte, wpe, V)

    def enc_bwd():
        from step_gpt_train_gb300 import data
        tok = torch.from_numpy(data.token_stream("zipf", N, 3).reshape(B, T)).cuda()
        dx0 = rnd(N, C)
        dwte, dwpe = torch.zeros(Vp, C, device=dev), torch.zeros(T, C, device=dev)
        lib = g.load_library()
        sc = torch.empty(lib.gpt2_op_encoder_backward_scratch(B, T, C), dtype=torch.uint8, device=dev)
        return lambda: g.check(lib.gpt2_op_encoder_backward(1, dwte.data_ptr(), dwpe.data_ptr(), dx0.data_ptr(),
                                                            tok.data_ptr(), B, T, C, Vp, sc.data_ptr(), sc.numel(),
                                                            torch.cuda.current_stream().cuda_stream))

    ops["encoder_fwd"] = (enc_fwd, N * (3.0 * C * 2 + 4), "byte")
    ops["encoder_bwd"] = (enc_bwd, N * (C * 2 * 2.0 + 8) + T * C * 4.0, "byte")

    if args.ops == "step_gemms":
        names = list(STEP_GEMMS)
    elif args.ops == "cublas_step_gemms":  # cuBLAS on the step's plain matmul shapes, for comparison
        names = [n for n in ops if n.startswith("cublas_")]
    else:
        names = list(ops) if args.ops == "all" else args.ops.split(",")
    for name in names:
        setup, work, kind = ops[name]
        run = setup()
        for _ in range(args.warmup):
            run()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.iters):
            run()
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1000.0 / args.iters
        if kind == "flop":
            achieved = work / (us * 1e-6) / 1e12
            rec = {"op": name, "us": us, "tflops": achieved, "frac_of_bf16_peak": achieved / tc}
        elif kind == "flop8":  # e4m3 dense peak: twice the bf16 one (the nominal ratio)
            achieved = work / (us * 1e-6) / 1e12
            rec = {"op": name, "us": us, "tflops": achieved, "frac_of_fp8_peak": achieved / (2 * tc)}
        else:
            achieved = work / (us * 1e-6) / 1e9
            rec = {"op": name, "us": us, "gbs": achieved, "frac_of_hbm": achieved / hbm}
        rec["peaks"] = src
        print(json.dumps(rec), flush=True)
        del run
        torch.cuda.empty_cache()


if __name__ == "__main__":
    main()
