"""FP8 linear layers in the training step (the modded-nanogpt project page,
"NanoGPT (124M) in 90 seconds", "How it works": FP8 for the MLP forward and
backward passes, the QKV projections and the head): the transposing
quantizer and the general FP8 product against the oracle, then whole steps
with FP8 linears against the oracle's step with the same linears quantized
(oracle.gpt2_ref forward/backward with fp8=...), under the bf16 step's
acceptance bounds."""
import numpy as np
import pytest

from oracle import fp8_ref as F
from oracle import gpt2_ref as R
from step_gpt_train_gb300 import data
from tests._gpu_util import BF16_REL, assert_close, dev, host, inputs, rel_l2
from tests.test_gpu_step import HP, check_step, make_model, oracle_steps, rcfg, run_steps

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    from step_gpt_train_gb300 import gpt2 as g
    g.load_library(build=True)
    torch.cuda.set_device(0)
    return torch


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("R_, C", [(200, 136), (1000, 768), (64, 64), (4096, 3072)])
def test_quantize_fp8_transpose_bit_exact(torch_cuda, R_, C, fmt):
    """The transposing quantizer writes the codes gpt2_op_quantize_fp8 gives
    for the same values and scales, transposed (and untransposed when asked),
    bit for bit, ragged tiles included; and they are the oracle's codes."""
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import (FP8_E4M3, FP8_E5M2, gpt2_op_quantize_fp8,
                                           gpt2_op_quantize_fp8_transpose)
    code = FP8_E4M3 if fmt == "e4m3" else FP8_E5M2
    x = inputs(81, (R_, C), 1.0)
    x[::7, ::13] *= 50.0
    x = data.round_to_bf16(x)  # the values the device holds
    dx = dev(x)
    q = torch.empty((R_, C), dtype=torch.uint8, device="cuda")
    sc = torch.zeros(2, dtype=torch.float32, device="cuda")
    gpt2_op_quantize_fp8(q, sc, dx, code)
    qt = torch.full((C, R_), 0xAA, dtype=torch.uint8, device="cuda")
    q2 = torch.full((R_, C), 0xAA, dtype=torch.uint8, device="cuda")
    gpt2_op_quantize_fp8_transpose(qt, sc, dx, q=q2, fmt=code)
    qt_only = torch.full((C, R_), 0x55, dtype=torch.uint8, device="cuda")
    gpt2_op_quantize_fp8_transpose(qt_only, sc, dx, fmt=code)
    torch.cuda.synchronize()
    hq = q.cpu().numpy()
    assert np.array_equal(qt.cpu().numpy(), hq.T)
    assert np.array_equal(q2.cpu().numpy(), hq)
    assert np.array_equal(qt_only.cpu().numpy(), hq.T)
    ref_q, _ = F.quantize(x, fmt)
    assert np.array_equal(hq, ref_q)


# M, N, K, epi, d_fp32, accumulate, A format, bias
EX_CASES = [
    (768, 768, 32768, 0, 1, 0, "e5m2", False),   # a weight gradient: fp32 output, split-K partials
    (2304, 768, 8192, 0, 1, 1, "e5m2", False),   # ... added to the gradient held (accumulation)
    (300, 264, 272, 0, 1, 1, "e5m2", False),     # ragged
    (1000, 3072, 768, 1, 0, 0, "e4m3", True),    # the MLP's first linear with its GELU
    (300, 200, 272, 1, 0, 0, "e4m3", True),
    (1000, 3072, 768, 2, 0, 0, "e5m2", False),   # the input gradient through the GELU
    (300, 200, 272, 2, 0, 0, "e5m2", False),
]


@pytest.mark.parametrize("case", EX_CASES)
def test_matmul_fp8_ex(torch_cuda, case):
    """The general FP8 product against the oracle's product of the same codes
    and scales: fp32 (split-K, accumulated) weight-gradient outputs, the GELU
    forward epilogue (gelu'(u) and gelu(u) of u rounded to bf16) and the GELU
    backward epilogue (bf16 product times the factor)."""
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import FP8_E4M3, FP8_E5M2, gpt2_op_matmul_fp8_ex, gpt2_op_quantize_fp8
    M, N, K, epi, d_fp32, acc, fa, use_bias = case
    code = {"e4m3": FP8_E4M3, "e5m2": FP8_E5M2}
    A = inputs(91, (M, K), 1.0)
    W = inputs(92, (N, K), K ** -0.5)
    bias = inputs(93, (N,), 0.5) if use_bias else None
    qa = torch.empty((M, K), dtype=torch.uint8, device="cuda")
    qw = torch.empty((N, K), dtype=torch.uint8, device="cuda")
    sa = torch.zeros(2, dtype=torch.float32, device="cuda")
    sw = torch.zeros(2, dtype=torch.float32, device="cuda")
    gpt2_op_quantize_fp8(qa, sa, dev(A), code[fa])
    gpt2_op_quantize_fp8(qw, sw, dev(W), FP8_E4M3)
    ca, cw = qa.cpu().numpy(), qw.cpu().numpy()
    ref = F.matmul_fp8(ca, sa.cpu().numpy()[1], cw, sw.cpu().numpy()[1], bias, a_fmt=fa, b_fmt="e4m3")
    atol = (K / 32) * 2.0 ** -23 * 8 * float(np.abs(ref).max())  # fp32 accumulation over K
    if epi == 0:
        D0 = inputs(94, (M, N), 1.0, mode=0) if acc else np.full((M, N), np.nan, dtype=np.float32)
        D = dev(D0, mode=0)
        gpt2_op_matmul_fp8_ex(0, D, qa, sa, qw, sw, accumulate=bool(acc), a_fmt=code[fa])
        torch.cuda.synchronize()
        want = ref + (D0.astype(np.float64) if acc else 0.0)
        assert_close(host(D), want, 1e-5, atol=atol + 1e-6, what="fp8 fp32 product")
    elif epi == 1:
        D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        D2 = torch.empty_like(D)
        gpt2_op_matmul_fp8_ex(1, D, qa, sa, qw, sw, D2=D2, bias=dev(bias), a_fmt=code[fa])
        torch.cuda.synchronize()
        u = data.round_to_bf16(ref.astype(np.float32)).astype(np.float64)
        # u itself may round the other way where the accumulation differs: compare
        # where the two agree on u's bf16 value (nearly everywhere), and the rest loosely
        assert_close(host(D2), R.gelu_forward(u), BF16_REL, atol=2e-3 * max(1.0, float(np.abs(u).max())),
                     what="gelu(u)")
        assert rel_l2(host(D), R.gelu_backward(u, np.ones_like(u))) < 1e-2
    else:
        aux = inputs(95, (M, N), 0.5)
        D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        gpt2_op_matmul_fp8_ex(2, D, qa, sa, qw, sw, aux=dev(aux), a_fmt=code[fa])
        torch.cuda.synchronize()
        want = data.round_to_bf16(ref.astype(np.float32)).astype(np.float64) * aux
        assert_close(host(D), want, 2 * BF16_REL, atol=atol * float(np.abs(aux).max()) + 1e-30,
                     atol_frac=1e-3, what="bf16(AB) * aux")


FP8_SMALL = dict(n_layer=2, n_embd=128, n_head=2, vocab=1000, vocab_padded=1024, max_T=128, max_B=3, mode=1)
MASKS = {"qkv": 1, "mlp": 2, "head": 4}


# Gradient bound of the FP8 step against the oracle's FP8 step (relative L2
# per tensor). The device quantizes its bf16 values, the oracle its exact
# ones; where the two straddle a rounding boundary they pick neighbouring
# codes. e5m2 codes are 2^-2 apart (relative) and the bf16 values about
# 2^-8 off, so about 1 gradient code in 64 differs by one spacing: a relative
# L2 difference of about sqrt(1/64) * 2^-2 = 3% for each quantized gradient
# (e4m3: 1 in 32 by 2^-3, about 2%), which then passes through the layers
# below. The bf16 step's 3e-2 is the size of one such term, so the FP8 step
# is held to 0.1; the loss (forward only) and the masters keep the bf16
# step's bounds.
FP8_GRAD_TOL = 0.1


@pytest.mark.parametrize("sel", [("qkv",), ("mlp",), ("head",), ("qkv", "mlp", "head")])
def test_fp8_step_small_parity(torch_cuda, sel):
    """Two steps with FP8 linears (L2 C128 H2, B=3, T=112: B*T a multiple of 16,
    ragged 128-row tiles) against the oracle's step with the same linears
    quantized: loss 2e-2, gradients FP8_GRAD_TOL relative L2, masters 1e-3."""
    torch = torch_cuda
    cfg = FP8_SMALL
    tok, tgt = data.batches("zipf", 3, 112, 2, 17, vocab=1000)
    model = make_model(cfg)
    model.set_fp8(sum(MASKS[k] for k in sel))
    losses, grads, masters = run_steps(torch, model, tok, tgt, 2, warmup=5)
    model.close()
    c = rcfg(cfg)
    params = R.init_params(c, 1234)
    state = None
    for s in range(2):
        loss, g, params, state = R.train_step(c, params, tok[s], tgt[s], state, 3e-4 * min(1.0, (s + 1) / 5),
                                              HP["beta1"], HP["beta2"], HP["eps"], HP["weight_decay"], s + 1,
                                              dtype=np.float64, fp8=sel)
        worst = check_step(cfg, losses[s], grads[s], masters[s], (loss, g, params), 2e-2, FP8_GRAD_TOL, 1e-3)
        print(f"fp8 {sel} step {s}: loss {losses[s]:.5f} vs {loss:.5f}, worst grad rel L2 {worst:.3e}")


FP8_WIDE = dict(n_layer=1, n_embd=1600, n_head=25, vocab=1000, vocab_padded=1024, max_T=128, max_B=3, mode=1)


def test_fp8_step_wide_rows_parity(torch_cuda):
    """One FP8 step (every linear of the selection) at the 1.5B model's width,
    C = 1600 (one block, H=25, B=3, T=112), where the LayerNorm forward and
    backward take their wide-row forms and give the quantizer the amax of what
    they write: against the oracle's FP8 step at the bounds above."""
    torch = torch_cuda
    cfg = FP8_WIDE
    tok, tgt = data.batches("zipf", 3, 112, 1, 23, vocab=1000)
    model = make_model(cfg)
    model.set_fp8(7)
    losses, grads, masters = run_steps(torch, model, tok, tgt, 1, warmup=5)
    model.close()
    c = rcfg(cfg)
    params = R.init_params(c, 1234)
    loss, g, params, _ = R.train_step(c, params, tok[0], tgt[0], None, 3e-4 * min(1.0, 1 / 5), HP["beta1"],
                                      HP["beta2"], HP["eps"], HP["weight_decay"], 1, dtype=np.float64,
                                      fp8=("qkv", "mlp", "head"))
    worst = check_step(cfg, losses[0], grads[0], masters[0], (loss, g, params), 2e-2, FP8_GRAD_TOL, 1e-3)
    print(f"fp8 C=1600: loss {losses[0]:.5f} vs {loss:.5f}, worst grad rel L2 {worst:.3e}")


def test_fp8_step_differs_from_bf16_by_quantization(torch_cuda):
    """The FP8 linears are really used: the gradients of the same step with
    and without them differ by a quantization-sized amount."""
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import TENSOR_GRAD
    cfg = FP8_SMALL
    tok, tgt = data.batches("zipf", 3, 112, 1, 19, vocab=1000)
    out = []
    for mask in (0, 7):
        model = make_model(cfg)
        model.set_fp8(mask)
        model.forward(torch.from_numpy(tok[0]).cuda(), torch.from_numpy(tgt[0]).cuda())
        model.backward()
        out.append(model.tensors(TENSOR_GRAD))
        model.close()
    for name in ("h0.qkv.w", "h1.fc.w", "h1.fcproj.w", "wte"):
        err = rel_l2(out[1][name], out[0][name])
        assert 1e-3 < err < 0.2, (name, err)


def test_fp8_graph_step_equals_separate_calls(torch_cuda):
    """gpt2_step (one CUDA graph) with every FP8 linear gives the bits of the
    separate forward, backward and AdamW calls."""
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import TENSOR_MASTER
    cfg = FP8_SMALL
    tok, tgt = data.batches("zipf", 3, 112, 3, 23, vocab=1000)
    res = []
    for graph in (False, True):
        model = make_model(cfg)
        model.set_fp8(7)
        losses = []
        for s in range(3):
            tk, tg = torch.from_numpy(tok[s]).cuda(), torch.from_numpy(tgt[s]).cuda()
            if graph:
                losses.append(model.step(tk, tg, 3e-4, t=s + 1, **HP))
            else:
                losses.append(model.forward(tk, tg))
                model.backward()
                model.adamw_step(3e-4, t=s + 1, **HP)
        res.append((losses, model.tensors(TENSOR_MASTER)))
        model.close()
    assert res[0][0] == res[1][0]
    for k in res[0][1]:
        assert np.array_equal(res[0][1][k], res[1][1][k]), k


def test_fp8_rejects_sizes_and_modes(torch_cuda):
    """B*T not a multiple of 16 is an argument error with FP8 linears; FP8
    needs the bf16 mode."""
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import GPT2Error
    model = make_model(FP8_SMALL)
    model.set_fp8(2)
    tok, tgt = data.batches("zipf", 3, 100, 1, 29, vocab=1000)
    with pytest.raises(GPT2Error):
        model.forward(torch.from_numpy(tok[0]).cuda(), torch.from_numpy(tgt[0]).cuda())
    model.set_fp8(0)
    model.forward(torch.from_numpy(tok[0]).cuda(), torch.from_numpy(tgt[0]).cuda())
    model.close()
    fp32 = dict(FP8_SMALL, mode=0)
    m2 = make_model(fp32)
    with pytest.raises(GPT2Error):
        m2.set_fp8(1)
    m2.close()
