"""Degenerate sizes: every op of gpt2_ops.h called with an empty input, and
attention over a single position.

Collected late on purpose (second to last, before the allocation-free entry
point's file test_zz_no_alloc.py), so that a run that stops at the first
failure has already run the per-kernel and whole-step tests.
"""
import numpy as np
import pytest

from tests._gpu_util import assert_close, dev, host, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    from step_gpt_train_gb300 import gpt2 as g
    g.load_library(build=True)
    torch.cuda.set_device(0)
    return torch


def test_empty_inputs(torch_cuda):
    """Zero-size calls launch nothing and succeed; where the result is an empty
    sum it is written as zero (the bias gradient and the LayerNorm dgamma,
    dbeta over no rows, the position-embedding gradient of an empty batch),
    and nothing else is touched. Every pointer is a valid, aligned buffer (an
    empty torch tensor has none)."""
    torch = torch_cuda
    from step_gpt_train_gb300 import gpt2 as g
    lib = g.load_library()
    s = torch.cuda.current_stream().cuda_stream
    bf16 = 1  # the bf16 mode / dtype code
    C = 64

    def buf(n=1 << 16, dtype=torch.float32, fill=7.0):
        return torch.full((n,), fill, dtype=dtype, device="cuda")

    p = lambda t: t.data_ptr()
    src, out, f = buf(dtype=torch.bfloat16), buf(dtype=torch.bfloat16), buf()
    tok = torch.zeros(1 << 12, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    scratch = buf(1 << 20)
    nscr = scratch.numel() * 4
    out0 = out.clone()
    calls = {
        "matmul M=0": lib.gpt2_op_matmul(bf16, p(out), 0, p(src), 0, p(src), 0, None, 0, 64, 64, p(scratch), nscr,
                                         p(status), s),
        "matmul N=0": lib.gpt2_op_matmul(bf16, p(out), 0, p(src), 0, p(src), 0, None, 64, 0, 64, p(scratch), nscr,
                                         p(status), s),
        "gelu fwd": lib.gpt2_op_gelu_forward(bf16, p(out), p(src), 0, s),
        "gelu bwd": lib.gpt2_op_gelu_backward(bf16, p(out), p(src), p(src), 0, s),
        "residual fwd": lib.gpt2_op_residual_forward(bf16, p(out), p(src), p(src), 0, s),
        "residual bwd": lib.gpt2_op_residual_backward(bf16, p(out), p(src), 0, s),
        "layernorm fwd": lib.gpt2_op_layernorm_forward(bf16, p(out), p(f), p(f), p(src), p(src), p(src), 0, C, s),
        "attention fwd": lib.gpt2_op_attention_forward(bf16, p(out), p(f), p(src), 0, 64, 128, 2, s),
        "attention bwd": lib.gpt2_op_attention_backward(bf16, p(out), p(src), p(src), p(src), p(f), 0, 64, 128, 2,
                                                        p(scratch), nscr, s),
        "classifier": lib.gpt2_op_classifier(bf16, p(out), p(f), p(tok), 0, 1000, 1024, 1.0, p(status), s),
        "encoder fwd": lib.gpt2_op_encoder_forward(bf16, p(out), p(tok), p(src), p(src), 0, 8, C, 100, p(status), s),
        "adamw": lib.gpt2_op_adamw(p(f), p(out), p(f), p(f), p(f), 0, 1e-3, 0.9, 0.95, 1e-8, 0.1, 1, s),
        "quantize fp8": lib.gpt2_op_quantize_fp8(p(out), p(f), p(src), 0, 0, p(scratch), nscr, s),
        "matmul fp8": lib.gpt2_op_matmul_fp8(p(out), p(src), 0, p(f), p(src), 0, p(f), None, 0, 16, 32, p(status), s),
    }
    torch.cuda.synchronize()
    assert all(v == 0 for v in calls.values()), {k: v for k, v in calls.items() if v != 0}
    assert torch.equal(out, out0) and bool((f == 7.0).all()) and int(status.item()) == 0
    # empty sums are zero
    dbias = buf(C)
    assert lib.gpt2_op_bias_backward(bf16, p(dbias), p(src), 0, C, p(scratch), nscr, s) == 0
    dgamma, dbeta = buf(C), buf(C)
    need = lib.gpt2_op_layernorm_backward_scratch(0, C)
    assert 0 < need <= nscr
    assert lib.gpt2_op_layernorm_backward(bf16, p(out), p(dgamma), p(dbeta), p(src), p(src), p(src), p(f), p(f), 0, C,
                                          p(scratch), nscr, s) == 0
    dwte, dwpe = buf(128 * C), buf(16 * C)
    assert lib.gpt2_op_encoder_backward(bf16, p(dwte), p(dwpe), p(src), p(tok), 0, 8, C, 128, p(scratch), nscr,
                                        s) == 0
    torch.cuda.synchronize()
    assert bool((dbias == 0).all()) and bool((dgamma == 0).all()) and bool((dbeta == 0).all())
    assert bool((dwpe[:8 * C] == 0).all()) and bool((dwpe[8 * C:] == 7.0).all())  # rows t >= T untouched
    assert bool((dwte == 7.0).all())  # accumulated into: an empty batch adds nothing


@pytest.mark.parametrize("mode", [1, 0])
def test_attention_single_position(torch_cuda, mode):
    """T = 1: the one query sees only its own key, so P = 1 and, in closed
    form, o = v, lse = q.k / sqrt(hd), dV = dO, and dS = P (dP - D) = 0 because
    D = dO.o = dO.v = dP, so dQ = dK = 0 up to the rounding of dP and D."""
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import gpt2_op_attention_backward, gpt2_op_attention_forward
    B, T, H = 3, 1, 2
    hd = 64 if mode == 1 else 16
    C = H * hd
    qkv = inputs(52, (B, T, 3 * C), 1.0, mode)
    dout = inputs(53, (B, T, C), 1.0, mode)
    dq = dev(qkv, mode)
    o = torch.full((B, T, C), float("nan"), dtype=dq.dtype, device="cuda")
    lse = torch.full((B, H, T), float("nan"), device="cuda")
    gpt2_op_attention_forward(o, lse, dq, B, T, H)
    dqkv = torch.full_like(dq, float("nan"))
    gpt2_op_attention_backward(dqkv, dev(dout, mode), dq, o, lse, B, T, H)
    torch.cuda.synchronize()
    q, k, v = (qkv[..., i * C:(i + 1) * C].astype(np.float64) for i in range(3))
    tol = 2.0 ** -8 if mode == 1 else 1e-6
    assert_close(host(o), v, tol, atol=1e-30, what="o = v")
    qk = (q.reshape(B, H, hd) * k.reshape(B, H, hd)).sum(-1) / np.sqrt(hd)
    assert_close(host(lse).reshape(B, H), qk, 1e-5, atol=1e-4, what="lse = q.k/sqrt(hd)")
    g = host(dqkv)
    assert_close(g[..., 2 * C:], dout.astype(np.float64), tol, atol=1e-30, what="dV = dO")
    assert np.all(np.isfinite(g))
    small = 1e-3 if mode == 1 else 1e-4
    assert np.abs(g[..., :2 * C]).max() < small, np.abs(g[..., :2 * C]).max()  # dQ, dK
