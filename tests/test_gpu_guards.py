"""Out-of-bounds write guards. Every output buffer of the ops below sits
between two 4 KB guard bands filled with a byte pattern (compute-sanitizer is
not available on these GPUs); after the op, the bands must be intact. The
shapes are ragged (not multiples of the tile, row-block or vector widths), so
the kernels' edge handling is what is exercised."""
import math

import pytest

from step_gpt_train_gb300 import data
from tests._gpu_util import dev, inputs

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes on each side
PATTERN = 0xA5


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    from step_gpt_train_gb300 import gpt2 as g
    g.load_library(build=True)
    torch.cuda.set_device(0)
    return torch


class Guarded:
    """A device buffer of `shape` between two guard bands of PATTERN bytes."""

    def __init__(self, torch, shape, dtype, fill=None):
        self.torch = torch
        n = math.prod(shape)
        self.elem = torch.empty(0, dtype=dtype).element_size()
        self.g = GUARD // self.elem
        self.n = n
        self.buf = torch.empty(2 * self.g + n, dtype=dtype, device="cuda")
        self.buf.view(torch.uint8).fill_(PATTERN)
        self.t = self.buf[self.g:self.g + n].view(*shape)
        if fill is not None:
            self.t.copy_(fill)

    def intact(self):
        b = self.buf.view(self.torch.uint8)
        head, tail = b[:self.g * self.elem], b[(self.g + self.n) * self.elem:]
        return bool((head == PATTERN).all()) and bool((tail == PATTERN).all())


def test_guards_matmul(torch_cuda):
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import gpt2_op_matmul
    # linear forward, ragged M and N, bf16 out with bias
    M, N, K = 300, 392, 200
    D = Guarded(torch, (M, N), torch.bfloat16)
    gpt2_op_matmul(D.t, dev(inputs(1, (M, K))), 0, dev(inputs(2, (N, K))), 0, M, N, K, bias=dev(inputs(3, (N,))))
    # weight gradient: both operands MN-major, fp32 out, long K (split-K partials and their reduce)
    M, N, K = 392, 200, 8192
    W = Guarded(torch, (M, N), torch.float32)
    gpt2_op_matmul(W.t, dev(inputs(4, (K, M))), 1, dev(inputs(5, (K, N))), 1, M, N, K)
    torch.cuda.synchronize()
    assert D.intact() and W.intact()


def test_guards_fp8(torch_cuda):
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import FP8_E5M2, gpt2_op_matmul_fp8, gpt2_op_quantize_fp8
    M, N, K = 300, 200, 272
    qa, qw = Guarded(torch, (M, K), torch.uint8), Guarded(torch, (N, K), torch.uint8)
    sa, sw = Guarded(torch, (2,), torch.float32), Guarded(torch, (2,), torch.float32)
    gpt2_op_quantize_fp8(qa.t, sa.t, dev(inputs(6, (M, K))))
    gpt2_op_quantize_fp8(qw.t, sw.t, dev(inputs(7, (N, K), 0.02)))
    D = Guarded(torch, (M, N), torch.bfloat16)
    gpt2_op_matmul_fp8(D.t, qa.t, sa.t, qw.t, sw.t, bias=dev(inputs(8, (N,))))
    q_odd = Guarded(torch, (8 * 1001 + 3,), torch.uint8)  # the scalar tail of the quantizer
    gpt2_op_quantize_fp8(q_odd.t, sa.t, dev(inputs(9, (8 * 1001 + 3,))))
    # e5m2: the other quantizer instantiation, and an e5m2 x e4m3 product
    qg, sg = Guarded(torch, (M, K), torch.uint8), Guarded(torch, (2,), torch.float32)
    gpt2_op_quantize_fp8(qg.t, sg.t, dev(inputs(22, (M, K))), FP8_E5M2)
    D2 = Guarded(torch, (M, N), torch.bfloat16)
    gpt2_op_matmul_fp8(D2.t, qg.t, sg.t, qw.t, sw.t, a_fmt=FP8_E5M2)
    torch.cuda.synchronize()
    assert all(x.intact() for x in (qa, qw, sa, sw, D, q_odd, qg, sg, D2))


def test_guards_layernorm(torch_cuda):
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import gpt2_op_layernorm_backward, gpt2_op_layernorm_forward
    N, C = 37, 1600
    x, gamma, beta = dev(inputs(10, (N, C))), dev(inputs(11, (C,))), dev(inputs(12, (C,)))
    y = Guarded(torch, (N, C), torch.bfloat16)
    mean, rstd = Guarded(torch, (N,), torch.float32), Guarded(torch, (N,), torch.float32)
    gpt2_op_layernorm_forward(y.t, mean.t, rstd.t, x, gamma, beta)
    dx = Guarded(torch, (N, C), torch.bfloat16)
    dg, db = Guarded(torch, (C,), torch.float32), Guarded(torch, (C,), torch.float32)
    gpt2_op_layernorm_backward(dx.t, dg.t, db.t, dev(inputs(13, (N, C))), x, gamma, mean.t, rstd.t)
    torch.cuda.synchronize()
    assert all(v.intact() for v in (y, mean, rstd, dx, dg, db))


def test_guards_attention(torch_cuda):
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import gpt2_op_attention_backward, gpt2_op_attention_forward
    B, T, H = 2, 200, 2  # T not a multiple of the 128-row tiles
    C = 64 * H
    qkv = dev(inputs(14, (B, T, 3 * C)))
    o = Guarded(torch, (B, T, C), torch.bfloat16)
    lse = Guarded(torch, (B, H, T), torch.float32)
    gpt2_op_attention_forward(o.t, lse.t, qkv, B, T, H)
    dqkv = Guarded(torch, (B, T, 3 * C), torch.bfloat16)
    gpt2_op_attention_backward(dqkv.t, dev(inputs(15, (B, T, C))), qkv, o.t, lse.t, B, T, H)
    torch.cuda.synchronize()
    assert o.intact() and lse.intact() and dqkv.intact()


def test_guards_classifier_encoder_bias(torch_cuda):
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import gpt2_op_bias_backward, gpt2_op_classifier, gpt2_op_encoder_forward
    N, V, Vp = 37, 1000, 1024
    z = Guarded(torch, (N, Vp), torch.bfloat16, fill=dev(inputs(16, (N, Vp), 2.0)))
    losses = Guarded(torch, (N,), torch.float32)
    tgt = dev(data.token_stream("uniform", N, 17, vocab=V))
    gpt2_op_classifier(z.t, losses.t, tgt, V, 1.0 / N)
    B, T, C, Vw = 3, 50, 1600, 1000
    x0 = Guarded(torch, (B, T, C), torch.bfloat16)
    tokens = dev(data.token_stream("uniform", B * T, 18, vocab=Vw).reshape(B, T))
    gpt2_op_encoder_forward(x0.t, tokens, dev(inputs(19, (Vw, C))), dev(inputs(20, (T, C))), Vw)
    dbias = Guarded(torch, (392,), torch.float32)
    gpt2_op_bias_backward(dbias.t, dev(inputs(21, (300, 392))))
    torch.cuda.synchronize()
    assert all(v.intact() for v in (z, losses, x0, dbias))
