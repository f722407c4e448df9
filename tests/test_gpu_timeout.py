"""The failure path of the bounded device waits, made to run out on purpose
without faulting, trapping or hanging the GPU.

A test switch (gpt2_debug_stall_matmul) makes the tensor-core GEMM's MMA warp
wait, before its first product, on a barrier that nothing arrives at, and
gpt2_debug_set_wait_limit shortens every wait's bound to about a millisecond.
The kernel must then set the timeout bit of its status word, stop its other
warps, wait for its own copies in flight, free its tensor memory and return:
the same call right after, with the switch off, must succeed and be correct
(a kernel that had kept its tensor memory would leave the next one's
allocation waiting), and the model's calls must report GPT2_ERR_TIMEOUT.
Every wait stays bounded throughout; the switch and the bound are restored
in a finally block.
"""
import math

import numpy as np
import pytest

from step_gpt_train_gb300 import data
from tests._gpu_util import assert_close, dev, host, inputs

pytestmark = pytest.mark.gpu

SHORT_WAIT_CYCLES = 2_000_000  # about 1 ms at 2 GHz


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    from step_gpt_train_gb300 import gpt2 as g
    g.load_library(build=True)
    torch.cuda.set_device(0)
    return torch


def _stalled(lib, on):
    from step_gpt_train_gb300.gpt2 import check
    check(lib.gpt2_debug_set_wait_limit(SHORT_WAIT_CYCLES if on else 0), "gpt2_debug_set_wait_limit")
    check(lib.gpt2_debug_stall_matmul(1 if on else 0), "gpt2_debug_stall_matmul")


def test_matmul_wait_times_out_and_recovers(torch_cuda):
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import gpt2_op_matmul, load_library
    lib = load_library()
    M, N, K = 300, 392, 1000  # several k-blocks: the producer has copies in flight when the MMA warp gives up
    A = inputs(1, (M * K,), 1.0, 1)
    B = inputs(2, (N * K,), 1.0, 1)
    dA, dB = dev(A, 1), dev(B, 1)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    D = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
    try:
        _stalled(lib, True)
        gpt2_op_matmul(D, dA, 0, dB, 0, M, N, K, status=status)
        torch.cuda.synchronize()
    finally:
        _stalled(lib, False)
    assert int(status.item()) & 2, int(status.item())  # the timeout bit
    # the context is usable and the tensor memory was freed: the same GEMM now runs and is right
    status.zero_()
    gpt2_op_matmul(D, dA, 0, dB, 0, M, N, K, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = A.reshape(M, K).astype(np.float64) @ B.reshape(N, K).astype(np.float64).T
    assert_close(host(D), ref, 2.0 ** -8, atol=1e-3, what="D after recovery")


def test_model_reports_timeout_then_steps(torch_cuda):
    torch = torch_cuda
    from step_gpt_train_gb300 import gpt2 as g
    cfg = dict(n_layer=2, n_embd=128, n_head=2, vocab=1000, vocab_padded=1024, max_T=128, max_B=3, mode=1)
    model = g.GPT2(cfg, 1234)
    lib = g.load_library()
    tok, tgt = data.batches("zipf", 3, 100, 1, 9, vocab=1000)
    dt, dg = torch.from_numpy(tok[0]).cuda(), torch.from_numpy(tgt[0]).cuda()
    try:
        _stalled(lib, True)
        with pytest.raises(g.GPT2Error) as e:
            model.forward(dt, dg)
        torch.cuda.synchronize()
    finally:
        _stalled(lib, False)
    assert e.value.status == -5  # GPT2_ERR_TIMEOUT
    with pytest.raises(g.GPT2Error) as e:
        model.backward()  # the failed forward does not enable a backward
    assert e.value.status == -2
    loss = model.forward(dt, dg)
    assert math.isfinite(loss) and abs(loss - math.log(1000)) < 0.5
    model.backward()
    model.adamw_step(1e-4, t=1)
    model.close()
