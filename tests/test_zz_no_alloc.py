"""The allocation-free bias-gradient entry point against the regular one.

Some callers cannot lend this library scratch memory (their device memory
belongs to another runtime's allocator, or they must not call cudaMalloc).
gpt2_op_bias_backward_noalloc serves them with a fixed scratch array inside
the library. This file is collected last on purpose (its name sorts after
every other test file's), so that a run that stops at the first failure has
already run every other test. Each test passes both in a fresh process and
after the rest of the suite.
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


@pytest.mark.parametrize("mode", [1, 0])
def test_noalloc_matches_regular_entry_point_twice(torch_cuda, mode):
    torch = torch_cuda
    from step_gpt_train_gb300 import gpt2 as g
    # two calls in a row, different shapes: the shared scratch keeps the first
    # call's partials, which the second must not pick up
    # the third fills the fixed scratch exactly: ceil(32768/128) * 4096 = 1,048,576 partials
    for seed, (N, C) in ((200, (32768, 3072)), (201, (1000, 200)), (202, (32768, 4096))):
        dy = dev(inputs(seed, (N, C), 1.0, mode), mode)
        want = torch.full((C,), float("nan"), device="cuda")
        got = torch.full((C,), float("nan"), device="cuda")
        g.gpt2_op_bias_backward(want, dy)
        g.gpt2_op_bias_backward_noalloc(got, dy)
        torch.cuda.synchronize()
        assert np.all(np.isfinite(host(got)))
        assert_close(host(got), host(want), 1e-5, atol=1e-4, what=f"noalloc bias grad {N}x{C}")


def test_noalloc_many_row_chunks(torch_cuda):
    """C = 8 with 8.4M rows: 65,600 row chunks of 128, more than one launch's
    65,535 grid rows (within the fixed scratch: 524,800 partials)."""
    torch = torch_cuda
    from step_gpt_train_gb300 import gpt2 as g
    N, C = 65600 * 128, 8
    dy = dev(inputs(203, (N, C), 1.0, 1), 1)
    want = torch.full((C,), float("nan"), device="cuda")
    got = torch.full((C,), float("nan"), device="cuda")
    g.gpt2_op_bias_backward(want, dy)
    g.gpt2_op_bias_backward_noalloc(got, dy)
    torch.cuda.synchronize()
    ref = host(dy).sum(0)
    assert_close(host(got), host(want), 1e-5, atol=1e-4, what="noalloc bias grad, many chunks")
    assert_close(host(got), ref, 1e-5, atol=2e-2, what="bias grad, many chunks, against float64")


def test_noalloc_rejects_sizes_beyond_its_scratch(torch_cuda):
    torch = torch_cuda
    from step_gpt_train_gb300 import gpt2 as g
    N, C = 32768, 8192  # 256 chunks x 8192 columns > 1,048,576 partials
    dy = torch.zeros(8, dtype=torch.bfloat16, device="cuda")  # never read: rejected first
    out = torch.zeros(C, device="cuda")
    status = g.load_library().gpt2_op_bias_backward_noalloc(1, out.data_ptr(), dy.data_ptr(), N, C,
                                                            torch.cuda.current_stream().cuda_stream)
    assert status == -7  # GPT2_ERR_WORKSPACE
