"""Helpers for the GPU tests: seeded inputs, device transfer, comparisons."""
import numpy as np

from step_gpt_train_gb300 import data


def torch_dtype(mode):
    import torch
    return torch.bfloat16 if mode == 1 else torch.float32


def inputs(seed, shape, std=1.0, mode=1):
    """Seeded test values; exactly representable in bf16 when mode == 1."""
    x = data.normal(seed, shape, std, dtype=np.float32)
    return data.round_to_bf16(x) if mode == 1 else x


def dev(x, mode=1):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x))
    if t.dtype in (torch.float32, torch.float64):
        t = t.to(torch_dtype(mode))
    return t.cuda()


def dev_f32(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def host(t):
    import torch
    return t.detach().to(torch.float64).cpu().numpy()


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (den if den > 0 else 1.0))


def assert_close(got, ref, rtol, atol_frac=0.0, atol=0.0, what=""):
    """|got - ref| <= rtol |ref| + atol + atol_frac * rms(ref), elementwise."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    bound = rtol * np.abs(ref) + atol + atol_frac * rms
    err = np.abs(got - ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} out of tolerance; worst at {i}: "
                             f"got {got[i]!r} ref {ref[i]!r} (bound {bound[i]:.3g})")


BF16_REL = 2.0 ** -8  # one bf16 output rounding (2^-9) plus fp32 arithmetic, with margin
