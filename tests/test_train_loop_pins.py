"""Pins of the oracle's training-loop additions (CPU): AdamW with a gradient
scale, global-norm clipping and a weight-decay mask against torch's
clip_grad_norm_ and AdamW with parameter groups; gradient accumulation against
the full-batch gradient; the cosine learning-rate schedule against its closed
form (and the library's host implementation against the oracle's)."""
import math

import numpy as np
import pytest

from oracle import gpt2_ref as R


def test_clipped_masked_scaled_adamw_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    params = {"w": rng.normal(size=(6, 5)), "b": rng.normal(size=(6,)), "ln": rng.normal(size=(5,)),
              "e": rng.normal(size=(7, 5))}
    grads = {k: rng.normal(size=v.shape) * 3.0 for k, v in params.items()}
    m0 = {k: rng.normal(size=v.shape) * 0.1 for k, v in params.items()}
    v0 = {k: rng.random(size=v.shape) * 0.1 for k, v in params.items()}
    lr, b1, b2, eps, wd, t, scale, max_norm = 1e-2, 0.9, 0.95, 1e-8, 0.1, 3, 0.5, 1.0
    norm = R.global_grad_norm(grads)
    clip = R.clip_factor(norm, max_norm, scale)
    assert clip < 1.0  # the case exercises clipping
    ours = {k: R.adamw_update_ex(params[k], grads[k], m0[k], v0[k], lr, b1, b2, eps,
                                 wd if R.decays(k, params[k]) else 0.0, t, scale, clip)[0] for k in params}
    tp = {k: torch.tensor(v, dtype=torch.float64, requires_grad=True) for k, v in params.items()}
    for k, p in tp.items():
        p.grad = torch.tensor(grads[k] * scale, dtype=torch.float64)
    torch.nn.utils.clip_grad_norm_(list(tp.values()), max_norm)
    opt = torch.optim.AdamW([{"params": [tp[k] for k in tp if params[k].ndim == 2], "weight_decay": wd},
                             {"params": [tp[k] for k in tp if params[k].ndim != 2], "weight_decay": 0.0}],
                            lr=lr, betas=(b1, b2), eps=eps, foreach=False)
    for k, p in tp.items():  # moments after t - 1 earlier steps
        opt.state[p] = {"step": torch.tensor(float(t - 1)), "exp_avg": torch.tensor(m0[k]),
                        "exp_avg_sq": torch.tensor(v0[k])}
    opt.step()
    for k in params:
        np.testing.assert_allclose(ours[k], tp[k].detach().numpy(), rtol=1e-12, atol=1e-14, err_msg=k)


def test_no_clip_and_no_scale_is_plain_adamw():
    rng = np.random.default_rng(6)
    th, g = rng.normal(size=10), rng.normal(size=10)
    a = R.adamw_update(th, g, np.zeros(10), np.zeros(10), 1e-3, 0.9, 0.95, 1e-8, 0.1, 1)
    b = R.adamw_update_ex(th, g, np.zeros(10), np.zeros(10), 1e-3, 0.9, 0.95, 1e-8, 0.1, 1, 1.0,
                          R.clip_factor(R.global_grad_norm({"g": g}), 0.0))
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_gradient_accumulation_is_the_sum_over_micro_batches():
    """Each micro-batch's gradient is that of its own mean loss, so two halves of a
    batch sum to twice the full batch's gradient."""
    cfg = R.Config(1, 16, 2, 32, 32, 8)
    params = R.init_params(cfg, 11)
    rng = np.random.default_rng(3)
    tok = rng.integers(0, 32, size=(2, 8))
    tgt = rng.integers(0, 32, size=(2, 8))
    full = R.backward(cfg, R.forward(cfg, params, tok, tgt)[1])
    h1 = R.backward(cfg, R.forward(cfg, params, tok[:1], tgt[:1])[1])
    h2 = R.backward(cfg, R.forward(cfg, params, tok[1:], tgt[1:])[1])
    for k in full:
        np.testing.assert_allclose(h1[k] + h2[k], 2.0 * full[k], rtol=1e-9, atol=1e-14, err_msg=k)


def test_lr_cosine_closed_form():
    lr_max, lr_min, warm, total = 6e-4, 6e-5, 10, 110
    assert R.lr_cosine(1, warm, total, lr_max, lr_min) == pytest.approx(lr_max / warm)
    assert R.lr_cosine(warm, warm, total, lr_max, lr_min) == pytest.approx(lr_max)
    assert R.lr_cosine(60, warm, total, lr_max, lr_min) == pytest.approx((lr_max + lr_min) / 2)  # half way
    assert R.lr_cosine(total, warm, total, lr_max, lr_min) == lr_min
    assert R.lr_cosine(total + 50, warm, total, lr_max, lr_min) == lr_min
    vals = [R.lr_cosine(t, warm, total, lr_max, lr_min) for t in range(warm, total + 1)]
    assert all(a >= b for a, b in zip(vals, vals[1:]))


def test_library_lr_cosine_equals_oracle():
    from step_gpt_train_gb300.gpt2 import gpt2_lr_cosine
    for t in (0, 1, 5, 10, 11, 37, 60, 109, 110, 500):
        for warm, total in ((10, 110), (0, 100), (20, 20)):
            ref = R.lr_cosine(t, warm, total, 6e-4, 6e-5)
            assert gpt2_lr_cosine(t, warm, total, 6e-4, 6e-5) == pytest.approx(ref, rel=1e-6, abs=1e-12), (t, warm)
