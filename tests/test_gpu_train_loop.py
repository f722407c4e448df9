"""The training loop around the step through the C ABI: gradient accumulation
over micro-batches, the global gradient norm, and AdamW with a gradient scale,
global-norm clipping and the weight-decay mask, against the oracle."""
import numpy as np
import pytest

from oracle import gpt2_ref as R
from step_gpt_train_gb300 import data
from tests._gpu_util import rel_l2
from tests.test_gpu_step import HP, SMALL_BF16, TINY, make_model, rcfg

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    from step_gpt_train_gb300 import gpt2 as g
    g.load_library(build=True)
    torch.cuda.set_device(0)
    return torch


def oracle_grads(cfg, params, tok, tgt):
    return R.backward(rcfg(cfg), R.forward(rcfg(cfg), params, tok, tgt)[1])


@pytest.mark.parametrize("cfg, tol", [(TINY, 1e-4), (SMALL_BF16, 3e-2)])
def test_grad_accumulation_matches_oracle_sum(torch_cuda, cfg, tol):
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import TENSOR_GRAD
    B, T = (4, 64) if cfg is TINY else (3, 100)
    kind = "uniform" if cfg is TINY else "zipf"
    tok, tgt = data.batches(kind, B, T, 2, 99, vocab=cfg["vocab"])
    model = make_model(cfg)
    model.zero_grad()
    model.set_grad_accumulation(True)
    for s in range(2):
        model.forward(torch.from_numpy(tok[s]).cuda(), torch.from_numpy(tgt[s]).cuda())
        model.backward()
    got = model.tensors(TENSOR_GRAD)
    params = R.init_params(rcfg(cfg), 1234)
    g1, g2 = oracle_grads(cfg, params, tok[0], tgt[0]), oracle_grads(cfg, params, tok[1], tgt[1])
    worst = max(rel_l2(got[k], g1[k] + g2[k]) for k in g1 if np.linalg.norm(g1[k] + g2[k]) > 0)
    assert worst <= tol, worst
    assert np.all(got["wte"][cfg["vocab"]:] == 0)
    # back to overwriting: one more backward holds only its own batch's gradient
    model.set_grad_accumulation(False)
    model.forward(torch.from_numpy(tok[1]).cuda(), torch.from_numpy(tgt[1]).cuda())
    model.backward()
    got = model.tensors(TENSOR_GRAD)
    worst = max(rel_l2(got[k], g2[k]) for k in g2 if np.linalg.norm(g2[k]) > 0)
    assert worst <= tol, worst
    model.close()


def test_grad_norm_and_clipped_masked_scaled_adamw(torch_cuda):
    """The update from the library's own gradients and masters, against the oracle's
    AdamW on those same values (float64), with clipping active."""
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import TENSOR_GRAD, TENSOR_MASTER
    tok, tgt = data.batches("uniform", 4, 64, 1, 5, vocab=512)
    model = make_model(TINY)
    model.forward(torch.from_numpy(tok[0]).cuda(), torch.from_numpy(tgt[0]).cuda())
    model.backward()
    grads = model.tensors(TENSOR_GRAD)
    masters = model.tensors(TENSOR_MASTER)
    norm = R.global_grad_norm(grads)
    assert model.grad_norm() == pytest.approx(norm, rel=1e-5)
    scale, lr = 0.5, 1e-3
    max_norm = 0.25 * norm * scale  # clipping active
    clip = R.clip_factor(norm, max_norm, scale)
    assert clip < 1.0
    model.adamw_step(lr, t=1, grad_scale=scale, max_grad_norm=max_norm, decay_mask=True, **HP)
    got = model.tensors(TENSOR_MASTER)
    for k in masters:
        th = masters[k].astype(np.float64)
        wd = HP["weight_decay"] if R.decays(k, th) else 0.0
        ref = R.adamw_update_ex(th, grads[k].astype(np.float64), np.zeros_like(th), np.zeros_like(th), lr,
                                HP["beta1"], HP["beta2"], HP["eps"], wd, 1, scale, clip)[0]
        assert rel_l2(got[k], ref) <= 1e-6, k
    model.close()


@pytest.mark.parametrize("cfg", [TINY, SMALL_BF16])
def test_sharded_adamw_equals_full_step(torch_cuda, cfg):
    """ZeRO-1 style update: AdamW over shards that tile the flat parameter layout
    gives the full step's masters, moments and compute copy bit for bit (the
    update is elementwise), and the shards' gradient sums of squares add up to
    the squared global norm."""
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import TENSOR_ADAM_M, TENSOR_ADAM_V, TENSOR_GRAD, TENSOR_MASTER, TENSOR_PARAM
    B, T = (4, 64) if cfg is TINY else (3, 100)
    tok, tgt = data.batches("uniform", B, T, 2, 31, vocab=cfg["vocab"])
    models = [make_model(cfg), make_model(cfg)]
    for m in models:
        m.forward(torch.from_numpy(tok[0]).cuda(), torch.from_numpy(tgt[0]).cuda())
        m.backward()
    full, sharded = models
    n = sharded.flat_params()
    cut1, cut2 = 2048 * (n // (3 * 2048)), 2048 * (2 * n // (3 * 2048))
    bounds = [(0, cut1), (cut1, cut2 - cut1), (cut2, n - cut2)]
    assert all(c > 0 for _, c in bounds)
    sumsq = sum(sharded.grad_sumsq_range(b, c) for b, c in bounds)
    assert sumsq == pytest.approx(R.global_grad_norm(sharded.tensors(TENSOR_GRAD)) ** 2, rel=1e-5)
    for t in (1, 2):
        lr = 1e-3 * t
        full.adamw_step(lr, t=t, grad_scale=0.5, decay_mask=True, **HP)
        for b, c in reversed(bounds):  # any order: the shards are disjoint
            sharded.adamw_step_shard(b, c, lr, t=t, grad_scale=0.5, decay_mask=True, **HP)
        if t == 1:
            for m in models:
                m.forward(torch.from_numpy(tok[1]).cuda(), torch.from_numpy(tgt[1]).cuda())
                m.backward()
    kinds = (TENSOR_MASTER, TENSOR_ADAM_M, TENSOR_ADAM_V) + ((TENSOR_PARAM,) if cfg["mode"] == 1 else ())
    for kind in kinds:
        a, b = full.tensors(kind), sharded.tensors(kind)
        for k in a:
            assert np.array_equal(a[k], b[k]), (kind, k)
    for m in models:
        m.close()


def test_shard_arguments_checked(torch_cuda):
    from step_gpt_train_gb300.gpt2 import GPT2Error
    torch = torch_cuda
    tok, tgt = data.batches("uniform", 4, 64, 1, 5, vocab=512)
    model = make_model(TINY)
    with pytest.raises(GPT2Error):  # before any backward
        model.adamw_step_shard(0, 2048, 1e-3)
    model.forward(torch.from_numpy(tok[0]).cuda(), torch.from_numpy(tgt[0]).cuda())
    model.backward()
    n = model.flat_params()
    for begin, count in ((1024, 2048), (0, 6), (0, n + 4), (-2048, 2048)):
        with pytest.raises(GPT2Error):
            model.adamw_step_shard(begin, count, 1e-3)
    model.adamw_step_shard(0, n, 1e-3)
    model.close()


@pytest.mark.parametrize("cfg", [TINY, SMALL_BF16])
def test_step_graph_equals_separate_calls(torch_cuda, cfg):
    """gpt2_step (forward, backward, clip and AdamW replayed as one captured CUDA
    graph) gives the losses, masters and moments of the separate calls bit for
    bit, with the learning rate changing every step and a change of options
    (which captures a second graph) on the way."""
    torch = torch_cuda
    from step_gpt_train_gb300.gpt2 import TENSOR_ADAM_M, TENSOR_ADAM_V, TENSOR_MASTER
    B, T = (4, 64) if cfg is TINY else (3, 100)
    tok, tgt = data.batches("uniform", B, T, 6, 41, vocab=cfg["vocab"])
    sep, graph = make_model(cfg), make_model(cfg)
    for s in range(6):
        # steps 0-2: no clip, no mask (eager, capture, replay); 3-5: clip and mask (a new graph)
        opts = dict(grad_scale=0.5, max_grad_norm=0.05 if s >= 3 else 0.0, decay_mask=s >= 3, **HP)
        lr = 1e-3 * (1 + s)
        tt, gg = torch.from_numpy(tok[s]).cuda(), torch.from_numpy(tgt[s]).cuda()
        la = sep.forward(tt, gg)
        sep.backward()
        sep.adamw_step(lr, t=s + 1, **opts)
        lb = graph.step(tt, gg, lr, t=s + 1, **opts)
        assert la == lb, (s, la, lb)
    for kind in (TENSOR_MASTER, TENSOR_ADAM_M, TENSOR_ADAM_V):
        a, b = sep.tensors(kind), graph.tensors(kind)
        for k in a:
            assert np.array_equal(a[k], b[k]), (kind, k)
    sep.close()
    graph.close()
