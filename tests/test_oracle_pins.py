"""Pins for the CPU oracle (no GPU).

The oracle is checked against facts that do not come from itself: torch
library routines and autograd, central finite differences of its own forward,
closed forms and exact special cases, and published constants. The pages
print no worked example of the step, so these are the pins.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import gpt2_ref as R
from step_gpt_train_gb300 import data
from tests._torch_gpt2 import torch_loss_and_grads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

MICRO = R.Config(n_layer=1, n_embd=16, n_head=2, vocab=32, vocab_padded=40, max_T=8)
TINY = R.Config(n_layer=2, n_embd=64, n_head=4, vocab=512, vocab_padded=512, max_T=64)


def random_params(cfg, seed, std=0.3):
    """Random parameters with O(1) scale, so that every term of the step matters."""
    params = {}
    for i, (name, shape, how) in enumerate(R.param_specs(cfg)):
        a = data.normal(seed * 1000 + i, shape, std, dtype=np.float64)
        if how == "one":
            a = 1.0 + a
        if name == "wte":
            a[cfg.vocab:] = 0.0
        params[name] = a
    return params


def rel_l2(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (den if den > 0 else 1.0)


# ---------------------------------------------------------------- generators

def test_splitmix64_published_vector():
    g = json.load(open(os.path.join(GOLDEN, "splitmix64.json")))
    want = [int(x) for x in g["first_outputs"]]
    got = [int(x) for x in data.splitmix64_stream(g["seed"], 0, len(want))]
    assert got == want
    # the oracle's own copy of the generator (same definition, separate code)
    s = np.array([g["seed"]], dtype=np.uint64)
    got2 = []
    for _ in want:
        s, z = R._splitmix_next(s)
        got2.append(int(z[0]))
    assert got2 == want


def test_init_normal_is_standard_normal():
    from scipy import stats
    z = R.init_normal(1234, 3, 400_000, 1.0).astype(np.float64)
    assert abs(z.mean()) < 5 * (1 / math.sqrt(len(z)))
    assert abs(z.std() - 1.0) < 0.01
    assert stats.kstest(z, "norm").pvalue > 1e-3
    # counter-based: a slice drawn alone equals the same slice of a longer draw
    z2 = R.init_normal(1234, 3, 1000, 1.0)
    assert np.array_equal(z2, z[:1000].astype(np.float32))
    # different tensor index -> independent stream
    z3 = R.init_normal(1234, 4, 1000, 1.0)
    assert abs(np.corrcoef(z2, z3)[0, 1]) < 0.15


def test_param_layout_and_counts():
    facts = json.load(open(os.path.join(GOLDEN, "gpt2_facts.json")))
    c124 = R.Config(12, 768, 12, 50257, 50257, 1024)
    assert R.num_params(c124) == facts["num_params_124m_unpadded"]["value"]
    c124p = R.Config(12, 768, 12, 50257, 50304, 1024)
    assert R.num_params(c124p) == facts["num_params_124m_unpadded"]["value"] + 47 * 768
    assert facts["vocab_padded"]["value"] % facts["vocab_padded"]["multiple_of"] == 0


def test_init_params_scheme():
    cfg = R.Config(n_layer=4, n_embd=64, n_head=4, vocab=500, vocab_padded=512, max_T=64)
    p = R.init_params(cfg, 1234)
    assert np.all(p["wte"][500:] == 0.0)
    assert abs(p["wte"][:500].std() - 0.02) < 0.001
    assert abs(p["h0.qkv.w"].std() - 0.02) < 0.001
    assert abs(p["h1.proj.w"].std() - 0.02 / math.sqrt(8)) < 0.0005
    assert abs(p["h2.fcproj.w"].std() - 0.02 / math.sqrt(8)) < 0.0005
    assert np.all(p["h3.ln1.g"] == 1.0) and np.all(p["h3.ln2.b"] == 0.0)
    assert np.all(p["h0.fc.b"] == 0.0) and np.all(p["lnf.g"] == 1.0)
    q = R.init_params(cfg, 1234)
    assert all(np.array_equal(p[k], q[k]) for k in p)
    r = R.init_params(cfg, 1235)
    assert not np.array_equal(p["wte"], r["wte"])


# ---------------------------------------------------------------- single ops vs torch

def test_layernorm_vs_torch():
    x = data.normal(1, (3, 5, 48), 2.0, np.float64) + 3.0
    g = data.normal(2, (48,), 1.0, np.float64)
    b = data.normal(3, (48,), 1.0, np.float64)
    dy = data.normal(4, (3, 5, 48), 1.0, np.float64)
    y, mean, rstd = R.layernorm_forward(x, g, b)
    xt = torch.tensor(x, requires_grad=True)
    gt = torch.tensor(g, requires_grad=True)
    bt = torch.tensor(b, requires_grad=True)
    yt = F.layer_norm(xt, (48,), gt, bt, eps=1e-5)
    yt.backward(torch.tensor(dy))
    assert np.allclose(y, yt.detach().numpy(), rtol=1e-12, atol=1e-12)
    dx, dg, db = R.layernorm_backward(dy, x, g, mean, rstd)
    assert np.allclose(dx, xt.grad.numpy(), rtol=1e-10, atol=1e-12)
    assert np.allclose(dg, gt.grad.numpy(), rtol=1e-10, atol=1e-12)
    assert np.allclose(db, bt.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_layernorm_identities():
    x = data.normal(5, (7, 32), 1.0, np.float64)
    one, zero = np.ones(32), np.zeros(32)
    y, _, _ = R.layernorm_forward(x, one, zero)
    assert np.allclose(y.mean(-1), 0.0, atol=1e-12)
    # shift and positive scale invariance (exact up to eps)
    y2, _, _ = R.layernorm_forward(3.0 * x + 7.0, one, zero, eps=0.0)
    y3, _, _ = R.layernorm_forward(x, one, zero, eps=0.0)
    assert np.allclose(y2, y3, atol=1e-12)
    # a constant row normalises to beta
    beta = data.normal(6, (32,), 1.0, np.float64)
    yc, _, _ = R.layernorm_forward(np.full((2, 32), 4.5), one, beta)
    assert np.allclose(yc, beta, atol=1e-12)
    # dx sums to zero along the row, for any dy
    dy = data.normal(7, (7, 32), 1.0, np.float64)
    _, mean, rstd = R.layernorm_forward(x, one, zero)
    dx, _, _ = R.layernorm_backward(dy, x, one, mean, rstd)
    assert np.allclose(dx.sum(-1), 0.0, atol=1e-12)


def test_gelu_vs_torch_and_special_values():
    u = np.linspace(-8, 8, 1001)
    dg = data.normal(8, u.shape, 1.0, np.float64)
    ut = torch.tensor(u, requires_grad=True)
    gt = F.gelu(ut, approximate="tanh")
    gt.backward(torch.tensor(dg))
    assert np.allclose(R.gelu_forward(u), gt.detach().numpy(), rtol=1e-13, atol=1e-15)
    assert np.allclose(R.gelu_backward(u, dg), ut.grad.numpy(), rtol=1e-11, atol=1e-14)
    assert R.gelu_forward(np.array(0.0)) == 0.0
    assert R.gelu_backward(np.array(0.0), np.array(1.0)) == 0.5
    assert abs(R.gelu_forward(np.array(10.0)) - 10.0) < 1e-12
    # tanh is odd, so gelu(-x) = gelu(x) - x
    assert np.allclose(R.gelu_forward(-u), R.gelu_forward(u) - u, atol=1e-12)


def test_attention_vs_torch():
    B, T, H, hd = 2, 13, 3, 8
    C = H * hd
    qkv = data.normal(9, (B, T, 3 * C), 1.0, np.float64)
    do = data.normal(10, (B, T, C), 1.0, np.float64)
    o, lse = R.attention_forward(qkv, H)
    qt = torch.tensor(qkv, requires_grad=True)
    q, k, v = qt.split(C, dim=-1)
    q, k, v = (a.view(B, T, H, hd).transpose(1, 2) for a in (q, k, v))
    ot = F.scaled_dot_product_attention(q, k, v, is_causal=True)
    ot = ot.transpose(1, 2).reshape(B, T, C)
    ot.backward(torch.tensor(do))
    assert np.allclose(o, ot.detach().numpy(), rtol=1e-11, atol=1e-12)
    s = (q @ k.transpose(-1, -2)) / math.sqrt(hd)
    s = s.masked_fill(torch.ones(T, T, dtype=torch.bool).triu(1), float("-inf"))
    assert np.allclose(lse, torch.logsumexp(s, -1).detach().numpy(), rtol=1e-12)
    dqkv = R.attention_backward(do, qkv, lse, H)
    assert np.allclose(dqkv, qt.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_attention_special_cases():
    H, hd = 2, 4
    C = H * hd
    qkv = data.normal(11, (3, 1, 3 * C), 1.0, np.float64)
    o, lse = R.attention_forward(qkv, H)
    assert np.allclose(o, qkv[..., 2 * C:], atol=1e-15)  # T = 1: o = v
    # equal keys: softmax is uniform over the causal prefix, so o_t = mean of v_0..v_t
    T = 6
    qkv = data.normal(12, (1, T, 3 * C), 1.0, np.float64)
    qkv[..., C:2 * C] = qkv[:, :1, C:2 * C]
    o, _ = R.attention_forward(qkv, H)
    v = qkv[0, :, 2 * C:]
    want = np.cumsum(v, axis=0) / np.arange(1, T + 1)[:, None]
    assert np.allclose(o[0], want, atol=1e-12)


def test_classifier_vs_torch():
    N, V, Vp = 37, 50, 56
    logits = data.normal(13, (N, Vp), 3.0, np.float64)
    logits[:, V:] = 1e3  # padded columns must not take part
    tgt = (np.arange(N) * 7) % V
    losses, dl = R.classifier(logits, tgt, V)
    lt = torch.tensor(logits[:, :V], requires_grad=True)
    loss = F.cross_entropy(lt, torch.tensor(tgt))
    loss.backward()
    assert abs(losses.mean() - loss.item()) < 1e-12
    assert np.allclose(dl[:, :V], lt.grad.numpy(), atol=1e-14)
    assert np.all(dl[:, V:] == 0.0)
    # softmax rows sum to 1; dlogits rows sum to 0
    probs = dl[:, :V] * N
    probs[np.arange(N), tgt] += 1.0
    assert np.allclose(probs.sum(-1), 1.0, atol=1e-12)
    assert np.allclose(dl.sum(-1), 0.0, atol=1e-15)


def test_linear_and_encoder_backward_vs_autograd():
    x = data.normal(14, (9, 5), 1.0, np.float64)
    w = data.normal(15, (7, 5), 1.0, np.float64)
    b = data.normal(16, (7,), 1.0, np.float64)
    dy = data.normal(17, (9, 7), 1.0, np.float64)
    xt, wt, bt = (torch.tensor(a, requires_grad=True) for a in (x, w, b))
    F.linear(xt, wt, bt).backward(torch.tensor(dy))
    dx, dw, db = R.linear_backward(dy, x, w)
    assert np.allclose(R.linear_forward(x, w, b), x @ w.T + b)
    assert np.allclose(dx, xt.grad.numpy()) and np.allclose(dw, wt.grad.numpy())
    assert np.allclose(db, bt.grad.numpy())
    # encoder: gather forward and scatter-add backward vs embedding autograd
    tok = np.array([[3, 1, 3, 0], [1, 1, 2, 3]])
    wte = data.normal(18, (6, 4), 1.0, np.float64)
    wpe = data.normal(19, (5, 4), 1.0, np.float64)
    dx0 = data.normal(20, (2, 4, 4), 1.0, np.float64)
    et, pt = torch.tensor(wte, requires_grad=True), torch.tensor(wpe, requires_grad=True)
    (F.embedding(torch.tensor(tok), et) + pt[:4]).backward(torch.tensor(dx0))
    dwte, dwpe = R.encoder_backward(dx0, tok, 6, 5)
    assert np.allclose(dwte, et.grad.numpy()) and np.allclose(dwpe, pt.grad.numpy())


def test_encoder_indexing_is_exact():
    V, C, T = 300, 8, 16
    wte = np.zeros((V, C), dtype=np.float32)
    wte[:, 0] = np.arange(V)
    wpe = np.zeros((T, C), dtype=np.float32)
    wpe[:, 1] = np.arange(T)
    tok = data.token_stream("uniform", 3 * T, 5, vocab=V).reshape(3, T)
    x0 = R.encoder_forward(wte, wpe, tok)
    assert np.array_equal(x0[..., 0].astype(np.int64), tok)
    assert np.array_equal(x0[..., 1].astype(np.int64), np.broadcast_to(np.arange(T), (3, T)))


def test_adamw_vs_torch_and_closed_form():
    theta0 = data.normal(21, (50,), 1.0, np.float64)
    grads = [data.normal(22 + i, (50,), 1.0, np.float64) for i in range(4)]
    lr, b1, b2, eps, wd = 3e-4, 0.9, 0.95, 1e-8, 0.1
    pt = torch.tensor(theta0, requires_grad=True)
    opt = torch.optim.AdamW([pt], lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd)
    th, m, v = theta0.copy(), np.zeros(50), np.zeros(50)
    for t, g in enumerate(grads, start=1):
        pt.grad = torch.tensor(g)
        opt.step()
        th, m, v = R.adamw_update(th, g, m, v, lr, b1, b2, eps, wd, t)
        if t == 1:  # m-hat = g, v-hat = g^2 at t = 1
            closed = theta0 - lr * (grads[0] / (np.abs(grads[0]) + eps) + wd * theta0)
            assert np.allclose(th, closed, rtol=0, atol=1e-15)
    assert np.allclose(th, pt.detach().numpy(), rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------- whole step

@pytest.mark.parametrize("cfg,B,T", [(MICRO, 2, 8), (TINY, 2, 32)])
def test_step_vs_torch_autograd(cfg, B, T):
    params = random_params(cfg, 3)
    tok = data.token_stream("uniform", B * T + 1, 7, vocab=cfg.vocab)
    tokens, targets = tok[:-1].reshape(B, T), tok[1:].reshape(B, T)
    loss, cache = R.forward(cfg, params, tokens, targets)
    grads = R.backward(cfg, cache)
    tl, tg, tlogits = torch_loss_and_grads(cfg, params, tokens, targets)
    assert abs(loss - tl) < 1e-11
    assert np.allclose(cache["logits"][..., :cfg.vocab], tlogits, rtol=1e-11, atol=1e-11)
    for name, g in grads.items():
        assert rel_l2(g, tg[name]) < 1e-10, name


def test_step_vs_finite_differences():
    cfg = MICRO
    B, T = 2, 8
    params = random_params(cfg, 4)
    tok = data.token_stream("uniform", B * T + 1, 8, vocab=cfg.vocab)
    tokens, targets = tok[:-1].reshape(B, T), tok[1:].reshape(B, T)
    _, cache = R.forward(cfg, params, tokens, targets)
    grads = R.backward(cfg, cache)
    h = 1e-5
    worst = 0.0
    for name in params:
        fd = np.zeros_like(params[name])
        flat = params[name].reshape(-1)
        for i in range(flat.size):
            old = flat[i]
            flat[i] = old + h
            lp, _ = R.forward(cfg, params, tokens, targets)
            flat[i] = old - h
            lm, _ = R.forward(cfg, params, tokens, targets)
            flat[i] = old
            fd.reshape(-1)[i] = (lp - lm) / (2 * h)
        err = rel_l2(grads[name], fd) if np.linalg.norm(fd) > 0 else np.abs(grads[name]).max()
        worst = max(worst, err)
        assert err < 1e-6, (name, err)
    assert np.all(grads["wte"][cfg.vocab:] == 0.0)


def test_zero_weights_give_log_vocab():
    for V, Vp in ((512, 512), (50257, 50304)):
        cfg = R.Config(n_layer=1, n_embd=16, n_head=2, vocab=V, vocab_padded=Vp, max_T=8)
        params = {n: np.zeros(s) for n, s, _ in R.param_specs(cfg)}
        tok = data.token_stream("uniform", 17, 1, vocab=V)
        loss, _ = R.forward(cfg, params, tok[:-1].reshape(2, 8), tok[1:].reshape(2, 8))
        assert abs(loss - math.log(V)) < 1e-12  # ln V, not ln Vp: padding is masked


def test_initial_loss_near_log_vocab():
    cfg = TINY
    params = R.init_params(cfg, 1234)
    tokens, targets = data.batches("uniform", 4, 64, 1, 1234, vocab=512)
    loss, _ = R.forward(cfg, params, tokens[0], targets[0])
    assert abs(loss - math.log(512)) < 0.05


def test_causality():
    cfg = TINY
    params = random_params(cfg, 5)
    B, T, t0 = 2, 40, 17
    tok = data.token_stream("uniform", B * T, 9, vocab=cfg.vocab).reshape(B, T)
    _, c1 = R.forward(cfg, params, tok)
    tok2 = tok.copy()
    tok2[:, t0 + 1:] = (tok2[:, t0 + 1:] + 101) % cfg.vocab
    _, c2 = R.forward(cfg, params, tok2)
    assert np.array_equal(c1["logits"][:, :t0 + 1], c2["logits"][:, :t0 + 1])
    assert not np.allclose(c1["logits"][:, t0 + 1:], c2["logits"][:, t0 + 1:])


def test_tied_embedding_gradient_is_head_plus_scatter():
    cfg = MICRO
    params = random_params(cfg, 6)
    tok = data.token_stream("uniform", 17, 10, vocab=cfg.vocab)
    tokens, targets = tok[:-1].reshape(2, 8), tok[1:].reshape(2, 8)
    _, cache = R.forward(cfg, params, tokens, targets)
    grads = R.backward(cfg, cache)
    # with a zero residual-stream gradient path the scatter part vanishes:
    # compare against the head part computed alone
    hf = cache["hf"].reshape(16, -1)
    head = cache["dlogits"].T @ hf
    scatter = grads["wte"] - head
    rows_unused = np.setdiff1d(np.arange(cfg.vocab_padded), tokens.reshape(-1))
    assert np.allclose(scatter[rows_unused], 0.0, atol=1e-15)
    assert np.abs(scatter[np.unique(tokens)]).max() > 0


def test_fp32_oracle_matches_fp64():
    cfg = TINY
    params = R.init_params(cfg, 1234)
    tokens, targets = data.batches("uniform", 4, 64, 1, 1234, vocab=512)
    l64, c64 = R.forward(cfg, params, tokens[0], targets[0], dtype=np.float64)
    g64 = R.backward(cfg, c64)
    l32, c32 = R.forward(cfg, params, tokens[0], targets[0], dtype=np.float32)
    g32 = R.backward(cfg, c32)
    assert abs(l32 - l64) < 1e-5
    for k in g64:
        if np.linalg.norm(g64[k]) > 0:
            assert rel_l2(g32[k], g64[k]) < 1e-5, k
