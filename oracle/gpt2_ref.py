"""Oracle: a plain numpy GPT-2 training step (test infrastructure only).

Source: llm.c "State of the Union [May 3, 2024]" (karpathy/llm.c discussion
#344). That page trains GPT-2 124M with bf16 activations and an fp32 master
copy ("Single GPU training"), uses a fused classifier that takes the loss
only at the label's index ("Single GPU training"), masks the padded vocab
columns 50257..50303 to -inf ("Fine print"), and lists the step's kernels
(encoder, layernorm, matmul, attention, GELU, residual, classifier, AdamW:
the kernel table under "Runtime, DRAM traffic, instructions").
The pages print no formula, so each function states the standard GPT-2
operation it computes.

Arithmetic runs in the dtype of the arrays (float64 by default, float32 for
the large shapes). Matmul, exp, log, tanh and sqrt are numpy library calls;
there is no fusion, blocking or reordering beyond the formulas written here.

Readings where the pages are silent (each is also listed in the design notes):
  * LayerNorm: eps = 1e-5, biased variance (divide by C).
  * GELU: tanh form, 0.5 u (1 + tanh(sqrt(2/pi) (u + 0.044715 u^3))).
  * Attention: scale 1/sqrt(hd), causal over the whole window (no document
    masking at EoS); q, k, v are the column blocks [0,C), [C,2C), [2C,3C) of
    the fused projection, head h at columns h*hd .. h*hd+hd-1 of each block.
  * Padded vocab rows of wte are initialised to 0; padded logits are left out
    of the softmax and their dlogits are 0.
  * Loss: mean over all B*T positions.
  * AdamW: bias-corrected moments, eps outside the square root, decoupled
    weight decay on theta before the update, applied to every tensor.
  * Init: N(0, 0.02) for wte, wpe and all matrices; N(0, 0.02/sqrt(2L)) for
    the two residual projections; biases 0; LayerNorm gain 1, bias 0.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

from oracle import fp8_ref as F8

LN_EPS = 1e-5
GELU_K = math.sqrt(2.0 / math.pi)
GELU_A = 0.044715


# --------------------------------------------------------------------------
# Configuration and parameter layout
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class Config:
    n_layer: int
    n_embd: int
    n_head: int
    vocab: int
    vocab_padded: int
    max_T: int

    @property
    def head_dim(self) -> int:
        return self.n_embd // self.n_head


def param_specs(cfg: Config):
    """Parameters in canonical order: (name, shape, init std or 'zero'/'one').

    Order: wte [Vp,C], wpe [max_T,C]; per layer ln1 gain/bias, fused qkv
    weight [3C,C] and bias, attention projection [C,C] and bias, ln2
    gain/bias, fc [4C,C] and bias, fc projection [C,4C] and bias; then the
    final LayerNorm gain/bias. Weights use the PyTorch Linear layout [out, in].
    """
    C, L = cfg.n_embd, cfg.n_layer
    std = 0.02
    std_res = 0.02 / math.sqrt(2.0 * L)
    specs = [("wte", (cfg.vocab_padded, C), std), ("wpe", (cfg.max_T, C), std)]
    for l in range(L):
        p = f"h{l}."
        specs += [
            (p + "ln1.g", (C,), "one"), (p + "ln1.b", (C,), "zero"),
            (p + "qkv.w", (3 * C, C), std), (p + "qkv.b", (3 * C,), "zero"),
            (p + "proj.w", (C, C), std_res), (p + "proj.b", (C,), "zero"),
            (p + "ln2.g", (C,), "one"), (p + "ln2.b", (C,), "zero"),
            (p + "fc.w", (4 * C, C), std), (p + "fc.b", (4 * C,), "zero"),
            (p + "fcproj.w", (C, 4 * C), std_res), (p + "fcproj.b", (C,), "zero"),
        ]
    specs += [("lnf.g", (C,), "one"), ("lnf.b", (C,), "zero")]
    return specs


def num_params(cfg: Config) -> int:
    return sum(int(np.prod(s)) for _, s, _ in param_specs(cfg))


# --------------------------------------------------------------------------
# Init: a counter-based normal generator
# --------------------------------------------------------------------------
# Element i of tensor k (canonical order) is drawn from counter c = k*2^40 + i.
# Its splitmix64 state starts at seed XOR (c * 0x9E3779B97F4A7C15 mod 2^64);
# two successive splitmix64 outputs r1, r2 (Steele, Lea and Flood 2014) give
# u1 = ((r1 >> 11) + 1) * 2^-53 in (0, 1] and u2 = (r2 >> 11) * 2^-53 in [0, 1),
# and the Box-Muller transform (Box and Muller 1958) gives
# z = sqrt(-2 ln u1) * cos(2 pi u2), all in float64. The stored weight is
# float32(std * z), rounded to nearest even.

_G = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _splitmix_next(state):
    with np.errstate(over="ignore"):
        state = state + _G
        z = (state ^ (state >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return state, z ^ (z >> np.uint64(31))


def init_normal(seed: int, tensor_index: int, n: int, std: float) -> np.ndarray:
    """float32 array of n N(0, std^2) draws for tensor `tensor_index` (see above)."""
    out = np.empty(n, dtype=np.float32)
    chunk = 1 << 22
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        c = np.uint64(tensor_index) * np.uint64(1 << 40) + np.arange(lo, hi, dtype=np.uint64)
        with np.errstate(over="ignore"):
            s = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) ^ (c * _G)
        s, r1 = _splitmix_next(s)
        s, r2 = _splitmix_next(s)
        u1 = ((r1 >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
        u2 = (r2 >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
        z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)
        out[lo:hi] = (std * z).astype(np.float32)
    return out


def init_params(cfg: Config, seed: int) -> dict:
    """Initial fp32 master weights, name -> float32 array (see param_specs)."""
    params = {}
    for k, (name, shape, how) in enumerate(param_specs(cfg)):
        n = int(np.prod(shape))
        if how == "zero":
            a = np.zeros(n, dtype=np.float32)
        elif how == "one":
            a = np.ones(n, dtype=np.float32)
        else:
            a = init_normal(seed, k, n, how)
        a = a.reshape(shape)
        if name == "wte":
            a[cfg.vocab:, :] = 0.0  # padded vocab rows start at zero
        params[name] = a
    return params


# --------------------------------------------------------------------------
# Forward operations
# --------------------------------------------------------------------------

def encoder_forward(wte, wpe, tokens):
    """x0[b,t,:] = wte[tokens[b,t],:] + wpe[t,:]."""
    T = tokens.shape[1]
    return wte[tokens] + wpe[:T][None, :, :]


def layernorm_forward(x, gamma, beta, eps=LN_EPS):
    """y = (x - mean) * rstd * gamma + beta over the last axis; biased variance.

    Returns y, mean, rstd (mean and rstd without the last axis).
    """
    mean = x.mean(axis=-1, keepdims=True)
    var = ((x - mean) ** 2).mean(axis=-1, keepdims=True)
    rstd = 1.0 / np.sqrt(var + eps)
    y = (x - mean) * rstd * gamma + beta
    return y, mean[..., 0], rstd[..., 0]


def linear_forward(x, w, b=None):
    """y = x @ w^T (+ b), w in the [out, in] layout."""
    y = x @ w.T
    if b is not None:
        y = y + b
    return y


def _fp8(a, fmt):
    """The values a per-tensor FP8 quantization of a (fp8_ref.quantize: scale
    fmax / amax, codes rounded to nearest, ties to even) stands for:
    decode(codes) * amax / fmax, in float64."""
    codes, scale_inv = F8.quantize(a, fmt)
    return F8.fp8_decode(codes, fmt) * float(scale_inv)


def linear_forward_fp8(x, w, b=None):
    """The FP8 linear layer (modded-nanogpt project page, "How it works":
    FP8 for the MLP, the QKV projections and the head): y = x w^T (+ b) with x
    and w each quantized per tensor to e4m3 first, the product of the
    quantized values in float64; returned in x's dtype."""
    y = _fp8(x, "e4m3") @ _fp8(w, "e4m3").T
    if b is not None:
        y = y + b
    return y.astype(np.asarray(x).dtype)


def _split_heads(qkv, n_head):
    B, T, C3 = qkv.shape
    C = C3 // 3
    hd = C // n_head

    def heads(a):
        return a.reshape(B, T, n_head, hd).transpose(0, 2, 1, 3)  # [B, H, T, hd]

    return heads(qkv[..., :C]), heads(qkv[..., C:2 * C]), heads(qkv[..., 2 * C:])


def _causal_scores(q, k):
    hd = q.shape[-1]
    T = q.shape[2]
    s = (q @ k.swapaxes(-1, -2)) / math.sqrt(hd)
    future = np.triu(np.ones((T, T), dtype=bool), k=1)  # key s > query t
    s = np.where(future, -np.inf, s)
    return s, future


def attention_forward(qkv, n_head):
    """Causal multi-head attention.

    Per (b, h): S = q k^T / sqrt(hd), S[t, s] = -inf for s > t,
    P = softmax over s, o = P v, lse[t] = max_s S[t, s] + log sum_s exp(S[t, s] - max).
    Returns o [B, T, C] (heads concatenated) and lse [B, H, T].
    """
    B, T, C3 = qkv.shape
    q, k, v = _split_heads(qkv, n_head)
    s, _ = _causal_scores(q, k)
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    l_ = e.sum(axis=-1, keepdims=True)
    p = e / l_
    o = p @ v
    lse = (m + np.log(l_))[..., 0]
    return o.transpose(0, 2, 1, 3).reshape(B, T, C3 // 3), lse


def gelu_forward(u):
    """GELU, tanh form: 0.5 u (1 + tanh(sqrt(2/pi) (u + 0.044715 u^3)))."""
    return 0.5 * u * (1.0 + np.tanh(GELU_K * (u + GELU_A * u ** 3)))


def classifier(logits, targets, vocab):
    """Softmax cross-entropy over the real vocabulary, with its gradient.

    logits [N, Vp]; only columns j < vocab take part. For each row i:
    lse_i = log sum_{j<V} exp(z_ij), loss_i = lse_i - z_i,target,
    dlogits_ij = (exp(z_ij - lse_i) - [j == target_i]) / N for j < V, 0 for j >= V.
    The 1/N factor is d(mean loss)/d(loss_i).
    Returns per-row losses [N] and dlogits [N, Vp].
    """
    N = logits.shape[0]
    z = logits[:, :vocab]
    m = z.max(axis=-1, keepdims=True)
    lse = m + np.log(np.exp(z - m).sum(axis=-1, keepdims=True))
    rows = np.arange(N)
    losses = lse[:, 0] - z[rows, targets]
    dlogits = np.zeros_like(logits)
    dlogits[:, :vocab] = np.exp(z - lse) / N
    dlogits[rows, targets] -= 1.0 / N
    return losses, dlogits


# --------------------------------------------------------------------------
# Backward operations
# --------------------------------------------------------------------------

def linear_backward(dy, x, w):
    """For y = x w^T + b: dx = dy w, dw = dy^T x, db = column sums of dy.

    dy [N, out], x [N, in] (leading axes flattened by the caller).
    """
    return dy @ w, dy.T @ x, dy.sum(axis=0)


def linear_backward_fp8(dy, x, w):
    """The FP8 linear layer's gradients: dy quantized per tensor to e5m2
    (the wider range of gradients), x and w to e4m3 (as in the forward),
    dx = dy w and dw = dy^T x of the quantized values in float64; db is the
    column sums of dy itself. Returned in dy's dtype."""
    dt = np.asarray(dy).dtype
    qdy, qx, qw = _fp8(dy, "e5m2"), _fp8(x, "e4m3"), _fp8(w, "e4m3")
    return (qdy @ qw).astype(dt), (qdy.T @ qx).astype(dt), dy.sum(axis=0)


def layernorm_backward(dy, x, gamma, mean, rstd):
    """Gradients of y = xhat * gamma + beta, xhat = (x - mean) * rstd.

    dxhat = dy * gamma;
    dx = rstd * (dxhat - mean(dxhat) - xhat * mean(dxhat * xhat)) (means over the row);
    dgamma = sum over rows of dy * xhat; dbeta = sum over rows of dy.
    """
    xhat = (x - mean[..., None]) * rstd[..., None]
    dxhat = dy * gamma
    dx = rstd[..., None] * (dxhat - dxhat.mean(axis=-1, keepdims=True)
                            - xhat * (dxhat * xhat).mean(axis=-1, keepdims=True))
    C = x.shape[-1]
    dgamma = (dy * xhat).reshape(-1, C).sum(axis=0)
    dbeta = dy.reshape(-1, C).sum(axis=0)
    return dx, dgamma, dbeta


def attention_backward(dout, qkv, lse, n_head):
    """Backward of attention_forward, with P recomputed from the saved lse.

    P = exp(S - lse) (0 where masked); o = P v; D_t = sum_d dO_td O_td;
    dV = P^T dO; dP = dO V^T; dS = P * (dP - D); dQ = dS K / sqrt(hd);
    dK = dS^T Q / sqrt(hd). Returns dqkv [B, T, 3C] in the fused layout.
    """
    B, T, C3 = qkv.shape
    C = C3 // 3
    hd = C // n_head
    q, k, v = _split_heads(qkv, n_head)
    do = dout.reshape(B, T, n_head, hd).transpose(0, 2, 1, 3)
    s, future = _causal_scores(q, k)
    p = np.where(future, 0.0, np.exp(s - lse[..., None]))
    o = p @ v
    D = (do * o).sum(axis=-1)
    dv = p.swapaxes(-1, -2) @ do
    dp = do @ v.swapaxes(-1, -2)
    ds = p * (dp - D[..., None])
    dq = (ds @ k) / math.sqrt(hd)
    dk = (ds.swapaxes(-1, -2) @ q) / math.sqrt(hd)

    def merge(a):
        return a.transpose(0, 2, 1, 3).reshape(B, T, C)

    return np.concatenate([merge(dq), merge(dk), merge(dv)], axis=-1)


def gelu_backward(u, dg):
    """du = dg * g'(u), g'(u) = 0.5 (1 + t) + 0.5 u (1 - t^2) sqrt(2/pi) (1 + 3*0.044715 u^2),
    t = tanh(sqrt(2/pi) (u + 0.044715 u^3))."""
    t = np.tanh(GELU_K * (u + GELU_A * u ** 3))
    d = 0.5 * (1.0 + t) + 0.5 * u * (1.0 - t * t) * GELU_K * (1.0 + 3.0 * GELU_A * u * u)
    return dg * d


def encoder_backward(dx0, tokens, vocab_padded, max_T):
    """dwte[v] = sum of dx0[b,t] over positions with tokens[b,t] == v; dwpe[t] = sum_b dx0[b,t]."""
    B, T, C = dx0.shape
    dwte = np.zeros((vocab_padded, C), dtype=dx0.dtype)
    np.add.at(dwte, tokens.reshape(-1), dx0.reshape(-1, C))
    dwpe = np.zeros((max_T, C), dtype=dx0.dtype)
    dwpe[:T] = dx0.sum(axis=0)
    return dwte, dwpe


def adamw_update(theta, g, m, v, lr, beta1, beta2, eps, weight_decay, t):
    """One AdamW step (Loshchilov and Hutter), t >= 1.

    m = b1 m + (1-b1) g; v = b2 v + (1-b2) g^2; mhat = m / (1 - b1^t);
    vhat = v / (1 - b2^t); theta = theta - lr (mhat / (sqrt(vhat) + eps) + wd theta).
    Returns new theta, m, v.
    """
    m = beta1 * m + (1.0 - beta1) * g
    v = beta2 * v + (1.0 - beta2) * g * g
    mhat = m / (1.0 - beta1 ** t)
    vhat = v / (1.0 - beta2 ** t)
    theta = theta - lr * (mhat / (np.sqrt(vhat) + eps) + weight_decay * theta)
    return theta, m, v


# --------------------------------------------------------------------------
# The training loop around the step (the "next" rows: gradient accumulation,
# global-norm clipping, a weight-decay mask, a cosine learning-rate schedule)
# --------------------------------------------------------------------------

def global_grad_norm(grads: dict):
    """||g||_2 over every parameter gradient, in float64."""
    return math.sqrt(sum(float(np.sum(np.asarray(g, dtype=np.float64) ** 2)) for g in grads.values()))


def clip_factor(norm, max_norm, grad_scale=1.0):
    """The global-norm clip applied to g * grad_scale: min(1, max_norm / (||g|| grad_scale + 1e-6));
    1 when max_norm is 0 (no clipping)."""
    if max_norm <= 0:
        return 1.0
    return min(1.0, max_norm / (norm * grad_scale + 1e-6))


def decays(name: str, arr) -> bool:
    """Weight decay applies to the 2-D tensors (wte, wpe, weight matrices), not
    to biases and LayerNorm parameters (the decay-mask reading)."""
    return np.ndim(arr) == 2


def adamw_update_ex(theta, g, m, v, lr, beta1, beta2, eps, weight_decay, t, grad_scale=1.0, clip=1.0):
    """AdamW on the gradient g * grad_scale * clip (the moments, bias correction and
    decoupled decay as in adamw_update)."""
    return adamw_update(theta, np.asarray(g) * (grad_scale * clip), m, v, lr, beta1, beta2, eps, weight_decay, t)


def lr_cosine(t, warmup, total, lr_max, lr_min):
    """Step t (1-based): linear warmup over `warmup` steps to lr_max, then
    lr_min + (lr_max - lr_min) (1 + cos(pi (t - warmup) / (total - warmup))) / 2
    up to step `total`, lr_min after it."""
    if t < 1:
        return 0.0
    if warmup > 0 and t <= warmup:
        return lr_max * t / warmup
    if t >= total:
        return lr_min
    frac = (t - warmup) / (total - warmup)
    return lr_min + 0.5 * (lr_max - lr_min) * (1.0 + math.cos(math.pi * frac))


# --------------------------------------------------------------------------
# The whole step
# --------------------------------------------------------------------------

def forward(cfg: Config, params: dict, tokens, targets=None, dtype=np.float64, fp8=()):
    """Forward pass. Returns (mean loss or None, cache for backward).

    Per layer: h1 = LN1(x); qkv = h1 Wqkv^T + b; o = attn(qkv); x1 = x + o Wproj^T + b;
    h2 = LN2(x1); u = h2 Wfc^T + b; g = gelu(u); x = x1 + g Wfcproj^T + b.
    Then hf = LNf(x); logits = hf wte^T (tied head, no bias).
    fp8: the linears that run as FP8 linear layers, any of "qkv", "mlp" (both
    MLP linears) and "head".
    """
    P = {k: np.asarray(v, dtype=dtype) for k, v in params.items()}
    tokens = np.asarray(tokens)
    B, T = tokens.shape
    C = cfg.n_embd
    lin = {k: (linear_forward_fp8 if k in fp8 else linear_forward) for k in ("qkv", "mlp", "head")}
    cache = {"tokens": tokens, "P": P, "layers": [], "fp8": tuple(fp8)}
    x = encoder_forward(P["wte"], P["wpe"], tokens)
    for l in range(cfg.n_layer):
        p = f"h{l}."
        lc = {"x": x}
        h1, lc["mean1"], lc["rstd1"] = layernorm_forward(x, P[p + "ln1.g"], P[p + "ln1.b"])
        qkv = lin["qkv"](h1, P[p + "qkv.w"], P[p + "qkv.b"])
        o, lse = attention_forward(qkv, cfg.n_head)
        x1 = x + linear_forward(o, P[p + "proj.w"], P[p + "proj.b"])
        h2, lc["mean2"], lc["rstd2"] = layernorm_forward(x1, P[p + "ln2.g"], P[p + "ln2.b"])
        u = lin["mlp"](h2, P[p + "fc.w"], P[p + "fc.b"])
        g = gelu_forward(u)
        x = x1 + lin["mlp"](g, P[p + "fcproj.w"], P[p + "fcproj.b"])
        lc.update(h1=h1, qkv=qkv, o=o, lse=lse, x1=x1, h2=h2, u=u, g=g)
        cache["layers"].append(lc)
    hf, meanf, rstdf = layernorm_forward(x, P["lnf.g"], P["lnf.b"])
    logits = lin["head"](hf, P["wte"])  # [B, T, Vp]
    cache.update(xL=x, hf=hf, meanf=meanf, rstdf=rstdf, logits=logits)
    if targets is None:
        return None, cache
    losses, dlogits = classifier(logits.reshape(B * T, -1), np.asarray(targets).reshape(-1),
                                 cfg.vocab)
    cache["losses"] = losses
    cache["dlogits"] = dlogits
    return float(losses.mean()), cache


def backward(cfg: Config, cache: dict) -> dict:
    """Gradients of the mean loss w.r.t. every parameter (name -> array)."""
    P = cache["P"]
    tokens = cache["tokens"]
    B, T = tokens.shape
    C = cfg.n_embd
    N = B * T
    grads = {}
    fp8 = cache.get("fp8", ())
    lin = {k: (linear_backward_fp8 if k in fp8 else linear_backward) for k in ("qkv", "mlp", "head")}
    dlogits = cache["dlogits"]
    hf = cache["hf"].reshape(N, C)
    dhf, dwte_head, _ = lin["head"](dlogits, hf, P["wte"])
    dx, grads["lnf.g"], grads["lnf.b"] = layernorm_backward(
        dhf.reshape(B, T, C), cache["xL"], P["lnf.g"], cache["meanf"], cache["rstdf"])
    for l in reversed(range(cfg.n_layer)):
        p = f"h{l}."
        lc = cache["layers"][l]
        # MLP branch: x_out = x1 + fcproj(gelu(fc(LN2(x1))))
        dg, grads[p + "fcproj.w"], grads[p + "fcproj.b"] = lin["mlp"](
            dx.reshape(N, C), lc["g"].reshape(N, 4 * C), P[p + "fcproj.w"])
        du = gelu_backward(lc["u"].reshape(N, 4 * C), dg)
        dh2, grads[p + "fc.w"], grads[p + "fc.b"] = lin["mlp"](
            du, lc["h2"].reshape(N, C), P[p + "fc.w"])
        dx1_ln, grads[p + "ln2.g"], grads[p + "ln2.b"] = layernorm_backward(
            dh2.reshape(B, T, C), lc["x1"], P[p + "ln2.g"], lc["mean2"], lc["rstd2"])
        dx1 = dx + dx1_ln  # residual join
        # attention branch: x1 = x + proj(attn(qkv(LN1(x))))
        do, grads[p + "proj.w"], grads[p + "proj.b"] = linear_backward(
            dx1.reshape(N, C), lc["o"].reshape(N, C), P[p + "proj.w"])
        dqkv = attention_backward(do.reshape(B, T, C), lc["qkv"], lc["lse"], cfg.n_head)
        dh1, grads[p + "qkv.w"], grads[p + "qkv.b"] = lin["qkv"](
            dqkv.reshape(N, 3 * C), lc["h1"].reshape(N, C), P[p + "qkv.w"])
        dx_ln, grads[p + "ln1.g"], grads[p + "ln1.b"] = layernorm_backward(
            dh1.reshape(B, T, C), lc["x"], P[p + "ln1.g"], lc["mean1"], lc["rstd1"])
        dx = dx1 + dx_ln  # residual join
    dwte_enc, grads["wpe"] = encoder_backward(dx, tokens, cfg.vocab_padded, cfg.max_T)
    grads["wte"] = dwte_head + dwte_enc  # tied embedding / LM head
    return grads


def train_step(cfg: Config, params: dict, tokens, targets, state: dict | None,
               lr, beta1, beta2, eps, weight_decay, t, dtype=np.float64, fp8=()):
    """forward -> backward -> AdamW. Returns (loss, grads, new_params, new_state).

    state holds the moments {"m": {name: arr}, "v": {...}}; None means zeros (t = 1).
    fp8: the FP8 linear layers (see forward).
    """
    loss, cache = forward(cfg, params, tokens, targets, dtype=dtype, fp8=fp8)
    grads = backward(cfg, cache)
    new_params, m_new, v_new = {}, {}, {}
    for name, theta in params.items():
        theta = np.asarray(theta, dtype=dtype)
        m = np.zeros_like(theta) if state is None else np.asarray(state["m"][name], dtype=dtype)
        v = np.zeros_like(theta) if state is None else np.asarray(state["v"][name], dtype=dtype)
        new_params[name], m_new[name], v_new[name] = adamw_update(
            theta, grads[name], m, v, lr, beta1, beta2, eps, weight_decay, t)
    return loss, grads, new_params, {"m": m_new, "v": v_new}


def position_losses(cfg: Config, params: dict, tokens, targets, dtype=np.float64):
    """Per-position losses [B, T] of the forward pass (no backward)."""
    _, cache = forward(cfg, params, tokens, targets, dtype=dtype)
    return cache["losses"].reshape(np.asarray(tokens).shape)
