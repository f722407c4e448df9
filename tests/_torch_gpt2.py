"""GPT-2 built from torch library routines, for pinning the oracle.

Each operation is a torch.nn.functional call (embedding, layer_norm, linear,
scaled_dot_product_attention, gelu with the tanh approximation,
cross_entropy), and gradients come from autograd. It shares no arithmetic
with the oracle's hand-written forward and backward; it only composes the
same architecture (pre-LN blocks, tied LM head, masked padded vocabulary).
"""
import torch
import torch.nn.functional as F


def torch_loss_and_grads(cfg, params: dict, tokens, targets, dtype=torch.float64):
    P = {k: torch.tensor(v, dtype=dtype, requires_grad=True) for k, v in params.items()}
    tok = torch.as_tensor(tokens, dtype=torch.long)
    tgt = torch.as_tensor(targets, dtype=torch.long)
    B, T = tok.shape
    C, H = cfg.n_embd, cfg.n_head
    x = F.embedding(tok, P["wte"]) + P["wpe"][:T]
    for l in range(cfg.n_layer):
        p = f"h{l}."
        h = F.layer_norm(x, (C,), P[p + "ln1.g"], P[p + "ln1.b"], eps=1e-5)
        qkv = F.linear(h, P[p + "qkv.w"], P[p + "qkv.b"])
        q, k, v = qkv.split(C, dim=-1)
        q, k, v = (a.view(B, T, H, C // H).transpose(1, 2) for a in (q, k, v))
        o = F.scaled_dot_product_attention(q, k, v, is_causal=True)
        o = o.transpose(1, 2).reshape(B, T, C)
        x = x + F.linear(o, P[p + "proj.w"], P[p + "proj.b"])
        h = F.layer_norm(x, (C,), P[p + "ln2.g"], P[p + "ln2.b"], eps=1e-5)
        g = F.gelu(F.linear(h, P[p + "fc.w"], P[p + "fc.b"]), approximate="tanh")
        x = x + F.linear(g, P[p + "fcproj.w"], P[p + "fcproj.b"])
    h = F.layer_norm(x, (C,), P["lnf.g"], P["lnf.b"], eps=1e-5)
    logits = F.linear(h, P["wte"])[..., :cfg.vocab]
    loss = F.cross_entropy(logits.reshape(B * T, -1), tgt.reshape(-1))
    loss.backward()
    return loss.item(), {k: t.grad.numpy() for k, t in P.items()}, logits.detach().numpy()
