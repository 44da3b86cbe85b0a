"""An independent fp64 CPU model assembled from torch.nn.functional routines.

Used only to pin the oracle: it shares no code with it (the oracle is numpy),
and each step is a library routine (layer_norm, linear, gelu,
scaled_dot_product_attention, cross_entropy) rather than a retyped formula;
its gradients come from torch's autograd.
"""
import numpy as np
import torch
import torch.nn.functional as F

from workloads.configs import PRE_NORM, GELU_TANH


def _t(a):
    return torch.from_numpy(np.asarray(a, np.float64))


def forward(cfg, w, ids, targets=None):
    loss, logits = _forward(cfg, w, ids, targets, _t)
    return (None if loss is None else float(loss)), logits.detach().numpy()


def grads(cfg, w, ids, targets):
    """(loss, gradients keyed like the weight dict) by torch autograd through the same functional model."""
    leaves = {}

    def leaf(a):
        key = id(a)
        if key not in leaves:
            leaves[key] = (a, _t(a).clone().requires_grad_(True))
        return leaves[key][1]

    loss, _ = _forward(cfg, w, ids, targets, leaf)
    loss.backward()

    def g(a):
        t = leaves.get(id(a))
        return np.zeros(np.shape(a)) if t is None or t[1].grad is None else t[1].grad.numpy()

    out = {k: g(w[k]) for k in ("wte", "wpe", "lnf_g", "lnf_b", "head") if k in w}
    out["layers"] = [{k: g(v) for k, v in p.items()} for p in w["layers"]]
    return float(loss.detach()), out


def _forward(cfg, w, ids, targets, _t):
    E = _t(w["wte"])
    P = _t(w["wpe"])
    ids_t = torch.from_numpy(np.asarray(ids, np.int64))
    B, T = ids_t.shape
    x = E[ids_t] + P[:T]
    approx = "tanh" if cfg.gelu == GELU_TANH else "none"
    C, H = cfg.C, cfg.H
    D = C // H

    def attn(a, p):
        qkv = F.linear(a, _t(p["attn_w"]), _t(p["attn_b"]))
        q, k, v = qkv.split(C, dim=-1)
        q = q.view(B, T, H, D).transpose(1, 2)
        k = k.view(B, T, H, D).transpose(1, 2)
        v = v.view(B, T, H, D).transpose(1, 2)
        y = F.scaled_dot_product_attention(q, k, v, is_causal=True)
        y = y.transpose(1, 2).reshape(B, T, C)
        return F.linear(y, _t(p["proj_w"]), _t(p["proj_b"]))

    def mlp(a, p):
        g = F.gelu(F.linear(a, _t(p["fc_w"]), _t(p["fc_b"])), approximate=approx)
        return F.linear(g, _t(p["mp_w"]), _t(p["mp_b"]))

    def ln(a, g, b):
        return F.layer_norm(a, (C,), _t(g), _t(b), eps=cfg.ln_eps)

    for p in w["layers"]:
        if cfg.norm_mode == PRE_NORM:
            x = x + attn(ln(x, p["ln1_g"], p["ln1_b"]), p)
            x = x + mlp(ln(x, p["ln2_g"], p["ln2_b"]), p)
        else:
            n = ln(x + attn(x, p), p["ln1_g"], p["ln1_b"])
            x = ln(n + mlp(n, p), p["ln2_g"], p["ln2_b"])
    if cfg.final_ln:
        x = ln(x, w["lnf_g"], w["lnf_b"])
    head = _t(w["head"]) if getattr(cfg, "untied_head", 0) else E
    logits = x @ head.T
    loss = None
    if targets is not None:
        tg = torch.from_numpy(np.asarray(targets, np.int64)).reshape(-1)
        loss = F.cross_entropy(logits.reshape(-1, logits.shape[-1]), tg)
    return loss, logits
