"""Seeded inputs on the CUDA device (torch), for the GPU tests, the smoke run and the
benchmark.

``to_dev`` / ``lora_dev`` move the host inputs of ``synth.inputs`` to the device in the
storage types the library reads.  ``device_layer`` draws the inputs of one large layer
directly on the device with torch's seeded generator (the host generator would take
minutes at S = 2048), with the distributions of ``synth.inputs``: weights N(0,
weight_std^2) in bf16, activations, caches and dOut N(0, 1), attention rows a causal
softmax of N(0, attn_logit_std^2) logits, LoRA A and B N(0, 0.02^2), h = x A^T, AdamW
moments zero.  Nothing here computes a gradient.
"""
from __future__ import annotations

import numpy as np

WEIGHTS = ("w_down", "w_gate", "w_up", "w_o", "w_q", "w_k", "w_v")


def to_dev(d: dict, wtype: str):
    """numpy inputs -> torch CUDA tensors (weights in their storage dtype)."""
    import torch
    out = {}
    for k, v in d.items():
        if not isinstance(v, np.ndarray):
            out[k] = v
            continue
        if k in WEIGHTS:
            if wtype == "bf16":
                out[k] = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to("cuda").to(torch.bfloat16)
            elif wtype == "ternary":
                out[k] = torch.from_numpy(np.ascontiguousarray(v, dtype=np.int8)).to("cuda")
            elif wtype == "ternary2":
                out[k] = torch.from_numpy(np.ascontiguousarray(v, dtype=np.uint8)).to("cuda")
            else:
                out[k] = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to("cuda")
        else:
            out[k] = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to("cuda")
    return out


def lora_dev(t: dict):
    """Copies of the adapter tensors and their moments, keyed the way the binding's
    lora() expects."""
    out = {}
    for tag in ("q", "v"):
        for k in ("a_", "b_", "m_a_", "v_a_", "m_b_", "v_b_"):
            out[k + tag] = t[k + tag].clone()
    return out


def device_layer(cfg, layer, seed=0):
    """One layer's weights, caches, adapters and dOut drawn on the device (bf16 weights)."""
    import torch
    g = torch.Generator(device="cuda")
    g.manual_seed(1000003 * seed + 7919 * layer + 17)
    S, L, H, I, qd, kvd, r = cfg.seq_len, cfg.cache_len, cfg.dim, cfg.ffn_dim, cfg.q_dim, cfg.kv_dim, cfg.rank
    n = lambda *shape, std=1.0: torch.randn(*shape, device="cuda", generator=g) * std
    t = {}
    wshapes = [("w_down", (I, H)), ("w_gate", (H, I)), ("w_up", (H, I)), ("w_o", (qd, H))]
    if getattr(cfg, "exact_din", False):
        wshapes += [("w_q", (H, qd)), ("w_k", (H, kvd)), ("w_v", (H, kvd))]
    for k, shape in wshapes:
        t[k] = n(*shape, std=cfg.weight_std).to(torch.bfloat16)
    for k, shape in (("x", (S, H)), ("gate", (S, I)), ("up", (S, I)), ("dout", (S, H)),
                     ("k", (L, kvd)), ("v", (L, kvd))):
        t[k] = n(*shape)
    t["silu_gate"] = torch.nn.functional.silu(t["gate"])
    pos0 = L - S
    mask = torch.arange(L, device="cuda")[None, :] > (pos0 + torch.arange(S, device="cuda"))[:, None]
    if getattr(cfg, "recompute_p", False):
        # queries after RoPE and each row's logsumexp of attn_scale q k^T over its keys; the
        # weights themselves are not kept (they are recomputed where they are used)
        t["q"] = n(S, qd)
        kh = t["k"].view(L, cfg.n_kv_heads, cfg.head_dim)
        lse = torch.empty(cfg.n_heads, S, device="cuda")
        grp = cfg.n_heads // cfg.n_kv_heads
        for h in range(cfg.n_heads):
            z = cfg.attn_scale * t["q"][:, h * cfg.head_dim:(h + 1) * cfg.head_dim] @ kh[:, h // grp, :].t()
            lse[h] = torch.logsumexp(z.masked_fill_(mask, float("-inf")), dim=-1)
        t["lse"] = lse
    else:
        attn = torch.empty(cfg.n_heads, S, L, device="cuda")
        for h in range(cfg.n_heads):
            logits = n(S, L, std=cfg.attn_logit_std).masked_fill_(mask, float("-inf"))
            attn[h] = torch.softmax(logits, dim=-1)
        t["attn"] = attn
    for k, shape in (("a_q", (r, H)), ("b_q", (qd, r)), ("a_v", (r, H)), ("b_v", (kvd, r))):
        t[k] = n(*shape, std=0.02)
        t["m_" + k] = torch.zeros_like(t[k])
        t["v_" + k] = torch.zeros_like(t[k])
    t["lora_q_h"] = t["x"] @ t["a_q"].t()
    t["lora_v_h"] = t["x"] @ t["a_v"].t()
    if cfg.qk_norm:                       # Q projection before the per-head norm, the norm's gain
        t["q_raw"] = n(S, qd)
        t["g_q"] = torch.rand(cfg.head_dim, device="cuda", generator=g) + 0.5
    if getattr(cfg, "exact_din", False):
        t["x_in"] = n(S, H)
        if "q" not in t:
            t["q"] = n(S, qd)
        if cfg.pre_norm:
            t["g_attn"] = torch.rand(H, device="cuda", generator=g) + 0.5
        if cfg.qk_norm:
            t["k_raw"] = n(S, kvd)
            t["g_k"] = torch.rand(cfg.head_dim, device="cuda", generator=g) + 0.5
    return t
