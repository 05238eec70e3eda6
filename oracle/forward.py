"""Consistent float64 forward of the layer the backward differentiates.

TEST INFRASTRUCTURE ONLY: used by the finite-difference pins of the oracle.  It
assembles the forward the pages describe ([FFN] "Forward"; [ATT] "Gradient
Flow", read in forward order; [RS] LayerActivations) for S query rows at
positions L - S .. L - 1 over a cache of L keys:

  h_q = n1 A_q^T             q = RoPE([QKNorm](n1 W_Q + s h_q B_q^T))      s = alpha / rank
  k   = RoPE([QKNorm](n1 W_K))                h_v = n1 A_v^T      v = n1 W_V + s h_v B_v^T
      (QKNorm: RMSNorm of each head's head_dim values, gains g_q and g_k of length
       head_dim shared by the heads, when the QK-norm is on; [RS] LayerActivations caches
       q and k after it and RoPE)
  P   = softmax(scale q k^T) over keys j <= position(i)          ctx = P v (per head, GQA)
  a   = [RMSNorm(ctx; g_sub_attn)] (s_o W_O)                     r1 = [x +] a
  n2  = [RMSNorm(r1; g_ffn)]   gate = n2 s_g W_g   up = n2 s_u W_u   hid = act(gate) up
  out = [r1 +] [RMSNorm(hid; g_sub_ffn)] (s_d W_d)

n1 (the normalised attention input) is an independent input here: the pages stop
the gradient at the Q/V projection outputs, so the backward treats n1 as a
constant.  ``r1_delta`` adds a perturbation to r1 so that finite differences can
reach the gradient the backward hands to the layer below.  With ``cfg.exact_din``
n1 = [RMSNorm(x_in; g_attn)] instead, so that finite differences in x_in reach the
exact layer-input gradient (cached k for the S new positions depends on x_in too).
"""
from __future__ import annotations

import numpy as np

from .ops import f64


def rmsnorm(x, gamma, eps):
    x = f64(x)
    rms = np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return x / rms * f64(gamma)


def rope(x, pos, base):
    """Forward NeoX rotation R(theta) of x [rows, heads, hd]."""
    x = f64(x)
    hd = x.shape[-1]
    half = hd // 2
    d = np.arange(half, dtype=np.float64)
    th = (f64(pos).reshape(-1, 1) * np.power(float(base), -2.0 * d / hd))[:, None, :]
    c, s = np.cos(th), np.sin(th)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x1 * s + x2 * c], axis=-1)


def gated(gate, up, act):
    g = f64(gate)
    if act == "relu2_mul":
        return np.maximum(0.0, g) ** 2 * f64(up)
    return g / (1.0 + np.exp(-g)) * f64(up)


def layer_forward(cfg, p, n1, x_in, k_prev, v_prev, r1_delta=None):
    """Returns (out [S, H], cache dict in the layouts the backward reads).

    ``p`` holds float64 weights w_q [H, q_dim], w_k/w_v [H, kv_dim], w_o, w_gate,
    w_up, w_down (stored [in, out]) with scales s_o, s_gate, s_up, s_down, the
    gammas and the adapters a_q, b_q, a_v, b_v.  ``k_prev``/``v_prev`` are the
    [n_kv, L - S, hd] cache entries of earlier positions (k already rotated).
    """
    S = n1.shape[0]
    nh, nkv, hd = cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    pos = cfg.pos0 + np.arange(S)
    s = cfg.lora_alpha / cfg.rank
    exact = getattr(cfg, "exact_din", False)
    if exact:
        n1 = rmsnorm(x_in, p["g_attn"], cfg.norm_eps) if cfg.pre_norm else f64(x_in)
    n1 = f64(n1)
    hq = n1 @ f64(p["a_q"]).T
    q = (n1 @ (p.get("s_q", 1.0) * f64(p["w_q"])) + s * hq @ f64(p["b_q"]).T).reshape(S, nh, hd)
    k = (n1 @ (p.get("s_k", 1.0) * f64(p["w_k"]))).reshape(S, nkv, hd)
    q_raw = q.reshape(S, nh * hd)
    k_raw = k.reshape(S, nkv * hd)
    if cfg.qk_norm:
        q, k = rmsnorm(q, p["g_q"], cfg.norm_eps), rmsnorm(k, p["g_k"], cfg.norm_eps)
    if cfg.rope:
        q, k = rope(q, pos, cfg.rope_base), rope(k, pos, cfg.rope_base)
    hv = n1 @ f64(p["a_v"]).T
    v = (n1 @ (p.get("s_v", 1.0) * f64(p["w_v"])) + s * hv @ f64(p["b_v"]).T).reshape(S, nkv, hd)
    K = np.concatenate([f64(k_prev), k.transpose(1, 0, 2)], axis=1)       # [nkv, L, hd]
    V = np.concatenate([f64(v_prev), v.transpose(1, 0, 2)], axis=1)
    L = K.shape[1]
    vis = np.arange(L)[None, :] <= pos[:, None]
    P = np.zeros((nh, S, L))
    ctx = np.zeros((S, nh, hd))
    group = nh // nkv
    for h in range(nh):
        kvh = h // group
        logits = cfg.attn_scale * q[:, h, :] @ K[kvh].T
        logits = np.where(vis, logits, -np.inf)
        e = np.exp(logits - logits.max(axis=-1, keepdims=True))
        P[h] = e / e.sum(axis=-1, keepdims=True)
        ctx[:, h, :] = P[h] @ V[kvh]
    ctx = ctx.reshape(S, nh * hd)
    c = rmsnorm(ctx, p["g_sub_attn"], cfg.norm_eps) if cfg.sub_norm else ctx
    a = c @ (p["s_o"] * f64(p["w_o"]))
    r1 = f64(x_in) + a if cfg.residual else a
    if r1_delta is not None:
        r1 = r1 + r1_delta
    n2 = rmsnorm(r1, p["g_ffn"], cfg.norm_eps) if cfg.pre_norm else r1
    gate = n2 @ (p["s_gate"] * f64(p["w_gate"]))
    up = n2 @ (p["s_up"] * f64(p["w_up"]))
    hid = gated(gate, up, cfg.act)
    fin = rmsnorm(hid, p["g_sub_ffn"], cfg.norm_eps) if cfg.sub_norm else hid
    f = fin @ (p["s_down"] * f64(p["w_down"]))
    out = r1 + f if cfg.residual else f
    if cfg.kv_layout == "hsd":
        kc, vc = K, V
    else:
        kc = K.transpose(1, 0, 2).reshape(L, nkv * hd)
        vc = V.transpose(1, 0, 2).reshape(L, nkv * hd)
    cache = dict(x=n1, gate=gate, up=up, silu_gate=f64(gate) / (1.0 + np.exp(-f64(gate))),
                 hidden=hid, r1=r1, ctx=ctx, k=kc, v=vc, attn=P, lora_q_h=hq, lora_v_h=hv,
                 q_raw=q_raw, k_raw=k_raw, q=q.reshape(S, nh * hd), x_in=f64(x_in))
    return out, cache


def stack_forward(cfg, params, n1s, x_in, k_prevs, v_prevs):
    """Layers 0 .. n-1 applied in order ([RS] backward_through_layers runs them in reverse):
    layer l's output is layer l+1's input x_in (its residual input and, with
    ``cfg.exact_din``, the input of its attention pre-norm).  Without ``exact_din`` each
    layer's n1 is its own independent input, as in ``layer_forward``.
    Returns (output of the last layer, [cache of each layer])."""
    x = f64(x_in)
    caches = []
    for l in range(len(params)):
        x, c = layer_forward(cfg, params[l], n1s[l], x, k_prevs[l], v_prevs[l])
        caches.append(c)
    return x, caches
