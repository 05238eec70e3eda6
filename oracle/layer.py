"""The layer backward composed from the single steps in ``oracle.ops``.

TEST INFRASTRUCTURE ONLY (see ``oracle.ops``).

``cfg`` is any object with the attributes of a layer configuration (shapes,
flags, hyperparameters); ``d`` holds the cached activations, weights and adapter
state of one layer as float arrays.  Order of the steps:

  FFN ([FFN] "Backward (reverse)"; [RS] backward_through_layers, "FFN backward")
    dF   = dOut W_down^T                         (scale of a ternary weight included)
    dh   = RMSNorm_bwd(hidden, g_sub_ffn, dF)    if the FFN sub-norm is on, else dF
    dG, dU = gated activation backward           (ReLU^2 x Mul or SiLU x Mul)
    dN2  = dG W_gate^T + dU W_up^T
    dR1  = dOut + RMSNorm_bwd(r1, g_ffn, dN2)    residual on, pre-norm on
           (no pre-norm: RMSNorm_bwd is the identity; residual off: dOut is not added,
            which is the overwrite the Rust trainer performs)
  attention ([ATT] "Gradient Flow"; [RS] "Attention backward")
    dSub = dR1 W_O^T
    dCtx = RMSNorm_bwd(ctx, g_sub_attn, dSub)    if the attention sub-norm is on
    per head h (KV head h // (n_heads / n_kv_heads)):
      dAttn = dCtx_h V^T;  dS = softmax_bwd(attn_h, dAttn);  dQ_h = scale dS K
      dV   += attn_h^T dCtx_h
    dQpre = RoPE_bwd(dQ) at positions L - S + i  (if RoPE is on)
    dQpre = RMSNorm_bwd(q_raw_h, g_q, dQpre_h) per head over head_dim  (if the QK-norm is
            on: [RS] LayerActivations caches q after a QK-norm and RoPE; q_raw is the Q
            projection output before the norm)
    dV rows kept: the S newest cache positions (the tokens of this call)
  LoRA ([RS] "LoRA Q backward", "LoRA V backward"; LoRA+ learning rate on B)
    Q adapter from dQpre, V adapter from dV, both with x = attn_input
    AdamW on A (lr) and B (lr * lr_b_mult); B is read before its update.
  d_in = dR1 (the gradient handed to the next layer down).

With ``cfg.exact_din`` (beyond the pages, which stop at the projection outputs) d_in
is the exact gradient of the layer input x_in, n1 = [RMSNorm(x_in; g_attn)]:
    dK_h  = scale dS_h^T Q_h summed over the group, rows of the S new positions, then
            RoPE_bwd and, with the QK-norm, RMSNorm_bwd(k_raw, g_k, .) per head
    dn1   = s_q dQpre W_Q^T + s_k dK W_K^T + s_v dV W_V^T + gh_q A_q + gh_v A_v
            (gh = s G B with B and A before their update: the LoRA-A paths)
    d_in  = [dR1] + [RMSNorm_bwd(x_in, g_attn, dn1)]        (residual, pre-norm)
"""
from __future__ import annotations

import numpy as np

from .ops import (adamw, apply_backward, attention_from_logsumexp, f64, linear_backward, lora_backward,
                  relu2_mul_backward, rmsnorm_backward, rope_backward, score_backward_k,
                  score_backward_q, silu_mul_backward, softmax_backward, unpack_ternary2,
                  value_backward)


def W(cfg, d, name) -> np.ndarray:
    """A weight matrix [in, out] as values (packed ternary storage decoded)."""
    w = d[name]
    return unpack_ternary2(w) if getattr(cfg, "wtype", "") == "ternary2" else w


def kv_heads_first(a, cfg) -> np.ndarray:
    """K or V cache as [n_kv, L, hd] whatever its stored layout."""
    a = f64(a)
    if cfg.kv_layout == "hsd":
        return a.reshape(cfg.n_kv_heads, cfg.cache_len, cfg.head_dim)
    return a.reshape(cfg.cache_len, cfg.n_kv_heads, cfg.head_dim).transpose(1, 0, 2)


def ffn_backward(cfg, d, dout) -> dict:
    eps = cfg.norm_eps
    dout = f64(dout)
    dF = linear_backward(dout, W(cfg, d, "w_down"), d["s_down"])
    dh = rmsnorm_backward(d["hidden"], d["g_sub_ffn"], dF, eps) if cfg.sub_norm else dF
    if cfg.act == "relu2_mul":
        dG, dU = relu2_mul_backward(d["gate"], d["up"], dh)
    else:
        sg = d.get("silu_gate") if cfg.use_silu_cache else None
        dG, dU = silu_mul_backward(d["gate"], d["up"], dh, sg)
    dN2 = linear_backward(dG, W(cfg, d, "w_gate"), d["s_gate"]) + linear_backward(dU, W(cfg, d, "w_up"), d["s_up"])
    dN2r = rmsnorm_backward(d["r1"], d["g_ffn"], dN2, eps) if cfg.pre_norm else dN2
    dR1 = dout + dN2r if cfg.residual else dN2r
    return dict(dF=dF, dh=dh, dG=dG, dU=dU, dN2=dN2, dR1=dR1)


def attn_backward(cfg, d, dR1) -> dict:
    S, L, nh, nkv, hd = cfg.seq_len, cfg.cache_len, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    dSub = linear_backward(dR1, W(cfg, d, "w_o"), d["s_o"])
    dCtx = rmsnorm_backward(d["ctx"], d["g_sub_attn"], dSub, cfg.norm_eps) if cfg.sub_norm else dSub
    K, V = kv_heads_first(d["k"], cfg), kv_heads_first(d["v"], cfg)
    if getattr(cfg, "recompute_p", False):      # the weights from q, K and each row's logsumexp
        attn = attention_from_logsumexp(f64(d["q"]).reshape(S, nh, hd), K, d["lse"], cfg.attn_scale, cfg.pos0,
                                        nkv)
    else:
        attn = f64(d["attn"])
    group = nh // nkv
    dQ = np.zeros((S, nh, hd))
    dS_all = np.zeros((nh, S, L))
    dV_all = np.zeros((nkv, L, hd))
    for h in range(nh):
        kvh = h // group
        dctx_h = dCtx[:, h * hd:(h + 1) * hd]
        dattn = apply_backward(dctx_h, V[kvh])
        dS = softmax_backward(attn[h], dattn)
        dS_all[h] = dS
        dQ[:, h, :] = score_backward_q(dS, K[kvh], cfg.attn_scale)
        dV_all[kvh] += value_backward(attn[h], dctx_h)
    pos = cfg.pos0 + np.arange(S)
    dQpre = rope_backward(dQ, pos, cfg.rope_base) if cfg.rope else dQ
    if getattr(cfg, "qk_norm", False):
        dQpre = rmsnorm_backward(f64(d["q_raw"]).reshape(S, nh, hd), d["g_q"], dQpre, cfg.norm_eps)
    dV = dV_all[:, cfg.pos0:, :].transpose(1, 0, 2).reshape(S, nkv * hd)
    out = dict(dSub=dSub, dCtx=dCtx, dS=dS_all, dQ=dQ.reshape(S, nh * hd),
               dQpre=dQpre.reshape(S, nh * hd), dV=dV)
    if getattr(cfg, "exact_din", False):
        # key gradient of the S new cache rows (the older rows are constants)
        Q = f64(d["q"]).reshape(S, nh, hd)
        dK_all = np.zeros((nkv, L, hd))
        for h in range(nh):
            dK_all[h // group] += score_backward_k(dS_all[h], Q[:, h, :], cfg.attn_scale)
        dK = dK_all[:, cfg.pos0:, :].transpose(1, 0, 2)                 # [S, nkv, hd]
        dKpre = rope_backward(dK, pos, cfg.rope_base) if cfg.rope else dK
        if getattr(cfg, "qk_norm", False):
            dKpre = rmsnorm_backward(f64(d["k_raw"]).reshape(S, nkv, hd), d["g_k"], dKpre, cfg.norm_eps)
        out["dKpre"] = dKpre.reshape(S, nkv * hd)
    return out


def input_backward(cfg, d, r) -> np.ndarray:
    """Exact layer-input gradient (``cfg.exact_din``): the attention input n1 feeds the
    Q, K and V projections and both LoRA A products; x_in reaches r1 through the
    residual and n1 through the attention pre-norm."""
    dn1 = (linear_backward(r["dQpre"], W(cfg, d, "w_q"), d.get("s_q", 1.0)) +
           linear_backward(r["dKpre"], W(cfg, d, "w_k"), d.get("s_k", 1.0)) +
           linear_backward(r["dV"], W(cfg, d, "w_v"), d.get("s_v", 1.0)) +
           r["gh_q"] @ f64(d["a_q"]) + r["gh_v"] @ f64(d["a_v"]))
    dx = rmsnorm_backward(d["x_in"], d["g_attn"], dn1, cfg.norm_eps) if cfg.pre_norm else dn1
    return r["dR1"] + dx if cfg.residual else dx


def lora_adamw(cfg, d, dQpre, dV) -> dict:
    out = {}
    for tag, g in (("q", dQpre), ("v", dV)):
        da, db, gh = lora_backward(g, d["lora_%s_h" % tag], d["x"], d["b_" + tag],
                                   cfg.lora_alpha, cfg.rank)
        out["dA_" + tag], out["dB_" + tag], out["gh_" + tag] = da, db, gh
        for p, grad, lr in (("a_" + tag, da, cfg.lr), ("b_" + tag, db, cfg.lr * cfg.lr_b_mult)):
            out[p], out["m_" + p], out["v_" + p] = adamw(
                d[p], grad, d["m_" + p], d["v_" + p], lr, cfg.beta1, cfg.beta2,
                cfg.adam_eps, cfg.weight_decay, cfg.step)
    out["sumsq_a"] = float(np.sum(out["dA_q"] ** 2) + np.sum(out["dA_v"] ** 2))
    out["sumsq_b"] = float(np.sum(out["dB_q"] ** 2) + np.sum(out["dB_v"] ** 2))
    return out


def layer_backward(cfg, d, dout) -> dict:
    r = ffn_backward(cfg, d, dout)
    r.update(attn_backward(cfg, d, r["dR1"]))
    r.update(lora_adamw(cfg, d, r["dQpre"], r["dV"]))
    r["d_in"] = input_backward(cfg, d, r) if getattr(cfg, "exact_din", False) else r["dR1"]
    return r


def stack_backward(cfg, layers, dout, keep=lambda name: True) -> dict:
    """Reverse loop over ``layers`` ([RS] backward_through_layers): the input gradient of
    layer l becomes the output gradient of layer l-1.  The returned gnorm is
    sqrt(sum of ||dA||^2) over every layer and both adapters, as the trainer reports it.
    ``keep`` filters which per-layer results are retained."""
    per_layer = [None] * len(layers)
    sa = sb = 0.0
    g = f64(dout)
    for li in reversed(range(len(layers))):
        r = layer_backward(cfg, layers[li], g)
        g = r["d_in"]
        sa += r["sumsq_a"]
        sb += r["sumsq_b"]
        per_layer[li] = {k: v for k, v in r.items() if keep(k)}
    return dict(layers=per_layer, d_in=g, sumsq_a=sa, sumsq_b=sb, gnorm=float(np.sqrt(sa)),
                gnorm_full=float(np.sqrt(sa + sb)))
