"""Seeded synthetic inputs for one layer backward (or a stack of them).

Every tensor comes from its own SplitMix64 stream keyed by
``(seed, config name, layer, tensor name)``.  The arrays returned are the exact
values both sides receive: float32 activations, weights in their storage type
(float32, bfloat16-exact float32, or int8 ternary), float32 scales.

Recipe (distributions follow the workload descriptions):
  * weights ~ N(0, weight_std^2) (bf16 configs: rounded to bfloat16);
    ternary weights take 0 with probability 1/3 and +-1 otherwise, with one
    per-tensor scale ~ U(0.5, 2);
  * LoRA A ~ N(0, lora_a_std^2), B ~ N(0, lora_b_std^2); AdamW moments zero
    (first step) or, for the warm case, m ~ N(0, 1e-2^2), v ~ U(0, 1e-4);
  * RMSNorm gammas ~ U(0.5, 1.5);
  * cached activations, K/V cache and the upstream gradient ~ N(0, 1);
  * attention rows: softmax of N(0, attn_logit_std^2) logits over the keys a
    query may see (key j visible to query i iff j <= L - S + i), zero elsewhere;
  * the cached SiLU output is silu(gate) and the cached LoRA activations are
    x @ A^T, both formed in float64 from the values above and then rounded;
  * with the QK-norm, the Q projection before it ~ N(0, 1) and its gain ~ U(0.5, 1.5);
  * with the attention recomputed: the queries after RoPE ~ N(0, 1) and each row's
    logsumexp of attn_scale q k^T over its visible keys (the cached weights are then that
    softmax too);
  * for the exact layer-input gradient: W_Q, W_K, W_V like the other weights, the layer
    input, the cached (rotated) q and, with the QK-norm, the new rows of k before it
    ~ N(0, 1), and the attention pre-norm and k-norm gains ~ U(0.5, 1.5).
"""
from __future__ import annotations

import numpy as np

from .configs import LayerConfig
from . import rng


def _n(seed, cfg, layer, name, shape, std=1.0):
    n = int(np.prod(shape))
    return rng.normal(rng.stream_key(seed, cfg.name, layer, name), n, 0.0, std).reshape(shape)


def _u(seed, cfg, layer, name, shape, lo, hi):
    n = int(np.prod(shape))
    return rng.uniform(rng.stream_key(seed, cfg.name, layer, name), n, lo, hi).reshape(shape)


def pack_ternary2(w: np.ndarray) -> np.ndarray:
    """Packed storage of a ternary [in, out] int8 matrix (out a multiple of 4): uint8 [in,
    out / 4], weight 4k + i of a row in bits 2i, 2i + 1 of byte k as the code w + 1."""
    w = np.asarray(w)
    assert w.shape[-1] % 4 == 0 and np.all(np.abs(w) <= 1)
    code = (w.astype(np.int16) + 1).astype(np.uint8)
    c = code.reshape(w.shape[:-1] + (w.shape[-1] // 4, 4))
    return (c[..., 0] | (c[..., 1] << 2) | (c[..., 2] << 4) | (c[..., 3] << 6)).astype(np.uint8)


def _weight(seed, cfg, layer, name, shape):
    """Returns (stored array, scale)."""
    if cfg.wtype in ("ternary", "ternary2"):
        w = rng.ternary(rng.stream_key(seed, cfg.name, layer, name), int(np.prod(shape)))
        scale = float(np.float32(_u(seed, cfg, layer, name + ".scale", (1,), 0.5, 2.0)[0]))
        w = w.reshape(shape)
        return (pack_ternary2(w) if cfg.wtype == "ternary2" else w), scale
    w = _n(seed, cfg, layer, name, shape, cfg.weight_std)
    if cfg.wtype == "bf16":
        return rng.round_to_bf16(w), 1.0
    return w.astype(np.float32), 1.0


def attention_rows(seed, cfg: LayerConfig, layer: int) -> np.ndarray:
    """[n_heads, S, L] float32 rows of a masked softmax of normal logits."""
    S, L, nh = cfg.seq_len, cfg.cache_len, cfg.n_heads
    logits = _n(seed, cfg, layer, "attn_logits", (nh, S, L), cfg.attn_logit_std)
    vis = np.arange(L)[None, :] <= (cfg.pos0 + np.arange(S))[:, None]      # [S, L]
    logits = np.where(vis[None], logits, -np.inf)
    logits -= logits.max(axis=-1, keepdims=True)
    e = np.exp(logits)
    return (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)


def layer_inputs(cfg: LayerConfig, layer: int = 0, seed: int = 0, with_dout: bool = True) -> dict:
    S, L, H, I = cfg.seq_len, cfg.cache_len, cfg.dim, cfg.ffn_dim
    qd, kvd, r = cfg.q_dim, cfg.kv_dim, cfg.rank
    f32 = np.float32
    d: dict = {}
    # weights, stored [in, out]
    d["w_down"], d["s_down"] = _weight(seed, cfg, layer, "w_down", (I, H))
    d["w_gate"], d["s_gate"] = _weight(seed, cfg, layer, "w_gate", (H, I))
    d["w_up"], d["s_up"] = _weight(seed, cfg, layer, "w_up", (H, I))
    d["w_o"], d["s_o"] = _weight(seed, cfg, layer, "w_o", (qd, H))
    if cfg.sub_norm:
        d["g_sub_ffn"] = _u(seed, cfg, layer, "g_sub_ffn", (I,), 0.5, 1.5).astype(f32)
        d["g_sub_attn"] = _u(seed, cfg, layer, "g_sub_attn", (qd,), 0.5, 1.5).astype(f32)
    if cfg.pre_norm:
        d["g_ffn"] = _u(seed, cfg, layer, "g_ffn", (H,), 0.5, 1.5).astype(f32)
    # cached activations
    d["x"] = _n(seed, cfg, layer, "attn_input", (S, H)).astype(f32)
    d["gate"] = _n(seed, cfg, layer, "gate", (S, I)).astype(f32)
    d["up"] = _n(seed, cfg, layer, "up", (S, I)).astype(f32)
    if cfg.act == "silu_mul" and cfg.use_silu_cache:
        g = d["gate"].astype(np.float64)
        d["silu_gate"] = (g / (1.0 + np.exp(-g))).astype(f32)
    if cfg.sub_norm:
        d["hidden"] = _n(seed, cfg, layer, "hidden", (S, I)).astype(f32)
        d["ctx"] = _n(seed, cfg, layer, "context", (S, qd)).astype(f32)
    if cfg.pre_norm:
        d["r1"] = _n(seed, cfg, layer, "resid1", (S, H)).astype(f32)
    kshape = (L, kvd) if cfg.kv_layout == "shd" else (cfg.n_kv_heads, L, cfg.head_dim)
    d["k"] = _n(seed, cfg, layer, "k_cache", kshape).astype(f32)
    d["v"] = _n(seed, cfg, layer, "v_cache", kshape).astype(f32)
    if cfg.recompute_p:
        # queries after RoPE and the logsumexp of each row's scaled logits over the keys it
        # sees (the forward's softmax statistics); the cached weights are the same softmax
        q = _n(seed, cfg, layer, "q_cache", (S, qd)).astype(f32)
        d["q"] = q
        kh = (d["k"].reshape(L, cfg.n_kv_heads, cfg.head_dim).transpose(1, 0, 2) if cfg.kv_layout == "shd"
              else d["k"]).astype(np.float64)
        qh = q.astype(np.float64).reshape(S, cfg.n_heads, cfg.head_dim)
        vis = np.arange(L)[None, :] <= (cfg.pos0 + np.arange(S))[:, None]
        lse = np.zeros((cfg.n_heads, S))
        attn = np.zeros((cfg.n_heads, S, L))
        g = cfg.n_heads // cfg.n_kv_heads
        for h in range(cfg.n_heads):
            z = np.where(vis, cfg.attn_scale * qh[:, h, :] @ kh[h // g].T, -np.inf)
            m = z.max(axis=-1, keepdims=True)
            lse[h] = (m + np.log(np.exp(z - m).sum(axis=-1, keepdims=True)))[:, 0]
            attn[h] = np.exp(z - lse[h][:, None])
        d["lse"] = lse.astype(f32)
        d["attn"] = attn.astype(f32)
    else:
        d["attn"] = attention_rows(seed, cfg, layer)
    if cfg.qk_norm:
        d["q_raw"] = _n(seed, cfg, layer, "q_raw", (S, qd)).astype(f32)
        d["g_q"] = _u(seed, cfg, layer, "g_q", (cfg.head_dim,), 0.5, 1.5).astype(f32)
    if cfg.exact_din:
        d["w_q"], d["s_q"] = _weight(seed, cfg, layer, "w_q", (H, qd))
        d["w_k"], d["s_k"] = _weight(seed, cfg, layer, "w_k", (H, kvd))
        d["w_v"], d["s_v"] = _weight(seed, cfg, layer, "w_v", (H, kvd))
        d["x_in"] = _n(seed, cfg, layer, "layer_input", (S, H)).astype(f32)
        if "q" not in d:
            d["q"] = _n(seed, cfg, layer, "q_cache", (S, qd)).astype(f32)
        if cfg.pre_norm:
            d["g_attn"] = _u(seed, cfg, layer, "g_attn", (H,), 0.5, 1.5).astype(f32)
        if cfg.qk_norm:
            d["k_raw"] = _n(seed, cfg, layer, "k_raw", (S, kvd)).astype(f32)
            d["g_k"] = _u(seed, cfg, layer, "g_k", (cfg.head_dim,), 0.5, 1.5).astype(f32)
    # LoRA adapters and their AdamW state
    d["a_q"] = _n(seed, cfg, layer, "lora_a_q", (r, H), cfg.lora_a_std).astype(f32)
    d["b_q"] = _n(seed, cfg, layer, "lora_b_q", (qd, r), cfg.lora_b_std).astype(f32)
    d["a_v"] = _n(seed, cfg, layer, "lora_a_v", (r, H), cfg.lora_a_std).astype(f32)
    d["b_v"] = _n(seed, cfg, layer, "lora_b_v", (kvd, r), cfg.lora_b_std).astype(f32)
    for p in ("a_q", "b_q", "a_v", "b_v"):
        if cfg.adam_state == "warm":
            d["m_" + p] = _n(seed, cfg, layer, "m_" + p, d[p].shape, 1e-2).astype(f32)
            d["v_" + p] = _u(seed, cfg, layer, "v_" + p, d[p].shape, 0.0, 1e-4).astype(f32)
        else:
            d["m_" + p] = np.zeros_like(d[p])
            d["v_" + p] = np.zeros_like(d[p])
    x64 = d["x"].astype(np.float64)
    d["lora_q_h"] = (x64 @ d["a_q"].astype(np.float64).T).astype(f32)
    d["lora_v_h"] = (x64 @ d["a_v"].astype(np.float64).T).astype(f32)
    if with_dout:
        d["dout"] = _n(seed, cfg, layer, "grad_out", (S, H)).astype(f32)
    return d


def layer_inputs_sample(cfg: LayerConfig, seed: int = 0) -> dict:
    """A full-size draw for CPU timing samples only: the tensors of ``layer_inputs`` with
    the same shapes and distributions, drawn with numpy's PCG64 (``layer_inputs`` takes
    minutes at S = 2048 on the host).  The values differ from ``layer_inputs``; no parity
    check reads them."""
    S, L, H, I = cfg.seq_len, cfg.cache_len, cfg.dim, cfg.ffn_dim
    qd, kvd, r = cfg.q_dim, cfg.kv_dim, cfg.rank
    g = np.random.default_rng(seed)
    f32 = np.float32
    n = lambda shape, std=1.0: (g.standard_normal(shape, dtype=f32) * f32(std))
    d: dict = {}
    for k, shape in (("w_down", (I, H)), ("w_gate", (H, I)), ("w_up", (H, I)), ("w_o", (qd, H))):
        w = n(shape, cfg.weight_std)
        if cfg.wtype == "bf16":                 # round to nearest bfloat16 (finite values)
            b = w.view(np.uint32)
            b += np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
            b &= np.uint32(0xFFFF0000)
        d[k] = w
        d["s_" + k[2:]] = 1.0
    for k, shape in (("x", (S, H)), ("gate", (S, I)), ("up", (S, I)), ("dout", (S, H))):
        d[k] = n(shape)
    d["silu_gate"] = (d["gate"] / (1.0 + np.exp(-d["gate"]))).astype(f32)
    kshape = (L, kvd) if cfg.kv_layout == "shd" else (cfg.n_kv_heads, L, cfg.head_dim)
    d["k"], d["v"] = n(kshape), n(kshape)
    vis = np.arange(L)[None, :] <= (cfg.pos0 + np.arange(S))[:, None]
    attn = np.empty((cfg.n_heads, S, L), dtype=f32)
    for h in range(cfg.n_heads):
        lg = np.where(vis, n((S, L), cfg.attn_logit_std), -np.inf)
        lg -= lg.max(axis=-1, keepdims=True)
        np.exp(lg, out=lg)
        attn[h] = lg / lg.sum(axis=-1, keepdims=True)
    d["attn"] = attn
    for p, shape in (("a_q", (r, H)), ("b_q", (qd, r)), ("a_v", (r, H)), ("b_v", (kvd, r))):
        d[p] = n(shape, 0.02)
        d["m_" + p] = np.zeros_like(d[p])
        d["v_" + p] = np.zeros_like(d[p])
    d["lora_q_h"] = d["x"] @ d["a_q"].T
    d["lora_v_h"] = d["x"] @ d["a_v"].T
    if cfg.exact_din:
        for k, shape in (("w_q", (H, qd)), ("w_k", (H, kvd)), ("w_v", (H, kvd))):
            d[k], d["s_" + k[2:]] = n(shape, cfg.weight_std), 1.0
        d["x_in"], d["q"] = n((S, H)), n((S, qd))
        if cfg.pre_norm:
            d["g_attn"] = g.uniform(0.5, 1.5, H).astype(f32)
    return d


def row_slice(cfg: LayerConfig, d: dict, r0: int, r1: int):
    """Query rows r0 .. r1-1 of a layer problem as a problem of their own: S = r1 - r0
    rows over the first L = pos0 + r1 cache entries (the keys those rows may see).  The
    slices of a partition of the rows together hold exactly the layer's work."""
    L = cfg.pos0 + r1
    sub = cfg.with_(seq_len=r1 - r0, cache_len=L)
    rows = ("x", "gate", "up", "silu_gate", "dout", "lora_q_h", "lora_v_h", "hidden", "r1", "ctx",
            "q_raw", "x_in", "q", "k_raw")
    out = {}
    for k, v in d.items():
        if k in rows:
            out[k] = v[r0:r1]
        elif k in ("k", "v"):
            out[k] = v[:L] if cfg.kv_layout == "shd" else v[:, :L]
        elif k == "attn":
            out[k] = v[:, r0:r1, :L]
        else:
            out[k] = v
    return sub, out


def stack_dout(cfg: LayerConfig, seed: int = 0) -> np.ndarray:
    """Upstream gradient entering the top layer of a stack, [S, H] ~ N(0, 1)."""
    return _n(seed, cfg, "top", "grad_hidden", (cfg.seq_len, cfg.dim)).astype(np.float32)


def vector(seed: int, name: str, n: int, dist: str = "normal") -> np.ndarray:
    """Float32 vector for standalone kernel cases (``dist``: normal, or 'u01')."""
    key = rng.stream_key(seed, "vector", name)
    if dist == "u01":
        return rng.uniform(key, n).astype(np.float32)
    return rng.normal(key, n).astype(np.float32)
