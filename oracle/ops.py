"""Single steps of the LoRA layer backward, in float64 numpy, one function per step.

TEST INFRASTRUCTURE ONLY: this module is the oracle the CUDA library is checked
against.  Only the tests, the package smoke check and the benchmark's CPU
baseline may import it; the product path never does.

Every function is the plain definition of its step as the pages state it.  All
inputs are widened to float64 first; nothing is blocked, fused or reordered.
Sources (page, section):
  [FFN]  Hesper API, "Hesper/Training/FFNBackward" ("FFN Backward GPU Kernels")
  [ATT]  Hesper API, "Hesper/Training/AttentionBackward" ("Attention Backward GPU Kernels")
  [RS]   entrenar "train/transformer_trainer/wgpu_backward.rs" (aprender-train 0.34.0)
"""
from __future__ import annotations

import numpy as np


def f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def unpack_ternary2(packed) -> np.ndarray:
    """Ternary weights [in, out] from their packed storage [in, out / 4] (uint8): four
    2-bit codes per byte along the row, the first weight in the lowest two bits; a code
    is the weight plus one (0 is -1, 1 is 0, 2 is +1: the BitLinear weight of [FFN],
    stored four to a byte).  Code 3 is not a ternary value and is refused."""
    b = np.asarray(packed, dtype=np.uint8)
    codes = np.stack([(b >> (2 * i)) & 3 for i in range(4)], axis=-1)      # [..., out/4, 4]
    if np.any(codes == 3):
        raise ValueError("code 3 in packed ternary weights")
    value = np.array([-1.0, 0.0, 1.0])
    return value[codes].reshape(b.shape[:-1] + (b.shape[-1] * 4,))


def attention_from_logsumexp(q, K, lse, scale: float, pos0: int, n_kv: int) -> np.ndarray:
    """Attention weights [nh, S, L] recomputed from the queries q [S, nh, hd] (after RoPE),
    the key cache K [n_kv, L, hd] and each row's logsumexp lse [nh, S]:
    attn[h, i, j] = exp(scale q_i,h . k_j - lse[h, i]) for j <= pos0 + i, else 0 (the
    softmax of the forward, given its normaliser; GQA head h reads KV head h // (nh / n_kv))."""
    q, K, lse = f64(q), f64(K), f64(lse)
    S, nh, hd = q.shape
    L = K.shape[1]
    vis = np.arange(L)[None, :] <= (pos0 + np.arange(S))[:, None]
    out = np.zeros((nh, S, L))
    g = nh // n_kv
    for h in range(nh):
        out[h] = np.where(vis, np.exp(scale * q[:, h, :] @ K[h // g].T - lse[h][:, None]), 0.0)
    return out


def linear_backward(dy, w, scale: float = 1.0) -> np.ndarray:
    """Input gradient of y = x @ (scale * W) with W stored [in, out]: dX = scale * dY @ W^T.

    [FFN] "Backward (reverse)": the W_down^T, W_gate^T and W_up^T products;
    [ATT] "Gradient Flow": the O-projection (BitLinear transpose);
    [RS] backward_through_layers, gemm_backward_a calls (C = A @ B^T with the
    weight stored pre-transposed).  A ternary BitLinear weight is scale * W.
    """
    return float(scale) * (f64(dy) @ f64(w).T)


def rmsnorm_backward(x, gamma, dy, eps: float) -> np.ndarray:
    """[ATT] "RMSNorm Backward": dx = (1/rms) (dy*g - x * dot(dy*g, x) / (n rms^2)).

    rms = sqrt(mean(x^2) + eps) over the last axis; each row is independent.
    """
    x, gamma, dy = f64(x), f64(gamma), f64(dy)
    n = x.shape[-1]
    rms = np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    dyg = dy * gamma
    dot = np.sum(dyg * x, axis=-1, keepdims=True)
    return (dyg - x * dot / (n * rms * rms)) / rms


def relu2_mul_backward(gate, up, dh):
    """[FFN] "ReLU^2 x Mul Backward": dGate = dH*up*2*max(0,g), dUp = dH*max(0,g)^2."""
    gate, up, dh = f64(gate), f64(up), f64(dh)
    r = np.maximum(0.0, gate)
    return dh * up * 2.0 * r, dh * r * r


def silu_mul_backward(gate, up, dsw, silu_gate=None):
    """[RS] backward_through_layers, "SiLU backward" block.

    sig = 1/(1+exp(-x)), y = x*sig, silu' = sig*(1 + x - y);
    dGate = dSw*up*silu', dUp = dSw*silu(gate) (the cached silu output when given).
    """
    x, up, dsw = f64(gate), f64(up), f64(dsw)
    sig = 1.0 / (1.0 + np.exp(-x))
    y = x * sig
    silu_prime = sig * (1.0 + x - y)
    s = y if silu_gate is None else f64(silu_gate)
    return dsw * up * silu_prime, dsw * s


def softmax_backward(attn, dattn) -> np.ndarray:
    """[ATT] "Softmax Backward": dS[h,s] = attn[h,s] (dAttn[h,s] - sum_s' attn[h,s'] dAttn[h,s'])."""
    attn, dattn = f64(attn), f64(dattn)
    dot = np.sum(attn * dattn, axis=-1, keepdims=True)
    return attn * (dattn - dot)


def apply_backward(dctx_h, v_h) -> np.ndarray:
    """[ATT] "Attention Apply Backward": dAttn[s] = sum_d dOutput[d] V[s, d] (one head; rows = queries)."""
    return f64(dctx_h) @ f64(v_h).T


def score_backward_q(dscores_h, k_h, scale: float) -> np.ndarray:
    """[ATT] "Attention Score Backward": dQ[d] = scale * sum_s dScores[s] K[s, d] (one head)."""
    return float(scale) * (f64(dscores_h) @ f64(k_h))


def score_backward_k(dscores_h, q_h, scale: float) -> np.ndarray:
    """Key gradient of scores = scale * q k^T (one head): dK[s] = scale * sum_q dScores[q, s] q[q].

    The pages stop the backward at the Q / V projection outputs and print no key
    gradient; this is the plain derivative, used only for the exact layer-input gradient.
    """
    return float(scale) * (f64(dscores_h).T @ f64(q_h))


def value_backward(attn_h, dctx_h) -> np.ndarray:
    """[RS] attention block: grad_v[k] += attn[q, k] * grad_context[q], summed over queries q."""
    return f64(attn_h).T @ f64(dctx_h)


def rope_angles(pos, head_dim: int, base: float) -> np.ndarray:
    """[ATT] "RoPE Backward": theta = pos * base^(-2d/headDim) for d in [0, headDim/2)."""
    pos = f64(pos).reshape(-1, 1)
    d = np.arange(head_dim // 2, dtype=np.float64).reshape(1, -1)
    return pos * np.power(float(base), -2.0 * d / head_dim)


def rope_backward(dy, pos, base: float) -> np.ndarray:
    """[ATT] "RoPE Backward (inverse rotation)", NeoX split-half layout.

    dy has shape [rows, heads, head_dim]; row r sits at position pos[r].
      dx[d]      =  dy[d] cos(theta) + dy[d+half] sin(theta)
      dx[d+half] = -dy[d] sin(theta) + dy[d+half] cos(theta)
    """
    dy = f64(dy)
    hd = dy.shape[-1]
    half = hd // 2
    th = rope_angles(pos, hd, base)[:, None, :]            # [rows, 1, half]
    c, s = np.cos(th), np.sin(th)
    y1, y2 = dy[..., :half], dy[..., half:]
    return np.concatenate([y1 * c + y2 * s, -y1 * s + y2 * c], axis=-1)


def lora_backward(g, h, x, b, alpha: float, rank: int):
    """[RS] "LoRA Q backward" / "LoRA V backward" blocks, with scaling = alpha / rank.

    dB[o, r] = scaling * sum_s G[s, o] h[s, r]
    gh[s, r] = scaling * sum_o G[s, o] B[o, r]        (B before its update)
    dA[r, i] = sum_s gh[s, r] x[s, i]
    Returns (dA, dB, gh).
    """
    g, h, x, b = f64(g), f64(h), f64(x), f64(b)
    scaling = float(alpha) / float(rank)
    db = scaling * (g.T @ h)
    gh = scaling * (g @ b)
    da = gh.T @ x
    return da, db, gh


def adamw(p, g, m, v, lr, beta1, beta2, eps, wd, step: int):
    """[RS] cpu_adamw: one AdamW step with bias correction 1/(1 - beta^t).

    m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g^2;
    p -= lr * (m*bc1 / (sqrt(v*bc2) + eps) + wd * p).   Returns (p, m, v).
    """
    p, g, m, v = f64(p), f64(g), f64(m), f64(v)
    bc1 = 1.0 / (1.0 - float(beta1) ** int(step))
    bc2 = 1.0 / (1.0 - float(beta2) ** int(step))
    m = beta1 * m + (1.0 - beta1) * g
    v = beta2 * v + (1.0 - beta2) * g * g
    p = p - lr * ((m * bc1) / (np.sqrt(v * bc2) + eps) + wd * p)
    return p, m, v
