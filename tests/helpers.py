"""Shared test utilities: moving synthetic inputs to the GPU and comparing results.

Tolerances (the stated parity bar):
  * float32 paths: relative L2 <= 1e-5 and max-abs <= 1e-4.  Max-abs is applied to
    the difference divided by max(1, rms(reference)), so O(1) tensors get the
    absolute bound and large-magnitude tensors (sums over thousands of terms) a
    bound relative to their own scale, where float32 rounding of the values alone
    exceeds 1e-4;
  * bf16 tensor-core paths: relative L2 <= 5e-3.
"""
from __future__ import annotations

import numpy as np

F32_REL_L2 = 1e-5
F32_MAX_ABS = 1e-4
BF16_REL_L2 = 5e-3

WEIGHTS = ("w_down", "w_gate", "w_up", "w_o")


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
            else:
                out[k] = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to("cuda")
        else:
            out[k] = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to("cuda")
    return out


def host(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def errors(gpu, ref):
    g = np.asarray(gpu, dtype=np.float64).ravel()
    r = np.asarray(ref, dtype=np.float64).ravel()
    if r.size == 0:
        return 0.0, 0.0
    nr = np.linalg.norm(r)
    rel = np.linalg.norm(g - r) / nr if nr > 0 else np.linalg.norm(g - r)
    rms = float(np.sqrt(np.mean(r * r)))
    mx = float(np.max(np.abs(g - r))) / max(1.0, rms)
    return float(rel), mx


def check(name, gpu, ref, rel_l2=F32_REL_L2, max_abs=F32_MAX_ABS):
    rel, mx = errors(gpu, ref)
    assert np.all(np.isfinite(np.asarray(gpu))), "%s: non-finite values" % name
    assert rel <= rel_l2, "%s: relative L2 %.3e > %.1e" % (name, rel, rel_l2)
    if max_abs is not None:
        assert mx <= max_abs, "%s: scaled max-abs %.3e > %.1e" % (name, mx, max_abs)
    return rel, mx


def cfg_to_abi(tlb, cfg, persistent=False):
    """synth LayerConfig -> the C ABI layer struct."""
    return tlb.layer_cfg(cfg.dim, cfg.ffn_dim, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim, cfg.rank,
                         cfg.lora_alpha, act=cfg.act, wtype=cfg.wtype, sub_norm=cfg.sub_norm,
                         pre_norm=cfg.pre_norm, residual=cfg.residual, rope=cfg.rope,
                         use_silu_cache=(cfg.act == "silu_mul" and cfg.use_silu_cache), causal=True,
                         rope_base=cfg.rope_base, norm_eps=cfg.norm_eps, attn_scale=cfg.attn_scale,
                         persistent=persistent, qk_norm=cfg.qk_norm)


def adam_to_abi(tlb, cfg):
    return tlb.adamw_cfg(cfg.lr, cfg.beta1, cfg.beta2, cfg.adam_eps, cfg.weight_decay, cfg.step,
                         cfg.lr_b_mult)


def lora_dev(t: dict):
    """Adapter tensors keyed the way the binding's lora() expects."""
    out = {}
    for tag in ("q", "v"):
        out["a_" + tag] = t["a_" + tag].clone()
        out["b_" + tag] = t["b_" + tag].clone()
        out["m_a_" + tag] = t["m_a_" + tag].clone()
        out["v_a_" + tag] = t["v_a_" + tag].clone()
        out["m_b_" + tag] = t["m_b_" + tag].clone()
        out["v_b_" + tag] = t["v_b_" + tag].clone()
    return out
