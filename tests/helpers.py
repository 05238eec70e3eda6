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

from synth.device import lora_dev, to_dev  # noqa: F401  (re-exported for the tests)


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
    return tlb.layer_cfg_of(cfg, persistent=persistent)


def adam_to_abi(tlb, cfg):
    return tlb.adamw_cfg_of(cfg)


def tc_attention_shape(cfg) -> bool:
    """The shapes the tensor-core attention takes (bf16 layers with S > 1): head_dim 64 or
    128, L and L - S multiples of 4 (16-byte starts of the attention rows)."""
    S, L = cfg.seq_len, cfg.cache_len
    return (cfg.wtype == "bf16" and S > 1 and L % 4 == 0 and (L - S) % 4 == 0 and cfg.head_dim in (64, 128)
            and cfg.n_heads % cfg.n_kv_heads == 0 and not cfg.recompute_p)


def tc_recompute_shape(cfg) -> bool:
    """The recomputed attention (flash-style) runs on tcgen05 on the same shapes, without
    the exact input gradient (whose key gradient then recomputes on CUDA cores)."""
    return (tc_attention_shape(cfg.with_(recompute_p=False)) and cfg.recompute_p and not cfg.exact_din)


def assert_route(cfg, names):
    """bf16 layers with S > 1 must run their weight products on the tcgen05 GEMM and, where
    the shape allows, their attention on the tcgen05 kernels: a silent fall-back to the
    CUDA-core kernels would still pass the bf16 tolerance."""
    if cfg.wtype != "bf16" or cfg.seq_len <= 1:
        return
    assert "tcgen05 gemm" in names, ("tcgen05 GEMM did not run", names)
    if tc_recompute_shape(cfg):
        for k in ("attn_tc_dv_rc", "attn_tc_dsum", "attn_tc_dq_rc"):
            assert k in names, ("%s did not run" % k, names)
        assert "attn_dq_tiled" not in names, ("CUDA-core attention ran", names)
    assert "gemm_nt_simt" not in names, ("CUDA-core GEMM ran on a bf16 sequence layer", names)
    if tc_attention_shape(cfg):
        for k in ("attn_tc_dq", "attn_tc_dv"):
            assert k in names, ("%s did not run" % k, names)
        for k in ("attn_dq_tiled", "attn_rows"):
            assert k not in names, ("CUDA-core attention ran", names)
        if cfg.rank == 16:       # the adapters' passes run on the tensor cores beside it
            for k in ("lora_tc_gpass", "lora_tc_xpass"):
                assert k in names, ("%s did not run" % k, names)
            assert "lora_gpass" not in names, ("CUDA-core LoRA pass ran", names)
