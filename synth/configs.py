"""Shapes and hyperparameters of the synthetic workloads.

Each ``LayerConfig`` fixes one layer-backward problem: model shapes, the number of
query rows ``seq_len`` (S) handled by one call, the number of cached keys
``cache_len`` (L >= S; query row i sits at position L - S + i), the gated
activation, the weight storage type and the composition flags.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass


@dataclass(frozen=True)
class LayerConfig:
    name: str
    dim: int                 # hidden size H
    ffn_dim: int             # intermediate size I
    n_heads: int
    n_kv_heads: int
    head_dim: int
    rank: int                # LoRA rank r (Q and V)
    lora_alpha: float
    seq_len: int             # S: query rows in one call
    cache_len: int           # L: keys visible to the last query row
    n_layers: int = 1
    act: str = "relu2_mul"   # "relu2_mul" (ReLU^2 x Mul) or "silu_mul" (SwiGLU)
    wtype: str = "f32"       # "f32", "bf16", "ternary" (int8 {-1,0,1} + scale) or "ternary2"
                             # (the same values packed four 2-bit codes to a byte)
    sub_norm: bool = False   # RMSNorm after attention context and after the FFN hidden
    pre_norm: bool = False   # RMSNorm before the FFN (backward adds into the residual)
    residual: bool = True    # out = r1 + f and r1 = x + a
    rope: bool = True        # NeoX split-half rotary embedding on q and k
    qk_norm: bool = False    # per-head RMSNorm of q and k over head_dim, before RoPE
    exact_din: bool = False  # the layer-input gradient also through the Q/K/V projections,
                             # their LoRA paths and the attention pre-norm (the pages stop
                             # at the projection outputs); oracle only
    recompute_p: bool = False  # attention weights recomputed from q, the K cache and each row's
                               # logsumexp instead of read from the cached [nh, S, L] weights
    kv_layout: str = "shd"   # "shd": [L, n_kv*hd]   "hsd": [n_kv, L, hd]
    rope_base: float = 10000.0
    norm_eps: float = 1e-6
    weight_std: float = 0.02
    lora_a_std: float = 0.02
    lora_b_std: float = 0.02
    attn_logit_std: float = 1.0   # attn rows = softmax(N(0, std^2)) (masked causally)
    use_silu_cache: bool = True   # SwiGLU: read the cached silu(gate)
    lr: float = 1e-4
    beta1: float = 0.9
    beta2: float = 0.999
    adam_eps: float = 1e-8
    weight_decay: float = 0.01
    step: int = 1
    lr_b_mult: float = 16.0
    adam_state: str = "zeros"     # "zeros" (first step) or "warm" (m ~ N(0,1e-2), v ~ U(0,1e-4))

    @property
    def q_dim(self) -> int:
        return self.n_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    @property
    def pos0(self) -> int:
        return self.cache_len - self.seq_len

    @property
    def attn_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def with_(self, **kw) -> "LayerConfig":
        return dataclasses.replace(self, **kw)


# Tiny single layer, fp32 (ReLU^2 x Mul FFN, RMSNorm sub- and pre-norms, causal).
TINY = LayerConfig(
    name="tiny", dim=64, ffn_dim=256, n_heads=4, n_kv_heads=2, head_dim=16,
    rank=4, lora_alpha=8.0, seq_len=32, cache_len=32, act="relu2_mul", wtype="f32",
    sub_norm=True, pre_norm=True, residual=True, rope=True, kv_layout="shd",
    weight_std=0.05, lora_a_std=0.05, lora_b_std=0.02)

# Single-token decode backward of one BitNet-style layer (ternary weights).
DECODE = LayerConfig(
    name="decode", dim=2560, ffn_dim=6912, n_heads=20, n_kv_heads=5, head_dim=128,
    rank=16, lora_alpha=32.0, seq_len=1, cache_len=1024, act="relu2_mul", wtype="ternary",
    sub_norm=True, pre_norm=True, residual=True, rope=True, kv_layout="hsd",
    attn_logit_std=1.0 / math.sqrt(128.0))

# Sequence backward of one SwiGLU layer, bf16 weights, S = 512.
SEQ512 = LayerConfig(
    name="seq512", dim=2560, ffn_dim=9728, n_heads=32, n_kv_heads=8, head_dim=128,
    rank=16, lora_alpha=32.0, seq_len=512, cache_len=512, act="silu_mul", wtype="bf16",
    sub_norm=False, pre_norm=False, residual=True, rope=True, kv_layout="shd")

# 36-layer stack, same layer as SEQ512 with S = 2048.
STACK2048 = SEQ512.with_(name="stack2048", seq_len=2048, cache_len=2048, n_layers=36)

CONFIGS = {c.name: c for c in (TINY, DECODE, SEQ512, STACK2048)}
