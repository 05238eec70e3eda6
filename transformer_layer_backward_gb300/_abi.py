"""ctypes mirror of ``include/tlb.h`` and the loader of ``lib/libtlb.so``.

The library is loaded from this package's ``lib`` folder only; if it is missing
the loader raises (build it with ``transformer_layer_backward_gb300.build``).
"""
from __future__ import annotations

import ctypes as C
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libtlb.so")

TLB_OK, TLB_EINVAL, TLB_EUNSUPPORTED, TLB_ENONFINITE, TLB_ETIMEOUT, TLB_ECUDA = 0, -1, -2, -3, -4, -5
ACT_RELU2_MUL, ACT_SILU_MUL = 0, 1
W_F32, W_BF16, W_TERNARY_I8, W_TERNARY_2B = 0, 1, 2, 3
SUB_NORM, PRE_NORM, RESIDUAL, ROPE, USE_SILU_CACHE, CAUSAL, PERSISTENT, QK_NORM = 1, 2, 4, 8, 16, 32, 64, 128
CHECK_FINITE, EXACT_DIN, RECOMPUTE_P = 256, 512, 1024

vp, i32, i64, f32, sz = C.c_void_p, C.c_int32, C.c_int64, C.c_float, C.c_size_t


class LayerCfg(C.Structure):
    _fields_ = [("dim", i32), ("ffn_dim", i32), ("n_heads", i32), ("n_kv_heads", i32),
                ("head_dim", i32), ("rank", i32), ("lora_alpha", f32), ("rope_base", f32),
                ("norm_eps", f32), ("attn_scale", f32), ("act", i32), ("wtype", i32),
                ("flags", i32)]


class Weight(C.Structure):
    _fields_ = [("w", vp), ("scale", f32)]


class LayerWeights(C.Structure):
    _fields_ = [("w_down", Weight), ("w_gate", Weight), ("w_up", Weight), ("w_o", Weight),
                ("gamma_sub_ffn", vp), ("gamma_ffn", vp), ("gamma_sub_attn", vp), ("gamma_q", vp),
                ("w_q", Weight), ("w_k", Weight), ("w_v", Weight), ("gamma_attn", vp), ("gamma_k", vp)]


class LayerActs(C.Structure):
    _fields_ = [("x", vp), ("gate", vp), ("up", vp), ("silu_gate", vp), ("hidden", vp),
                ("r1", vp), ("ctx", vp), ("k", vp), ("v", vp), ("kv_stride_head", i64),
                ("kv_stride_pos", i64), ("attn", vp), ("lora_q_h", vp), ("lora_v_h", vp),
                ("q_raw", vp), ("x_in", vp), ("q", vp), ("k_raw", vp), ("lse", vp)]


class Lora(C.Structure):
    _fields_ = [("a", vp), ("b", vp), ("m_a", vp), ("v_a", vp), ("m_b", vp), ("v_b", vp),
                ("grad_a", vp), ("grad_b", vp)]


class AdamwCfg(C.Structure):
    _fields_ = [("lr", C.c_double), ("beta1", C.c_double), ("beta2", C.c_double),
                ("eps", C.c_double), ("weight_decay", C.c_double), ("lr_b_mult", C.c_double),
                ("step", i32)]


P = C.POINTER
SIGNATURES = {
    "tlb_last_error": (C.c_char_p, []),
    "tlb_build_info": (C.c_char_p, []),
    "tlb_launch_count": (C.c_uint64, []),
    "tlb_launch_name": (C.c_char_p, [C.c_uint64]),
    "tlb_debug_skip_barrier_arrival": (C.c_int, [i32]),
    "tlb_profile_events": (None, [C.POINTER(C.c_void_p), i32]),
    "tlb_profile_kernel_name": (C.c_char_p, [i32]),
    "tlb_linear_workspace_bytes": (sz, [i32, i64, i64, i64]),
    "tlb_linear_backward": (C.c_int, [i32, vp, f32, vp, i64, i64, i64, vp, i32, vp, sz, vp]),
    "tlb_softmax_backward": (C.c_int, [vp, vp, vp, i64, i64, vp]),
    "tlb_act_backward": (C.c_int, [i32, vp, vp, vp, vp, vp, vp, i64, vp]),
    "tlb_rmsnorm_backward": (C.c_int, [vp, vp, vp, vp, i64, i64, f32, i32, vp]),
    "tlb_rope_backward": (C.c_int, [vp, vp, i64, i32, i32, i64, f32, vp]),
    "tlb_adamw": (C.c_int, [vp, vp, vp, vp, i64, P(AdamwCfg), f32, vp, vp]),
    "tlb_workspace_bytes": (sz, [P(LayerCfg), i64, i64]),
    "tlb_workspace_status": (C.c_int, [vp, sz, vp]),
    "tlb_ffn_backward": (C.c_int, [P(LayerCfg), i64, vp, P(LayerWeights), P(LayerActs), vp, vp,
                                   sz, vp]),
    "tlb_attn_backward": (C.c_int, [P(LayerCfg), i64, i64, vp, P(LayerWeights), P(LayerActs), vp,
                                    vp, vp, sz, vp]),
    "tlb_lora_grad_adamw": (C.c_int, [i64, i32, i32, i32, f32, vp, vp, vp, P(Lora), P(AdamwCfg),
                                      vp, vp, sz, vp]),
    "tlb_lora_grad_adamw_noalloc": (C.c_int, [i64, i32, i32, i32, f32, vp, vp, vp, P(Lora),
                                              P(AdamwCfg), vp, vp]),
    "tlb_layer_backward": (C.c_int, [P(LayerCfg), i64, i64, P(LayerWeights), P(LayerActs),
                                     P(Lora), P(Lora), P(AdamwCfg), vp, vp, vp, sz, vp]),
    "tlb_stack_workspace_bytes": (sz, [P(LayerCfg), i64, i64]),
    "tlb_stack_backward": (C.c_int, [P(LayerCfg), i64, i64, i32, P(LayerWeights), P(LayerActs),
                                     P(Lora), P(Lora), P(AdamwCfg), vp, vp, vp, sz, vp]),
}

_lib = None


def load(path: str = LIB_PATH):
    """Load the shared library (once) and declare every exported signature."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError("CUDA library %s is missing: build it first "
                           "(python -m transformer_layer_backward_gb300.build)" % path)
    lib = C.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class TlbError(RuntimeError):
    def __init__(self, code: int, fn: str, msg: str):
        super().__init__("%s returned %d: %s" % (fn, code, msg))
        self.code = code


def call(name: str, *args) -> int:
    lib = load()
    rc = getattr(lib, name)(*args)
    if rc != TLB_OK:
        raise TlbError(rc, name, lib.tlb_last_error().decode())
    return rc
