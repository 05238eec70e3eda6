"""Python binding of the C ABI: one function per entry point, with the same names.

Each function checks devices, dtypes and contiguity of torch tensors, then passes
raw device pointers to the library.  No arithmetic of the backward pass happens
here; every step runs in the CUDA kernels of ``lib/libtlb.so``.
"""
from __future__ import annotations

import ctypes as C
import math

import torch

from . import _abi as A

_WDTYPE = {A.W_F32: torch.float32, A.W_BF16: torch.bfloat16, A.W_TERNARY_I8: torch.int8,
           A.W_TERNARY_2B: torch.uint8}
_WCODE = {"f32": A.W_F32, "bf16": A.W_BF16, "ternary": A.W_TERNARY_I8, "ternary2": A.W_TERNARY_2B}


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def _ptr(t, dtype=torch.float32, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be on a CUDA device" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return C.c_void_p(t.data_ptr()) if t.numel() else None


# ------------------------------------------------------------------ standalone steps

def softmax_backward(attn, dattn, out=None, stream=None):
    """dS = attn * (dAttn - rowsum(attn * dAttn)) over the last axis."""
    out = torch.empty_like(attn) if out is None else out
    rows = attn.numel() // attn.shape[-1] if attn.dim() and attn.shape[-1] else 0
    A.call("tlb_softmax_backward", _ptr(attn, name="attn"), _ptr(dattn, name="dattn"),
           _ptr(out, name="out"), rows, attn.shape[-1] if attn.dim() else 0, _stream(stream))
    return out


def act_backward(act, gate, up, dh, silu_gate=None, dgate=None, dup=None, stream=None):
    """Gated activation backward; act is 'relu2_mul' or 'silu_mul'."""
    code = {"relu2_mul": A.ACT_RELU2_MUL, "silu_mul": A.ACT_SILU_MUL}[act]
    dgate = torch.empty_like(gate) if dgate is None else dgate
    dup = torch.empty_like(gate) if dup is None else dup
    A.call("tlb_act_backward", code, _ptr(gate, name="gate"), _ptr(up, name="up"),
           _ptr(silu_gate, name="silu_gate"), _ptr(dh, name="dh"), _ptr(dgate, name="dgate"),
           _ptr(dup, name="dup"), gate.numel(), _stream(stream))
    return dgate, dup


def rmsnorm_backward(x, gamma, dy, eps=1e-6, out=None, accumulate=False, stream=None):
    """Row-wise RMSNorm backward over the last axis; accumulate adds into out."""
    out = torch.empty_like(x) if out is None else out
    n = x.shape[-1]
    rows = x.numel() // n if n else 0
    A.call("tlb_rmsnorm_backward", _ptr(x, name="x"), _ptr(gamma, name="gamma"),
           _ptr(dy, name="dy"), _ptr(out, name="out"), rows, n, float(eps),
           1 if accumulate else 0, _stream(stream))
    return out


def rope_backward(dy, pos0, base=10000.0, out=None, stream=None):
    """Inverse NeoX rotation of dy [rows, n_heads, head_dim]; row r at position pos0 + r."""
    out = torch.empty_like(dy) if out is None else out
    rows, nh, hd = dy.shape
    A.call("tlb_rope_backward", _ptr(dy, name="dy"), _ptr(out, name="out"), rows, nh, hd,
           int(pos0), float(base), _stream(stream))
    return out


def linear_workspace(wtype, S, out_dim, in_dim, device="cuda"):
    code = _WCODE[wtype]
    n = int(A.load().tlb_linear_workspace_bytes(code, int(S), int(out_dim), int(in_dim)))
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device)


def linear_backward(wtype, W, dY, scale=1.0, out=None, accumulate=False, ws=None, stream=None):
    """dX = scale * dY @ W^T for W stored [in, out] (wtype 'f32', 'bf16', 'ternary', or
    'ternary2': uint8 [in, out / 4], four 2-bit codes per byte)."""
    code = _WCODE[wtype]
    in_dim, out_dim = W.shape
    if code == A.W_TERNARY_2B:
        out_dim *= 4
    S = dY.shape[0]
    out = torch.zeros(S, in_dim, device=dY.device) if out is None else out
    ws = linear_workspace(wtype, S, out_dim, in_dim, dY.device) if ws is None else ws
    A.call("tlb_linear_backward", code, _ptr(W, _WDTYPE[code], "W"), float(scale), _ptr(dY, name="dY"),
           S, out_dim, in_dim, _ptr(out, name="out"), 1 if accumulate else 0,
           _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream))
    return out


def launch_count() -> int:
    return int(A.load().tlb_launch_count())


def launch_names(first: int, last: int | None = None):
    """Names of the library's launches numbered first .. last - 1 (launch_count() values
    taken before and after a call); None where the log no longer holds one."""
    lib = A.load()
    last = launch_count() if last is None else last
    out = []
    for i in range(first, last):
        nm = lib.tlb_launch_name(i)
        out.append(nm.decode() if nm is not None else None)
    return out


def profile_events(events):
    """events[0] (torch.cuda.Event) is recorded at the start of each later layer call and
    events[k + 1] after its k-th kernel; None turns it off.  Returns the ctypes array,
    which must stay alive while in use."""
    lib = A.load()
    if events is None:
        lib.tlb_profile_events(None, 0)
        return None
    for e in events:            # torch creates the CUDA event on its first record
        e.record()
    arr = (C.c_void_p * len(events))(*[C.c_void_p(e.cuda_event) for e in events])
    lib.tlb_profile_events(arr, len(events))
    return arr


def adamw_cfg(lr, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=1, lr_b_mult=16.0):
    return A.AdamwCfg(lr, beta1, beta2, eps, weight_decay, lr_b_mult, int(step))


def adamw(p, g, m, v, cfg: A.AdamwCfg, lr_mult=1.0, sumsq=None, stream=None):
    """One AdamW step in place on p, m, v; sumsq (float64 device scalar) += sum(g^2)."""
    A.call("tlb_adamw", _ptr(p, name="p"), _ptr(g, name="g"), _ptr(m, name="m"),
           _ptr(v, name="v"), p.numel(), C.byref(cfg), float(lr_mult),
           _ptr(sumsq, torch.float64, "sumsq"), _stream(stream))


# ------------------------------------------------------------------ layer pieces

def layer_cfg(dim, ffn_dim, n_heads, n_kv_heads, head_dim, rank, lora_alpha, act="relu2_mul",
              wtype="f32", sub_norm=False, pre_norm=False, residual=True, rope=True,
              use_silu_cache=False, causal=True, rope_base=10000.0, norm_eps=1e-6,
              attn_scale=None, persistent=False, qk_norm=False, check_finite=False,
              exact_din=False, recompute_p=False) -> A.LayerCfg:
    flags = ((A.SUB_NORM if sub_norm else 0) | (A.PRE_NORM if pre_norm else 0) |
             (A.RESIDUAL if residual else 0) | (A.ROPE if rope else 0) |
             (A.USE_SILU_CACHE if use_silu_cache else 0) | (A.CAUSAL if causal else 0) |
             (A.PERSISTENT if persistent else 0) | (A.QK_NORM if qk_norm else 0) |
             (A.CHECK_FINITE if check_finite else 0) | (A.EXACT_DIN if exact_din else 0) |
             (A.RECOMPUTE_P if recompute_p else 0))
    return A.LayerCfg(dim, ffn_dim, n_heads, n_kv_heads, head_dim, rank, float(lora_alpha),
                      float(rope_base), float(norm_eps),
                      float(1.0 / math.sqrt(head_dim) if attn_scale is None else attn_scale),
                      {"relu2_mul": A.ACT_RELU2_MUL, "silu_mul": A.ACT_SILU_MUL}[act],
                      _WCODE[wtype], flags)


def layer_cfg_of(c, persistent=False, check_finite=False) -> A.LayerCfg:
    """The layer struct for any object with the attributes of a layer configuration
    (dim, ffn_dim, n_heads, n_kv_heads, head_dim, rank, lora_alpha, act, wtype, sub_norm,
    pre_norm, residual, rope, use_silu_cache, rope_base, norm_eps, attn_scale, qk_norm);
    the attention is causal."""
    return layer_cfg(c.dim, c.ffn_dim, c.n_heads, c.n_kv_heads, c.head_dim, c.rank, c.lora_alpha,
                     act=c.act, wtype=c.wtype, sub_norm=c.sub_norm, pre_norm=c.pre_norm,
                     residual=c.residual, rope=c.rope,
                     use_silu_cache=(c.act == "silu_mul" and c.use_silu_cache), causal=True,
                     rope_base=c.rope_base, norm_eps=c.norm_eps, attn_scale=c.attn_scale,
                     persistent=persistent, qk_norm=c.qk_norm, check_finite=check_finite,
                     exact_din=getattr(c, "exact_din", False), recompute_p=getattr(c, "recompute_p", False))


def adamw_cfg_of(c) -> A.AdamwCfg:
    """The AdamW struct for an object with lr, beta1, beta2, adam_eps, weight_decay, step
    and lr_b_mult attributes."""
    return adamw_cfg(c.lr, c.beta1, c.beta2, c.adam_eps, c.weight_decay, c.step, c.lr_b_mult)


def workspace_bytes(cfg: A.LayerCfg, S: int, L: int) -> int:
    return int(A.load().tlb_workspace_bytes(C.byref(cfg), int(S), int(L)))


def workspace(cfg: A.LayerCfg, S: int, L: int, device="cuda"):
    """A zeroed workspace tensor of the size the library asks for."""
    return torch.zeros(max(workspace_bytes(cfg, S, L), 256), dtype=torch.uint8, device=device)


def debug_skip_barrier_arrival(block: int):
    """Test hook of the device-side timeout path (see tlb_debug_skip_barrier_arrival)."""
    A.call("tlb_debug_skip_barrier_arrival", int(block))


def workspace_status(ws, stream=None):
    A.call("tlb_workspace_status", _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream))


def layer_weights(cfg: A.LayerCfg, t: dict):
    """Weights from a dict: w_down/w_gate/w_up/w_o (+ s_* scales); the gains g_sub_ffn,
    g_ffn, g_sub_attn, g_q are optional, and so are w_q/w_k/w_v, g_attn, g_k (the exact
    layer-input gradient)."""
    wd = _WDTYPE[cfg.wtype]

    def w(name):
        if name not in t:
            return A.Weight(None, 1.0)
        return A.Weight(_ptr(t[name], wd, name), float(t.get("s_" + name[2:], 1.0)))

    return A.LayerWeights(w("w_down"), w("w_gate"), w("w_up"), w("w_o"),
                          _ptr(t.get("g_sub_ffn"), name="g_sub_ffn"),
                          _ptr(t.get("g_ffn"), name="g_ffn"),
                          _ptr(t.get("g_sub_attn"), name="g_sub_attn"),
                          _ptr(t.get("g_q"), name="g_q"),
                          w("w_q"), w("w_k"), w("w_v"),
                          _ptr(t.get("g_attn"), name="g_attn"), _ptr(t.get("g_k"), name="g_k"))


def layer_acts(cfg: A.LayerCfg, t: dict, kv_layout: str, L: int):
    """Cached activations from a dict; kv_layout 'shd' = [L, kv_dim], 'hsd' = [n_kv, L, hd]."""
    hd = cfg.head_dim
    if kv_layout == "shd":
        sh, sp = hd, cfg.n_kv_heads * hd
    else:
        sh, sp = L * hd, hd
    g = lambda k: _ptr(t.get(k), name=k)
    return A.LayerActs(g("x"), g("gate"), g("up"), g("silu_gate"), g("hidden"), g("r1"),
                       g("ctx"), g("k"), g("v"), sh, sp, g("attn"), g("lora_q_h"), g("lora_v_h"),
                       g("q_raw"), g("x_in"), g("q"), g("k_raw"), g("lse"))


def lora(t: dict, tag: str, grads: dict | None = None):
    g = grads or {}
    p = lambda k: _ptr(t[k], name=k)
    return A.Lora(p("a_" + tag), p("b_" + tag), p("m_a_" + tag), p("v_a_" + tag),
                  p("m_b_" + tag), p("v_b_" + tag),
                  _ptr(g.get("dA_" + tag), name="dA"), _ptr(g.get("dB_" + tag), name="dB"))


def ffn_backward(cfg, S, d_out, weights, acts, d_residual, ws, stream=None):
    A.call("tlb_ffn_backward", C.byref(cfg), int(S), _ptr(d_out, name="d_out"), C.byref(weights),
           C.byref(acts), _ptr(d_residual, name="d_residual"), _ptr(ws, torch.uint8, "ws"),
           ws.numel(), _stream(stream))


def attn_backward(cfg, S, L, d_attn_out, weights, acts, d_qpre, d_v, ws, stream=None):
    A.call("tlb_attn_backward", C.byref(cfg), int(S), int(L), _ptr(d_attn_out, name="d_attn_out"),
           C.byref(weights), C.byref(acts), _ptr(d_qpre, name="d_qpre"), _ptr(d_v, name="d_v"),
           _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream))


def lora_grad_adamw(S, out_dim, in_dim, rank, alpha, G, h, x, lora_: A.Lora, adam: A.AdamwCfg,
                    sumsq, ws, stream=None):
    A.call("tlb_lora_grad_adamw", int(S), int(out_dim), int(in_dim), int(rank), float(alpha),
           _ptr(G, name="G"), _ptr(h, name="h"), _ptr(x, name="x"), C.byref(lora_), C.byref(adam),
           _ptr(sumsq, torch.float64, "sumsq"), _ptr(ws, torch.uint8, "ws"), ws.numel(),
           _stream(stream))


def lora_grad_adamw_noalloc(S, out_dim, in_dim, rank, alpha, G, h, x, lora_: A.Lora, adam: A.AdamwCfg,
                            sumsq, stream=None):
    """lora_grad_adamw without a workspace: for callers that cannot allocate device memory.
    Its scratch is a fixed array inside the library (S * rank <= 65536); calls sharing it
    must not overlap on the GPU."""
    A.call("tlb_lora_grad_adamw_noalloc", int(S), int(out_dim), int(in_dim), int(rank), float(alpha),
           _ptr(G, name="G"), _ptr(h, name="h"), _ptr(x, name="x"), C.byref(lora_), C.byref(adam),
           _ptr(sumsq, torch.float64, "sumsq"), _stream(stream))


def layer_backward(cfg, S, L, weights, acts, lora_q, lora_v, adam, d_hidden, sumsq, ws, stream=None):
    A.call("tlb_layer_backward", C.byref(cfg), int(S), int(L), C.byref(weights), C.byref(acts),
           C.byref(lora_q), C.byref(lora_v), C.byref(adam), _ptr(d_hidden, name="d_hidden"),
           _ptr(sumsq, torch.float64, "sumsq"), _ptr(ws, torch.uint8, "ws"), ws.numel(),
           _stream(stream))


def stack_workspace(cfg: A.LayerCfg, S: int, L: int, device="cuda"):
    """A zeroed workspace tensor for stack_backward."""
    n = int(A.load().tlb_stack_workspace_bytes(C.byref(cfg), int(S), int(L)))
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device)


def stack_backward(cfg, S, L, weights, acts, lora_q, lora_v, adam, d_hidden, sumsq, ws, stream=None):
    """Layers len(weights) - 1 .. 0 of a stack (entry l of each list is layer l); d_hidden
    holds the top layer's dOut on entry and layer 0's d_in on return."""
    n = len(weights)
    if not (len(acts) == len(lora_q) == len(lora_v) == n):
        raise ValueError("stack_backward: the four layer lists differ in length")
    W = (A.LayerWeights * max(n, 1))(*weights)
    X = (A.LayerActs * max(n, 1))(*acts)
    Q = (A.Lora * max(n, 1))(*lora_q)
    V = (A.Lora * max(n, 1))(*lora_v)
    A.call("tlb_stack_backward", C.byref(cfg), int(S), int(L), n, W, X, Q, V, C.byref(adam),
           _ptr(d_hidden, name="d_hidden"), _ptr(sumsq, torch.float64, "sumsq"), _ptr(ws, torch.uint8, "ws"),
           ws.numel(), _stream(stream))
