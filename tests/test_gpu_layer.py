"""GPU parity of the layer pieces (ffn_backward, attn_backward, lora_grad_adamw) and
of the whole layer / stack against the float64 oracle on the same seeded inputs.

Configurations: the tiny fp32 layer (all norms, RoPE, GQA, causal), the
single-token decode layer with ternary weights, small bf16 sequence layers with
ragged sequence and cache lengths, the S = 512 SwiGLU layer, and layers with the
per-head QK-norm on q.
"""
import numpy as np
import pytest

from oracle import layer as OL
from oracle import ops
from synth import DECODE, SEQ512, TINY, layer_inputs
from tests.helpers import (BF16_REL_L2, adam_to_abi, assert_route, cfg_to_abi, check, host, lora_dev,
                           to_dev)

pytestmark = pytest.mark.gpu

MINI_SEQ = SEQ512.with_(name="mini_seq", dim=256, ffn_dim=640, n_heads=8, n_kv_heads=2, head_dim=32,
                        rank=8, lora_alpha=16.0, seq_len=77, cache_len=77)
TINY_WARM = TINY.with_(name="tiny_warm", adam_state="warm", step=7)
# single-token variants: ragged cache lengths, MHA and 8-head groups, every head size
DEC_F32 = DECODE.with_(name="dec_f32_hd64", dim=256, ffn_dim=512, n_heads=8, n_kv_heads=2, head_dim=64,
                       rank=4, lora_alpha=8.0, cache_len=100, wtype="f32", weight_std=0.05)
DEC_BF16 = DECODE.with_(name="dec_bf16_mha_silu", dim=512, ffn_dim=768, n_heads=4, n_kv_heads=4,
                        head_dim=128, cache_len=77, wtype="bf16", act="silu_mul", sub_norm=False,
                        pre_norm=False, kv_layout="shd", adam_state="warm", step=5)
DEC_G8 = DECODE.with_(name="dec_g8_hd32", dim=256, ffn_dim=256, n_heads=16, n_kv_heads=2, head_dim=32,
                      rank=8, lora_alpha=16.0, cache_len=40, pre_norm=False)
DEC_HD256 = DECODE.with_(name="dec_hd256", dim=512, ffn_dim=1024, n_heads=4, n_kv_heads=1, head_dim=256,
                         cache_len=65, sub_norm=False, rope=True)
# bf16 sequence layers on the tensor-core attention: head_dim 64 with S ragged over both
# tile sizes; a cache longer than the sequence (4-head groups, MHA).  L = 301 is not a
# multiple of 4, which the tensor-core attention needs: that layer takes the CUDA-core one.
SEQ_HD64 = SEQ512.with_(name="seq_hd64", dim=512, ffn_dim=1024, n_heads=8, n_kv_heads=2, head_dim=64,
                        rank=8, lora_alpha=16.0, seq_len=200, cache_len=200)
SEQ_CACHE = SEQ512.with_(name="seq_cache", dim=512, ffn_dim=768, n_heads=4, n_kv_heads=1, head_dim=128,
                         seq_len=96, cache_len=300, adam_state="warm", step=4)
SEQ_MHA = SEQ512.with_(name="seq_mha", dim=256, ffn_dim=512, n_heads=4, n_kv_heads=4, head_dim=64,
                       rank=4, lora_alpha=8.0, seq_len=130, cache_len=258)
SEQ_ODD = SEQ512.with_(name="seq_odd_cache", dim=512, ffn_dim=768, n_heads=4, n_kv_heads=1, head_dim=128,
                       seq_len=45, cache_len=301)
# QK-norm on q before RoPE: the CUDA-core sequence path, the single-token chain (its
# persistent variant falls back to the chain) and the tensor-core sequence path
TINY_QK = TINY.with_(name="tiny_qknorm", qk_norm=True)
DEC_QK = DEC_F32.with_(name="dec_qknorm", qk_norm=True, cache_len=65)
SEQ_QK = SEQ_HD64.with_(name="seq_qknorm", qk_norm=True, seq_len=148, cache_len=180)
# the other compositions on the tensor-core route: pre-norm (dR1 from the RMSNorm kernel,
# converted for the O-projection product) with ReLU^2 x Mul in the fused epilogue;
# no residual (the [W_gate | W_up]^T product overwrites d_res and writes its bf16 copy);
# both norms (the unfused W_down^T product, sub-norm and activation kernels)
SEQ_PRENORM = SEQ_MHA.with_(name="seq_prenorm", pre_norm=True, act="relu2_mul")
SEQ_NORESID = SEQ_HD64.with_(name="seq_noresid", residual=False, seq_len=96, cache_len=96)
SEQ_NORMS = SEQ_HD64.with_(name="seq_norms", sub_norm=True, pre_norm=True, seq_len=64, cache_len=96)
# the exact layer-input gradient (through W_Q, W_K, W_V, the LoRA A paths and the
# attention pre-norm) on every route: row kernels (tiny, head_dim 16), the single-token
# chain (fp32 and ternary), CUDA-core tiled attention (bf16, head_dim 32), tensor-core
# attention with the three-segment tcgen05 product (with and without the pre-norm, with
# the QK-norm on q and k, a cache longer than the sequence) and S = 512
TINY_EXACT = TINY.with_(name="tiny_exact", exact_din=True)
TINY_EXACT_QK = TINY.with_(name="tiny_exact_qknorm", exact_din=True, qk_norm=True, adam_state="warm", step=3)
DEC_EXACT = DEC_F32.with_(name="dec_exact", exact_din=True)
DECODE_EXACT = DECODE.with_(name="decode_exact", exact_din=True)
MINI_SEQ_EXACT = MINI_SEQ.with_(name="mini_seq_exact", exact_din=True)
SEQ_EXACT = SEQ_HD64.with_(name="seq_exact", exact_din=True)
SEQ_EXACT_PN = SEQ_MHA.with_(name="seq_exact_prenorm_qknorm", exact_din=True, pre_norm=True, qk_norm=True)
SEQ512_EXACT = SEQ512.with_(name="seq512_exact", exact_din=True)
# packed 2-bit ternary weights ([FFN] BitLinear, four to a byte): the full single-token
# layer, a small one with 8-head groups, and its exact input gradient
DECODE_T2 = DECODE.with_(name="decode_t2", wtype="ternary2")
DEC_T2 = DEC_G8.with_(name="dec_t2_g8", wtype="ternary2")
DEC_T2_EXACT = DEC_T2.with_(name="dec_t2_exact", exact_din=True, pre_norm=True)
# attention weights recomputed from q, the K cache and the logsumexp (flash-style): the
# row kernels (tiny, head_dim 16; a single-token layer), the tiled CUDA-core kernels (bf16
# layers of head_dim 32, 64 and 128, a cache longer than the sequence), and with the exact
# input gradient (the key-gradient kernels recompute too)
TINY_RC = TINY.with_(name="tiny_recompute", recompute_p=True)
DEC_RC = DEC_F32.with_(name="dec_recompute", recompute_p=True)
MINI_SEQ_RC = MINI_SEQ.with_(name="mini_seq_recompute", recompute_p=True)
SEQ_RC = SEQ_HD64.with_(name="seq_recompute", recompute_p=True)
SEQ_RC_CACHE = SEQ_CACHE.with_(name="seq_recompute_cache", recompute_p=True)
SEQ_RC_EXACT = SEQ_HD64.with_(name="seq_recompute_exact", recompute_p=True, exact_din=True, seq_len=130,
                              cache_len=130)
TINY_RC_EXACT = TINY.with_(name="tiny_recompute_exact", recompute_p=True, exact_din=True, qk_norm=True)
# the flash-style tcgen05 kernels: head_dim 128 over three ragged 128-query / 128-key tiles
SEQ_RC_LONG = SEQ_CACHE.with_(name="seq_recompute_long", recompute_p=True, seq_len=300, cache_len=300)
# rank-16 adapters beside the tensor-core attention take the tcgen05 LoRA passes: three
# 128-token tiles with a ragged last one, and a V side of 1.5 column tiles (3 KV heads)
SEQ_LORA16 = SEQ_HD64.with_(name="seq_lora16", rank=16, lora_alpha=32.0, seq_len=300, cache_len=300)
SEQ_LORA16_KV3 = SEQ_HD64.with_(name="seq_lora16_kv3", n_heads=6, n_kv_heads=3, rank=16, lora_alpha=32.0,
                                seq_len=170, cache_len=170, adam_state="warm", step=6)
# a wide hidden size with few query columns: the O-projection product [128, 512] x K 4096
# runs stream-K with shared tiles, so the fixup writes the attention's tf32 dCtx^T copy
SEQ_WIDE = SEQ_HD64.with_(name="seq_wide_wo_streamk", dim=4096, ffn_dim=1024, seq_len=128, cache_len=160)
CASES = {c.name: c for c in (SEQ_WIDE, SEQ_LORA16, SEQ_LORA16_KV3, SEQ_RC_LONG, TINY_RC, DEC_RC, MINI_SEQ_RC, SEQ_RC, SEQ_RC_CACHE, SEQ_RC_EXACT, TINY_RC_EXACT,
                             DECODE_T2, DEC_T2, DEC_T2_EXACT,
                             TINY, TINY_WARM, DECODE, MINI_SEQ, SEQ512, DEC_F32, DEC_BF16, DEC_G8, DEC_HD256,
                             SEQ_HD64, SEQ_CACHE, SEQ_MHA, SEQ_ODD, TINY_QK, DEC_QK, SEQ_QK, SEQ_PRENORM,
                             SEQ_NORESID, SEQ_NORMS, TINY_EXACT, TINY_EXACT_QK, DEC_EXACT, DECODE_EXACT,
                             MINI_SEQ_EXACT, SEQ_EXACT, SEQ_EXACT_PN, SEQ512_EXACT)}


def tol(cfg):
    """(rel_l2, max_abs) of the path this config runs on."""
    return (BF16_REL_L2, None) if cfg.wtype == "bf16" and cfg.seq_len > 1 and _tc_path() else (1e-5, 1e-4)


def _tc_path():
    return True    # bf16 weights with S > 1 run the tcgen05 GEMMs (bf16 operands, fp32 accumulation)


@pytest.fixture(scope="module", params=sorted(CASES))
def case(request):
    cfg = CASES[request.param]
    d = layer_inputs(cfg, layer=0, seed=0)
    ref = OL.layer_backward(cfg, d, d["dout"])
    return cfg, d, ref


def kv_layout(cfg):
    return cfg.kv_layout


def test_ffn_backward(lib, case):
    import torch
    cfg, d, ref = case
    t = to_dev(d, cfg.wtype)
    c = cfg_to_abi(lib, cfg)
    ws = lib.workspace(c, cfg.seq_len, cfg.cache_len)
    w = lib.layer_weights(c, t)
    a = lib.layer_acts(c, t, cfg.kv_layout, cfg.cache_len)
    out = torch.empty_like(t["dout"])
    n0 = lib.launch_count()
    lib.ffn_backward(c, cfg.seq_len, t["dout"], w, a, out, ws)
    if cfg.wtype == "bf16" and cfg.seq_len > 1:
        assert "tcgen05 gemm" in lib.launch_names(n0)
    rl, ma = tol(cfg)
    check("dR1", host(out), ref["dR1"], rl, ma)
    # in place: d_residual aliases d_out
    inplace = t["dout"].clone()
    lib.ffn_backward(c, cfg.seq_len, inplace, w, a, inplace, ws)
    check("dR1 in place", host(inplace), ref["dR1"], rl, ma)


def test_attn_backward(lib, case):
    import torch
    cfg, d, ref = case
    t = to_dev(d, cfg.wtype)
    c = cfg_to_abi(lib, cfg)
    ws = lib.workspace(c, cfg.seq_len, cfg.cache_len)
    w = lib.layer_weights(c, t)
    a = lib.layer_acts(c, t, cfg.kv_layout, cfg.cache_len)
    dr1 = torch.from_numpy(ref["dR1"].astype(np.float32)).cuda()
    dq = torch.empty(cfg.seq_len, cfg.q_dim, device="cuda")
    dv = torch.empty(cfg.seq_len, cfg.kv_dim, device="cuda")
    lib.attn_backward(c, cfg.seq_len, cfg.cache_len, dr1, w, a, dq, dv, ws)
    # the oracle from the same float32 dR1 the GPU received
    d2 = dict(d)
    r2 = OL.attn_backward(cfg, d2, dr1.cpu().numpy())
    rl, ma = tol(cfg)
    check("dQpre", host(dq), r2["dQpre"], rl, ma)
    check("dV", host(dv), r2["dV"], rl, ma)


# The cached weights carry the causal mask as zeros ([ATT] "Softmax Backward" reads them as
# given), so the attention without the causal flag must give the same gradients.  The
# tensor-core kernels then take every key tile of the cache for every query tile (no tile
# is masked in place; a last tile past L is zero-filled by the copy): S = L = 512, a ragged
# S = L = 200, and a cache longer than the sequence (L = 300, S = 96).
@pytest.mark.parametrize("name", ["seq512", "seq_hd64", "seq_cache"])
def test_attn_backward_without_causal_flag(lib, name):
    import torch
    from transformer_layer_backward_gb300 import _abi
    cfg = CASES[name]
    d = layer_inputs(cfg, layer=0, seed=0)
    t = to_dev(d, cfg.wtype)
    c = cfg_to_abi(lib, cfg)
    c.flags &= ~_abi.CAUSAL
    ws = lib.workspace(c, cfg.seq_len, cfg.cache_len)
    w = lib.layer_weights(c, t)
    a = lib.layer_acts(c, t, cfg.kv_layout, cfg.cache_len)
    dr1_h = np.random.default_rng(11).standard_normal((cfg.seq_len, cfg.dim)).astype(np.float32)
    dr1 = torch.from_numpy(dr1_h).cuda()
    dq = torch.empty(cfg.seq_len, cfg.q_dim, device="cuda")
    dv = torch.empty(cfg.seq_len, cfg.kv_dim, device="cuda")
    n0 = lib.launch_count()
    lib.attn_backward(c, cfg.seq_len, cfg.cache_len, dr1, w, a, dq, dv, ws)
    names = lib.launch_names(n0)
    for k in ("attn_tc_dq", "attn_tc_dv"):
        assert k in names, ("%s did not run" % k, names)
    r2 = OL.attn_backward(cfg, dict(d), dr1_h)
    rl, ma = tol(cfg)
    check("dQpre", host(dq), r2["dQpre"], rl, ma)
    check("dV", host(dv), r2["dV"], rl, ma)


def test_lora_grad_adamw(lib, case):
    import torch
    cfg, d, ref = case
    t = to_dev(d, cfg.wtype)
    c = cfg_to_abi(lib, cfg)
    adam = adam_to_abi(lib, cfg)
    ws = lib.workspace(c, cfg.seq_len, cfg.cache_len)
    for tag, G, out_dim in (("q", ref["dQpre"], cfg.q_dim), ("v", ref["dV"], cfg.kv_dim)):
        Gf = G.astype(np.float32)
        L = lora_dev(t)
        grads = {"dA_" + tag: torch.empty_like(L["a_" + tag]), "dB_" + tag: torch.empty_like(L["b_" + tag])}
        ss = torch.zeros(2, dtype=torch.float64, device="cuda")
        lib.lora_grad_adamw(cfg.seq_len, out_dim, cfg.dim, cfg.rank, cfg.lora_alpha,
                            torch.from_numpy(Gf).cuda(), t["lora_%s_h" % tag], t["x"],
                            lib.lora(L, tag, grads), adam, ss, ws)
        da, db, _ = ops.lora_backward(Gf, d["lora_%s_h" % tag], d["x"], d["b_" + tag], cfg.lora_alpha, cfg.rank)
        check("dA_" + tag, host(grads["dA_" + tag]), da)
        check("dB_" + tag, host(grads["dB_" + tag]), db)
        # the step from the GPU's own gradients: a first AdamW step moves a parameter by about
        # lr sign(g), so a float32 gradient element near zero may flip it
        for p, g, lr in (("a_" + tag, host(grads["dA_" + tag]), cfg.lr),
                         ("b_" + tag, host(grads["dB_" + tag]), cfg.lr * cfg.lr_b_mult)):
            rp, rm, rv = ops.adamw(d[p], g, d["m_" + p], d["v_" + p], lr, cfg.beta1, cfg.beta2,
                                   cfg.adam_eps, cfg.weight_decay, cfg.step)
            check(p, host(L[p]), rp)
            check("m_" + p, host(L["m_" + p[0] + "_" + tag]), rm)
            check("v_" + p, host(L["v_" + p[0] + "_" + tag]), rv)
        s = ss.cpu().numpy()
        assert abs(s[0] - np.sum(da ** 2)) <= 1e-5 * np.sum(da ** 2)
        assert abs(s[1] - np.sum(db ** 2)) <= 1e-5 * np.sum(db ** 2)


@pytest.mark.parametrize("persistent", [False, True])
def test_layer_backward(lib, case, persistent):
    import torch
    cfg, d, ref = case
    if persistent and cfg.seq_len != 1:
        pytest.skip("the persistent schedule is for single-token layers")
    t = to_dev(d, cfg.wtype)
    c = cfg_to_abi(lib, cfg, persistent=persistent)
    adam = adam_to_abi(lib, cfg)
    ws = lib.workspace(c, cfg.seq_len, cfg.cache_len)
    L = lora_dev(t)
    grads = {k: torch.empty_like(L[k.replace("dA_", "a_").replace("dB_", "b_")])
             for k in ("dA_q", "dB_q", "dA_v", "dB_v")}
    dh = t["dout"].clone()
    ss = torch.zeros(2, dtype=torch.float64, device="cuda")
    n0 = lib.launch_count()
    lib.layer_backward(c, cfg.seq_len, cfg.cache_len, lib.layer_weights(c, t),
                       lib.layer_acts(c, t, cfg.kv_layout, cfg.cache_len), lib.lora(L, "q", grads),
                       lib.lora(L, "v", grads), adam, dh, ss, ws)
    names = lib.launch_names(n0)
    assert_route(cfg, names)
    if cfg is SEQ_WIDE:
        assert "tcgen05 gemm fixup" in names, ("the stream-K fixup did not run", names)
    lib.workspace_status(ws)
    rl, ma = tol(cfg)
    rel = check("d_in", host(dh), ref["d_in"], rl, ma)[0]
    if cfg.exact_din:
        print("%s: exact d_in relative L2 %.2e" % (cfg.name, rel))
    for k in ("dA_q", "dB_q", "dA_v", "dB_v"):
        check(k, host(grads[k]), ref[k], rl, ma)
    s = ss.cpu().numpy()
    assert abs(s[0] - ref["sumsq_a"]) <= max(rl, 1e-5) * 2 * ref["sumsq_a"]
    assert abs(s[1] - ref["sumsq_b"]) <= max(rl, 1e-5) * 2 * ref["sumsq_b"]
    # parameters: AdamW of the GPU's own gradients must match to float32 accuracy
    for tag in ("q", "v"):
        for p, lr in (("a_" + tag, cfg.lr), ("b_" + tag, cfg.lr * cfg.lr_b_mult)):
            g = host(grads["d" + p[0].upper() + "_" + tag])
            rp, rm, rv = ops.adamw(d[p], g, d["m_" + p], d["v_" + p], lr, cfg.beta1, cfg.beta2,
                                   cfg.adam_eps, cfg.weight_decay, cfg.step)
            check(p, host(L[p]), rp)
            check("m_" + p, host(L["m_" + p[0] + "_" + tag]), rm)
            if rl <= 1e-5:
                check(p + " vs oracle", host(L[p]), ref[p])


def test_stack_of_layers(lib):
    """Three tiny layers in reverse: the gradient of layer l feeds layer l - 1."""
    import torch
    cfg = TINY.with_(name="tiny_stack", n_layers=3)
    layers = [layer_inputs(cfg, layer=l, seed=0, with_dout=(l == cfg.n_layers - 1)) for l in range(3)]
    dout = layers[-1]["dout"]
    ref = OL.stack_backward(cfg, layers, dout)
    c = cfg_to_abi(lib, cfg)
    adam = adam_to_abi(lib, cfg)
    ws = lib.workspace(c, cfg.seq_len, cfg.cache_len)
    dh = torch.from_numpy(dout).cuda()
    ss = torch.zeros(2, dtype=torch.float64, device="cuda")
    devs = []
    for l in reversed(range(3)):
        t = to_dev(layers[l], cfg.wtype)
        L = lora_dev(t)
        devs.append((l, L))
        lib.layer_backward(c, cfg.seq_len, cfg.cache_len, lib.layer_weights(c, t),
                           lib.layer_acts(c, t, cfg.kv_layout, cfg.cache_len), lib.lora(L, "q"),
                           lib.lora(L, "v"), adam, dh, ss, ws)
    check("stack d_in", host(dh), ref["d_in"])
    gnorm = float(np.sqrt(ss[0].item()))
    assert abs(gnorm - ref["gnorm"]) <= 1e-5 * ref["gnorm"]
    for l, L in devs:
        for p in ("a_q", "b_q", "a_v", "b_v"):
            check("layer %d %s" % (l, p), host(L[p]), ref["layers"][l][p])
