"""Pins of the float64 oracle against facts that do not come from the oracle itself.

* central finite differences of the scalar loss <dOut, out> of a consistent
  forward, through the whole layer (every LoRA gradient and the gradient handed
  to the layer below), for every composition the configurations use;
* invariants: softmax-backward rows sum to zero, RoPE backward inverts the
  forward rotation and preserves norms, RMSNorm backward is orthogonal to x;
* closed forms: uniform / one-hot attention rows, constant RMSNorm rows, the
  RoPE angle law on a two-frequency head, SiLU'(0) = 1/2, AdamW moving each
  parameter by lr*sign(g) on its first step, decoupled weight decay;
* reductions: GQA equals MHA with duplicated KV heads; B = 0 kills dA;
* the page's own trainer test run in page-literal mode.
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import forward as F
from oracle import layer as Lyr
from oracle import ops
from synth.configs import LayerConfig

HERE = os.path.dirname(os.path.abspath(__file__))
pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def small_cfg(**kw):
    base = dict(name="pin", dim=8, ffn_dim=12, n_heads=4, n_kv_heads=2, head_dim=4, rank=2,
                lora_alpha=4.0, seq_len=3, cache_len=5, act="relu2_mul", wtype="f32",
                sub_norm=True, pre_norm=True, residual=True, rope=True, kv_layout="shd",
                rope_base=10.0, norm_eps=1e-6)
    base.update(kw)
    return LayerConfig(**base)


def make_problem(cfg, seed=1):
    rs = np.random.default_rng(seed)
    H, I, qd, kvd, r = cfg.dim, cfg.ffn_dim, cfg.q_dim, cfg.kv_dim, cfg.rank
    S, L, nkv, hd = cfg.seq_len, cfg.cache_len, cfg.n_kv_heads, cfg.head_dim
    p = dict(w_q=rs.normal(0, 0.4, (H, qd)), w_k=rs.normal(0, 0.4, (H, kvd)),
             w_v=rs.normal(0, 0.4, (H, kvd)), w_o=rs.normal(0, 0.4, (qd, H)),
             w_gate=rs.normal(0, 0.4, (H, I)), w_up=rs.normal(0, 0.4, (H, I)),
             w_down=rs.normal(0, 0.4, (I, H)),
             s_o=0.7, s_gate=1.3, s_up=0.9, s_down=1.1,
             g_sub_attn=rs.uniform(0.5, 1.5, qd), g_ffn=rs.uniform(0.5, 1.5, H),
             g_sub_ffn=rs.uniform(0.5, 1.5, I),
             a_q=rs.normal(0, 0.4, (r, H)), b_q=rs.normal(0, 0.4, (qd, r)),
             a_v=rs.normal(0, 0.4, (r, H)), b_v=rs.normal(0, 0.4, (kvd, r)))
    n1 = rs.normal(size=(S, H))
    x_in = rs.normal(size=(S, H))
    k_prev = rs.normal(size=(nkv, L - S, hd))
    v_prev = rs.normal(size=(nkv, L - S, hd))
    dout = rs.normal(size=(S, H))
    p["g_q"], p["g_k"] = rs.uniform(0.5, 1.5, hd), rs.uniform(0.5, 1.5, hd)
    p["g_attn"] = rs.uniform(0.5, 1.5, H)
    return p, n1, x_in, k_prev, v_prev, dout


def backward_inputs(cfg, p, cache):
    d = dict(cache)
    for k in ("w_o", "w_gate", "w_up", "w_down", "s_o", "s_gate", "s_up", "s_down",
              "g_sub_attn", "g_ffn", "g_sub_ffn", "g_q", "g_k", "g_attn", "w_q", "w_k", "w_v",
              "a_q", "b_q", "a_v", "b_v"):
        d[k] = p[k]
    for k in ("a_q", "b_q", "a_v", "b_v"):
        d["m_" + k] = np.zeros_like(p[k])
        d["v_" + k] = np.zeros_like(p[k])
    return d


FD_CASES = {
    "chunk_gqa_all_norms": small_cfg(),
    "decode_hsd": small_cfg(seq_len=1, cache_len=6, kv_layout="hsd"),
    "swiglu_residual_rope": small_cfg(act="silu_mul", sub_norm=False, pre_norm=False,
                                      seq_len=4, cache_len=4),
    "page_literal_flags0": small_cfg(act="silu_mul", sub_norm=False, pre_norm=False,
                                     residual=False, rope=False, seq_len=3, cache_len=3),
    "prenorm_only_mha": small_cfg(n_kv_heads=4, sub_norm=False, residual=False, rope=False,
                                  seq_len=2, cache_len=4),
    "qk_norm_gqa": small_cfg(qk_norm=True),
    "qk_norm_decode_swiglu": small_cfg(qk_norm=True, act="silu_mul", sub_norm=False, seq_len=1,
                                       cache_len=6, kv_layout="hsd"),
}


@pytest.mark.parametrize("case", sorted(FD_CASES))
def test_layer_backward_matches_finite_differences(case):
    cfg = FD_CASES[case]
    p, n1, x_in, k_prev, v_prev, dout = make_problem(cfg)
    out, cache = F.layer_forward(cfg, p, n1, x_in, k_prev, v_prev)
    r = Lyr.layer_backward(cfg, backward_inputs(cfg, p, cache), dout)

    def loss(pp, delta=None):
        o, _ = F.layer_forward(cfg, pp, n1, x_in, k_prev, v_prev, r1_delta=delta)
        return float(np.sum(dout * o))

    h = 1e-6
    for pname, gname in (("a_q", "dA_q"), ("b_q", "dB_q"), ("a_v", "dA_v"), ("b_v", "dB_v")):
        fd = np.zeros_like(p[pname])
        for idx in np.ndindex(*p[pname].shape):
            pp = dict(p)
            w = p[pname].copy()
            w[idx] += h
            pp[pname] = w
            lp = loss(pp)
            w = p[pname].copy()
            w[idx] -= h
            pp[pname] = w
            fd[idx] = (lp - loss(pp)) / (2 * h)
        an = r[gname]
        assert np.max(np.abs(fd - an)) <= 1e-6 * max(1.0, np.max(np.abs(an))), (case, gname)
        assert np.max(np.abs(an)) > 1e-3, (case, gname, "gradient unexpectedly tiny")
    fd = np.zeros((cfg.seq_len, cfg.dim))
    for idx in np.ndindex(*fd.shape):
        dl = np.zeros_like(fd)
        dl[idx] = h
        fd[idx] = (loss(p, dl) - loss(p, -dl)) / (2 * h)
    assert np.max(np.abs(fd - r["d_in"])) <= 1e-6 * max(1.0, np.max(np.abs(r["d_in"]))), case


EXACT_CASES = {
    "exact_all_norms_gqa": small_cfg(exact_din=True),
    "exact_qk_norm_swiglu": small_cfg(exact_din=True, qk_norm=True, act="silu_mul", sub_norm=False),
    "exact_decode_hsd": small_cfg(exact_din=True, seq_len=1, cache_len=6, kv_layout="hsd"),
    "exact_no_residual_no_prenorm_mha": small_cfg(exact_din=True, n_kv_heads=4, pre_norm=False,
                                                  residual=False, seq_len=4, cache_len=4),
}


@pytest.mark.parametrize("case", sorted(EXACT_CASES))
def test_exact_input_gradient_matches_finite_differences(case):
    """The exact layer-input gradient (through Q, K, V, their LoRA paths and the
    attention pre-norm, beyond the pages' truncation) against central differences in the
    layer input x_in of a forward where n1 = [RMSNorm(x_in)]."""
    cfg = EXACT_CASES[case]
    p, n1, x_in, k_prev, v_prev, dout = make_problem(cfg)
    out, cache = F.layer_forward(cfg, p, n1, x_in, k_prev, v_prev)
    r = Lyr.layer_backward(cfg, backward_inputs(cfg, p, cache), dout)

    def loss(xx):
        o, _ = F.layer_forward(cfg, p, n1, xx, k_prev, v_prev)
        return float(np.sum(dout * o))

    h = 1e-6
    fd = np.zeros_like(x_in)
    for idx in np.ndindex(*x_in.shape):
        xp, xm = x_in.copy(), x_in.copy()
        xp[idx] += h
        xm[idx] -= h
        fd[idx] = (loss(xp) - loss(xm)) / (2 * h)
    an = r["d_in"]
    assert np.max(np.abs(fd - an)) <= 1e-6 * max(1.0, np.max(np.abs(an))), case
    # the truncated reading differs from it by the Q / K / V paths, which are not small here
    assert np.max(np.abs(an - r["dR1"] * (1.0 if cfg.residual else 0.0))) > 1e-2, case


STACK_CASES = {
    "stack_truncated_all_norms_gqa": small_cfg(),
    "stack_truncated_swiglu_residual": small_cfg(act="silu_mul", sub_norm=False, pre_norm=False,
                                                 seq_len=4, cache_len=4),
    "stack_exact_prenorm_qk_norm": small_cfg(exact_din=True, qk_norm=True, sub_norm=False),
}


@pytest.mark.parametrize("case", sorted(STACK_CASES))
def test_stack_backward_matches_finite_differences(case):
    """The layer loop ([RS] backward_through_layers: layers in reverse, layer l's input
    gradient is layer l-1's output gradient, gnorm = sqrt of the sum over every layer of
    ||dA_q||^2 + ||dA_v||^2 with dB left out) against central differences of <dOut, out>
    of two composed layers with weights of their own, in both layers' adapters and in the
    stack input.  Also shows that the plausible mistakes (forward order, dOut handed to
    every layer, dB counted in the gnorm) would change the result by far more than the
    tolerance."""
    cfg = STACK_CASES[case]
    probs = [make_problem(cfg, seed=21 + l) for l in range(2)]
    params = [pr[0] for pr in probs]
    n1s = [pr[1] for pr in probs]
    x0 = probs[0][2]
    kps, vps = [pr[3] for pr in probs], [pr[4] for pr in probs]
    dout = probs[1][5]
    out, caches = F.stack_forward(cfg, params, n1s, x0, kps, vps)
    layers = [backward_inputs(cfg, params[l], caches[l]) for l in range(2)]
    res = Lyr.stack_backward(cfg, layers, dout)

    def loss(ps, x=x0):
        o, _ = F.stack_forward(cfg, ps, n1s, x, kps, vps)
        return float(np.sum(dout * o))

    h = 1e-6
    fd_sa = fd_sb = 0.0
    for l in range(2):
        for pname, gname in (("a_q", "dA_q"), ("b_q", "dB_q"), ("a_v", "dA_v"), ("b_v", "dB_v")):
            fd = np.zeros_like(params[l][pname])
            for idx in np.ndindex(*fd.shape):
                vals = []
                for sgn in (1.0, -1.0):
                    ps = [dict(p) for p in params]
                    w = params[l][pname].copy()
                    w[idx] += sgn * h
                    ps[l][pname] = w
                    vals.append(loss(ps))
                fd[idx] = (vals[0] - vals[1]) / (2 * h)
            an = res["layers"][l][gname]
            assert np.max(np.abs(fd - an)) <= 1e-6 * max(1.0, np.max(np.abs(an))), (case, l, gname)
            assert np.max(np.abs(an)) > 1e-3, (case, l, gname, "gradient unexpectedly tiny")
            if gname.startswith("dA"):
                fd_sa += float(np.sum(fd * fd))
            else:
                fd_sb += float(np.sum(fd * fd))
    fdx = np.zeros_like(x0)
    for idx in np.ndindex(*x0.shape):
        xp, xm = x0.copy(), x0.copy()
        xp[idx] += h
        xm[idx] -= h
        fdx[idx] = (loss(params, xp) - loss(params, xm)) / (2 * h)
    assert np.max(np.abs(fdx - res["d_in"])) <= 1e-6 * max(1.0, np.max(np.abs(res["d_in"]))), case
    # the reported norms against the finite-difference gradients themselves
    assert abs(res["gnorm"] - math.sqrt(fd_sa)) <= 1e-6 * math.sqrt(fd_sa), case
    assert abs(res["gnorm_full"] - math.sqrt(fd_sa + fd_sb)) <= 1e-6 * math.sqrt(fd_sa + fd_sb), case
    # the mistakes the pins must catch move the results well past the tolerance
    assert fd_sb > 1e-2 * fd_sa, (case, "dB too small to tell the gnorm readings apart")
    wrong = Lyr.layer_backward(cfg, layers[0], dout)          # layer 0 fed dOut, not d_in of layer 1
    assert np.max(np.abs(wrong["dA_q"] - res["layers"][0]["dA_q"])) > 1e-3 * np.max(np.abs(wrong["dA_q"])), case
    fwd = Lyr.layer_backward(cfg, layers[1], wrong["d_in"])    # forward order
    assert np.max(np.abs(fwd["dA_v"] - res["layers"][1]["dA_v"])) > 1e-3 * np.max(np.abs(fwd["dA_v"])), case


def test_packed_ternary_worked_bytes():
    """The 2-bit storage read by its definition (code = weight + 1): byte 0x91 = 10 01 00
    01 holds, from the lowest bits up, codes 1, 0, 1, 2 = 0, -1, 0, +1; 0x55 is four 0,
    0xAA four +1, 0x00 four -1; code 3 is refused."""
    got = ops.unpack_ternary2(np.array([[0x91, 0x00, 0x55, 0xAA]], dtype=np.uint8))
    assert got.tolist() == [[0, -1, 0, 1, -1, -1, -1, -1, 0, 0, 0, 0, 1, 1, 1, 1]]
    with pytest.raises(ValueError):
        ops.unpack_ternary2(np.array([[0x03]], dtype=np.uint8))


def test_packed_ternary_round_trip_and_layer():
    """The generator's packer and the oracle's unpacker are written apart: a round trip
    gives the ternary values back, and a layer with packed weights is the int8 layer."""
    from synth import DECODE, layer_inputs
    from synth.inputs import pack_ternary2
    w = np.random.default_rng(3).integers(-1, 2, size=(7, 64)).astype(np.int8)
    np.testing.assert_array_equal(ops.unpack_ternary2(pack_ternary2(w)), w)
    cfg = DECODE.with_(name="t2pin", dim=64, ffn_dim=128, n_heads=4, n_kv_heads=2, head_dim=16, rank=2,
                       lora_alpha=4.0, cache_len=9)
    d = layer_inputs(cfg)
    d2 = dict(d)
    for k in ("w_down", "w_gate", "w_up", "w_o"):
        d2[k] = pack_ternary2(d[k])
    a = Lyr.layer_backward(cfg, d, d["dout"])
    b = Lyr.layer_backward(cfg.with_(wtype="ternary2"), d2, d["dout"])
    for k in ("d_in", "dA_q", "dB_q", "dA_v", "dB_v"):
        np.testing.assert_array_equal(a[k], b[k])


def test_attention_from_logsumexp_is_the_softmax():
    """Recomputed weights exp(scale q.k - lse) against a softmax formed directly (max
    shift, exponent, row sum) over the visible keys, with GQA and a cache longer than the
    sequence: equal, masked keys zero, rows summing to one."""
    rs = np.random.default_rng(5)
    S, L, nh, nkv, hd, scale = 3, 7, 4, 2, 5, 0.37
    q = rs.normal(size=(S, nh, hd))
    K = rs.normal(size=(nkv, L, hd))
    pos0 = L - S
    want = np.zeros((nh, S, L))
    lse = np.zeros((nh, S))
    for h in range(nh):
        for i in range(S):
            z = np.array([scale * q[i, h] @ K[h // 2, j] for j in range(pos0 + i + 1)])
            e = np.exp(z - z.max())
            want[h, i, :pos0 + i + 1] = e / e.sum()
            lse[h, i] = z.max() + math.log(e.sum())
    got = ops.attention_from_logsumexp(q, K, lse, scale, pos0, nkv)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-14)
    np.testing.assert_allclose(got.sum(axis=-1), 1.0, rtol=0, atol=1e-14)


def test_recomputed_attention_layer_is_the_cached_one():
    """A layer whose attention weights are recomputed from q, K and the logsumexp gives the
    gradients of the same layer reading those weights from the cache (float64 on both
    sides), for the sequence and exact-gradient compositions."""
    from synth import layer_inputs
    for cfg in (small_cfg(name="rc", recompute_p=True, seq_len=3, cache_len=6),
                small_cfg(name="rc_exact", recompute_p=True, exact_din=True, qk_norm=True)):
        d = layer_inputs(cfg)
        K = Lyr.kv_heads_first(d["k"], cfg)
        q = d["q"].astype(np.float64).reshape(cfg.seq_len, cfg.n_heads, cfg.head_dim)
        d2 = dict(d)
        d2["attn"] = ops.attention_from_logsumexp(q, K, d["lse"], cfg.attn_scale, cfg.pos0, cfg.n_kv_heads)
        a = Lyr.layer_backward(cfg, d, d["dout"])
        b = Lyr.layer_backward(cfg.with_(recompute_p=False), d2, d["dout"])
        for k in ("d_in", "dA_q", "dB_q", "dA_v", "dB_v", "dQpre", "dV"):
            np.testing.assert_array_equal(a[k], b[k])


def test_linear_backward_is_the_adjoint():
    rs = np.random.default_rng(2)
    x, w, dy = rs.normal(size=(5, 7)), rs.normal(size=(7, 3)), rs.normal(size=(5, 3))
    lhs = np.sum(dy * (x @ (1.7 * w)))
    rhs = np.sum(ops.linear_backward(dy, w, 1.7) * x)
    assert abs(lhs - rhs) < 1e-12 * max(1.0, abs(lhs))


# ---------------------------------------------------------------- softmax backward

def test_softmax_backward_rows_sum_to_zero():
    rs = np.random.default_rng(3)
    z = rs.normal(size=(6, 40))
    a = np.exp(z) / np.exp(z).sum(-1, keepdims=True)
    ds = ops.softmax_backward(a, rs.normal(size=z.shape))
    assert np.max(np.abs(ds.sum(-1))) < 1e-14


def test_softmax_backward_finite_differences():
    rs = np.random.default_rng(4)
    z, da = rs.normal(size=(3, 9)), rs.normal(size=(3, 9))

    def sm(zz):
        e = np.exp(zz - zz.max(-1, keepdims=True))
        return e / e.sum(-1, keepdims=True)

    ds = ops.softmax_backward(sm(z), da)
    h = 1e-6
    fd = np.zeros_like(z)
    for idx in np.ndindex(*z.shape):
        zp, zm = z.copy(), z.copy()
        zp[idx] += h
        zm[idx] -= h
        fd[idx] = (np.sum(da * sm(zp)) - np.sum(da * sm(zm))) / (2 * h)
    assert np.max(np.abs(fd - ds)) < 1e-8


def test_softmax_backward_closed_forms():
    rs = np.random.default_rng(5)
    L = 16
    da = rs.normal(size=(2, L))
    uni = np.full((2, L), 1.0 / L)
    assert np.allclose(ops.softmax_backward(uni, da), (da - da.mean(-1, keepdims=True)) / L,
                       atol=1e-15)
    hot = np.zeros((2, L))
    hot[0, 3] = hot[1, 11] = 1.0
    assert np.max(np.abs(ops.softmax_backward(hot, da))) == 0.0
    # one-hot rows also kill dQ
    k = rs.normal(size=(L, 4))
    assert np.max(np.abs(ops.score_backward_q(ops.softmax_backward(hot, da), k, 0.5))) == 0.0


# ---------------------------------------------------------------- RoPE backward

def test_rope_backward_inverts_forward_and_keeps_norm():
    rs = np.random.default_rng(6)
    x = rs.normal(size=(7, 3, 16))
    pos = np.array([0, 1, 5, 100, 1023, 2047, 4000])
    y = F.rope(x, pos, 10000.0)
    assert np.max(np.abs(ops.rope_backward(y, pos, 10000.0) - x)) < 1e-12
    dy = rs.normal(size=x.shape)
    dx = ops.rope_backward(dy, pos, 10000.0)
    assert np.allclose(np.linalg.norm(dx, axis=-1), np.linalg.norm(dy, axis=-1), rtol=1e-13)
    # adjoint: <dy, R x> = <R^T dy, x>
    assert abs(np.sum(dy * y) - np.sum(dx * x)) < 1e-11
    # position 0 is the identity
    assert np.array_equal(ops.rope_backward(dy[:1], [0], 10000.0), dy[:1])


def test_rope_backward_angle_law_closed_form():
    # head_dim 4 -> two frequencies: theta_0 = pos, theta_1 = pos * base^(-1/2)
    pos, base = 3, 100.0
    dy = np.array([[[0.3, -1.2, 0.7, 2.0]]])
    dx = ops.rope_backward(dy, [pos], base)[0, 0]
    t0, t1 = 3.0, 0.3
    exp = [0.3 * math.cos(t0) + 0.7 * math.sin(t0), -1.2 * math.cos(t1) + 2.0 * math.sin(t1),
           -0.3 * math.sin(t0) + 0.7 * math.cos(t0), 1.2 * math.sin(t1) + 2.0 * math.cos(t1)]
    assert np.allclose(dx, exp, atol=1e-15)


# ---------------------------------------------------------------- RMSNorm backward

def test_rmsnorm_backward_finite_differences_and_invariance():
    rs = np.random.default_rng(7)
    x, g, dy = rs.normal(size=(4, 10)), rs.uniform(0.5, 1.5, 10), rs.normal(size=(4, 10))
    dx = ops.rmsnorm_backward(x, g, dy, 1e-3)
    h = 1e-6
    fd = np.zeros_like(x)
    for idx in np.ndindex(*x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        fd[idx] = (np.sum(dy * F.rmsnorm(xp, g, 1e-3)) - np.sum(dy * F.rmsnorm(xm, g, 1e-3))) / (2 * h)
    assert np.max(np.abs(fd - dx)) < 1e-8
    # eps = 0: RMSNorm(c x) = RMSNorm(x), so the gradient is orthogonal to x
    dx0 = ops.rmsnorm_backward(x, g, dy, 0.0)
    assert np.max(np.abs(np.sum(dx0 * x, -1))) < 1e-12


def test_rmsnorm_backward_constant_row_closed_form():
    # gamma = 1, x = c * ones, eps = 0: rms = |c| and dx = (dy - mean(dy)) / |c|
    dy = np.array([[1.0, -2.0, 0.5, 4.0, 0.0]])
    c = -2.5
    dx = ops.rmsnorm_backward(np.full((1, 5), c), np.ones(5), dy, 0.0)
    assert np.allclose(dx, (dy - dy.mean()) / abs(c), atol=1e-15)


# ---------------------------------------------------------------- gated activations

@pytest.mark.parametrize("act", ["relu2_mul", "silu_mul"])
def test_gated_backward_finite_differences(act):
    rs = np.random.default_rng(8)
    g, u, dh = rs.normal(size=(3, 11)), rs.normal(size=(3, 11)), rs.normal(size=(3, 11))
    g[np.abs(g) < 1e-3] = 0.5          # keep FD away from the ReLU kink
    fn = ops.relu2_mul_backward if act == "relu2_mul" else ops.silu_mul_backward
    dg, du = fn(g, u, dh)
    h = 1e-6
    for arr, an in ((g, dg), (u, du)):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(*arr.shape):
            keep = arr[idx]
            arr[idx] = keep + h
            lp = np.sum(dh * F.gated(g, u, act))
            arr[idx] = keep - h
            lm = np.sum(dh * F.gated(g, u, act))
            arr[idx] = keep
            fd[idx] = (lp - lm) / (2 * h)
        assert np.max(np.abs(fd - an)) < 1e-8


def test_gated_backward_special_values():
    g = np.array([-3.0, -1e-9, 0.0, 2.0])
    u = np.array([1.5, 2.0, -1.0, 0.5])
    dh = np.ones(4)
    dg, du = ops.relu2_mul_backward(g, u, dh)
    assert np.all(dg[:3] == 0.0) and np.all(du[:3] == 0.0)
    assert dg[3] == 2.0 * 0.5 * 2.0 and du[3] == 4.0
    dg, du = ops.silu_mul_backward(np.zeros(1), np.full(1, 3.0), np.ones(1))
    assert dg[0] == 1.5 and du[0] == 0.0          # silu'(0) = 1/2, silu(0) = 0


# ---------------------------------------------------------------- attention pieces

def test_gqa_equals_mha_with_duplicated_kv_heads():
    cfg = small_cfg(sub_norm=False, pre_norm=False, seq_len=4, cache_len=4)
    rs = np.random.default_rng(9)
    S, L, nh, hd = 4, 4, 4, 4
    logits = rs.normal(size=(nh, S, L))
    vis = np.arange(L)[None, :] <= np.arange(S)[:, None]
    a = np.where(vis, np.exp(logits), 0.0)
    a /= a.sum(-1, keepdims=True)
    k = rs.normal(size=(L, 2 * hd))
    v = rs.normal(size=(L, 2 * hd))
    w_o = rs.normal(size=(nh * hd, cfg.dim))
    d = dict(w_o=w_o, s_o=1.0, k=k, v=v, attn=a)
    dr1 = rs.normal(size=(S, cfg.dim))
    g = Lyr.attn_backward(cfg, d, dr1)
    dup = lambda t: np.concatenate([t[:, :hd], t[:, :hd], t[:, hd:], t[:, hd:]], axis=1)
    mcfg = cfg.with_(n_kv_heads=4)
    m = Lyr.attn_backward(mcfg, dict(d, k=dup(k), v=dup(v)), dr1)
    assert np.allclose(g["dQ"], m["dQ"], atol=1e-13)
    mv = m["dV"]
    assert np.allclose(g["dV"][:, :hd], mv[:, :hd] + mv[:, hd:2 * hd], atol=1e-13)
    assert np.allclose(g["dV"][:, hd:], mv[:, 2 * hd:3 * hd] + mv[:, 3 * hd:], atol=1e-13)


def test_lora_backward_closed_forms():
    rs = np.random.default_rng(10)
    G, h, x = rs.normal(size=(1, 6)), rs.normal(size=(1, 3)), rs.normal(size=(1, 5))
    B = rs.normal(size=(6, 3))
    da, db, gh = ops.lora_backward(G, h, x, B, alpha=6.0, rank=3)
    assert np.allclose(db, 2.0 * np.outer(G[0], h[0]), atol=1e-14)
    assert np.allclose(gh[0], 2.0 * np.array([np.dot(G[0], B[:, j]) for j in range(3)]), atol=1e-14)
    assert np.allclose(da, np.outer(gh[0], x[0]), atol=1e-14)
    da0, _, _ = ops.lora_backward(G, h, x, np.zeros_like(B), 6.0, 3)
    assert np.max(np.abs(da0)) == 0.0


# ---------------------------------------------------------------- AdamW

def test_adamw_first_step_moves_by_lr_sign():
    rs = np.random.default_rng(11)
    p, g = rs.normal(size=50), rs.normal(size=50)
    z = np.zeros(50)
    p1, m1, v1 = ops.adamw(p, g, z, z, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1)
    assert np.allclose(p1 - p, -1e-3 * g / (np.abs(g) + 1e-8), atol=1e-15)
    assert np.allclose(m1, 0.1 * g) and np.allclose(v1, 0.001 * g * g)


def test_adamw_bias_correction_constant_gradient():
    # constant gradient from zero moments: m_hat = g and v_hat = g^2 at every step
    p = np.array([0.5, -0.25])
    g = np.array([0.3, -2.0])
    m = v = np.zeros(2)
    for t in range(1, 8):
        p_new, m, v = ops.adamw(p, g, m, v, 1e-2, 0.9, 0.999, 0.0, 0.0, t)
        assert np.allclose(p_new - p, -1e-2 * np.sign(g), atol=1e-13)
        p = p_new


def test_adamw_decoupled_weight_decay():
    # zero gradient, zero moments: p <- p (1 - lr wd)
    p = np.array([1.0, -3.0, 0.25])
    z = np.zeros(3)
    p1, _, _ = ops.adamw(p, z, z, z, 0.1, 0.9, 0.999, 1e-8, 0.5, 1)
    assert np.allclose(p1, p * (1 - 0.05), atol=1e-15)


def test_adamw_first_step_with_decay_uses_the_old_parameter():
    # t = 1: m_hat = g and sqrt(v_hat) = |g|, so p1 = p - lr (g / (|g| + eps) + wd p)
    p = np.array([2.0, -1.0, 0.5])
    g = np.array([0.4, 0.1, -3.0])
    z = np.zeros(3)
    p1, _, _ = ops.adamw(p, g, z, z, 0.1, 0.9, 0.999, 1e-8, 0.5, 1)
    assert np.allclose(p1, p - 0.1 * (g / (np.abs(g) + 1e-8) + 0.5 * p), atol=1e-14)
    # decaying after the update instead would differ by lr^2 wd g/|g| = 5e-3
    assert np.max(np.abs(p1 - (p - 0.1 * g / np.abs(g)) * (1 - 0.05))) > 1e-3


def test_lora_plus_learning_rate_on_b():
    cfg = small_cfg(weight_decay=0.0)
    p, n1, x_in, k_prev, v_prev, dout = make_problem(cfg, seed=12)
    _, cache = F.layer_forward(cfg, p, n1, x_in, k_prev, v_prev)
    r = Lyr.layer_backward(cfg, backward_inputs(cfg, p, cache), dout)
    for t in ("q", "v"):
        da, db = r["dA_" + t], r["dB_" + t]
        assert np.allclose(r["a_" + t] - p["a_" + t], -cfg.lr * da / (np.abs(da) + cfg.adam_eps), atol=1e-15)
        assert np.allclose(r["b_" + t] - p["b_" + t],
                           -16.0 * cfg.lr * db / (np.abs(db) + cfg.adam_eps), atol=1e-15)


# ---------------------------------------------------------------- the page's own test

def test_page_literal_trainer_test():
    fx = json.load(open(os.path.join(HERE, "golden", "page_literal_fixture.json")))
    sh, hy = fx["shapes"], fx["hyper"]
    s, h, i, r = sh["seq_len"], sh["hidden"], sh["intermediate"], sh["rank"]
    cfg = LayerConfig(name="page", dim=h, ffn_dim=i, n_heads=sh["n_heads"],
                      n_kv_heads=sh["n_kv_heads"], head_dim=sh["head_dim"], rank=r,
                      lora_alpha=hy["lora_alpha"], seq_len=s, cache_len=s, act="silu_mul",
                      sub_norm=False, pre_norm=False, residual=False, rope=False,
                      lr=hy["lr"], beta1=hy["beta1"], beta2=hy["beta2"], adam_eps=hy["eps"],
                      weight_decay=hy["weight_decay"], step=hy["step"])
    c, a = fx["weights_constant"], fx["activations"]
    ramp = (np.arange(s * h) - 8.0) * 0.1
    rs = np.random.default_rng(13)
    layers = []
    for _ in range(sh["n_layers"]):
        d = dict(w_gate=np.full((h, i), c), w_up=np.full((h, i), c), w_down=np.full((i, h), c),
                 w_o=np.full((sh["q_dim"], h), c), s_gate=1.0, s_up=1.0, s_down=1.0, s_o=1.0,
                 x=ramp.reshape(s, h), gate=np.full((s, i), a["gate_output"]),
                 up=np.full((s, i), a["up_output"]), silu_gate=np.full((s, i), a["silu_gate"]),
                 k=np.full((s, sh["kv_dim"]), a["k"]), v=np.full((s, sh["kv_dim"]), a["v"]),
                 attn=np.full((sh["n_heads"], s, s), a["attn_weights"]),
                 lora_q_h=np.full((s, r), a["lora_q_h"]), lora_v_h=np.full((s, r), a["lora_v_h"]),
                 a_q=rs.normal(0, 0.02, (r, h)), b_q=rs.normal(0, 0.02, (sh["q_dim"], r)),
                 a_v=rs.normal(0, 0.02, (r, h)), b_v=rs.normal(0, 0.02, (sh["kv_dim"], r)))
        for p in ("a_q", "b_q", "a_v", "b_v"):
            d["m_" + p] = np.zeros_like(d[p])
            d["v_" + p] = np.zeros_like(d[p])
        layers.append(d)
    dout = ((np.arange(s * h) - 8.0) * 0.01).reshape(s, h)
    res = Lyr.stack_backward(cfg, layers, dout)
    assert not np.array_equal(res["layers"][0]["a_q"], layers[0]["a_q"])
    assert not np.array_equal(res["layers"][0]["a_v"], layers[0]["a_v"])
    assert res["gnorm"] >= 0.0
    assert np.all(np.isfinite(res["d_in"]))
