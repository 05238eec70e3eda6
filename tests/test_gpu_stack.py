"""The stack entry point ([RS] backward_through_layers): layers n-1 .. 0, d_in of layer l
feeding layer l - 1.  Single-token layers overlap one layer's attention and LoRA kernels
with the next layer's GEMV chain on a second stream; the results must not depend on
that, so the stack is checked against the oracle's stack and against the same layers
called one at a time."""
import numpy as np
import pytest

from oracle import layer as OL
from synth import DECODE, TINY, layer_inputs
from oracle import ops
from tests.helpers import BF16_REL_L2, adam_to_abi, assert_route, cfg_to_abi, check, host, lora_dev, to_dev

pytestmark = pytest.mark.gpu

ADAPTER_KEYS = ("a_q", "b_q", "a_v", "b_v", "m_a_q", "v_a_q", "m_b_q", "v_b_q",
                "m_a_v", "v_a_v", "m_b_v", "v_b_v")


def device_stack(lib, cfg, layers, with_grads=False):
    """Each layer's inputs on the device; with_grads adds buffers the layer writes its
    adapter gradients into."""
    import torch
    devs = []
    for l, d in enumerate(layers):
        t = to_dev(d, cfg.wtype)
        L = lora_dev(t)
        c = cfg_to_abi(lib, cfg)
        g = ({k: torch.empty_like(L[k.replace("dA_", "a_").replace("dB_", "b_")])
              for k in ("dA_q", "dB_q", "dA_v", "dB_v")} if with_grads else None)
        devs.append(dict(t=t, L=L, g=g, w=lib.layer_weights(c, t), a=lib.layer_acts(c, t, cfg.kv_layout, cfg.cache_len),
                         lq=lib.lora(L, "q", g), lv=lib.lora(L, "v", g)))
    return devs


@pytest.mark.parametrize("n_layers,wtype", [(1, "ternary"), (2, "ternary"), (4, "ternary"), (2, "ternary2")])
def test_decode_stack_against_oracle(lib, n_layers, wtype):
    import torch
    cfg = DECODE.with_(name="decode_stack" if wtype == "ternary" else "decode_stack_t2", n_layers=n_layers,
                       wtype=wtype)
    layers = [layer_inputs(cfg, layer=l, seed=0, with_dout=(l == n_layers - 1)) for l in range(n_layers)]
    dout = layers[-1]["dout"]
    ref = OL.stack_backward(cfg, layers, dout)
    c = cfg_to_abi(lib, cfg)
    adam = adam_to_abi(lib, cfg)
    devs = device_stack(lib, cfg, layers)
    ws = lib.stack_workspace(c, 1, cfg.cache_len)
    dh = torch.from_numpy(dout).cuda()
    ss = torch.zeros(2, dtype=torch.float64, device="cuda")
    lib.stack_backward(c, 1, cfg.cache_len, [d["w"] for d in devs], [d["a"] for d in devs],
                       [d["lq"] for d in devs], [d["lv"] for d in devs], adam, dh, ss, ws)
    lib.workspace_status(ws)
    check("stack d_in", host(dh), ref["d_in"])
    gnorm = float(np.sqrt(ss[0].item()))
    assert abs(gnorm - ref["gnorm"]) <= 1e-5 * ref["gnorm"]


@pytest.mark.parametrize("n_layers", [2, 5])
def test_decode_stack_matches_layer_calls(lib, n_layers):
    """Same layers, same inputs: the overlapped stack and n_layers separate calls."""
    import torch
    cfg = DECODE.with_(name="decode_stack", n_layers=n_layers)
    layers = [layer_inputs(cfg, layer=l, seed=3, with_dout=(l == n_layers - 1)) for l in range(n_layers)]
    # the gradient grows ~5e3 times per synthetic ternary layer; a small dOut keeps dA^2 of
    # the lowest of five layers within float range (everything before AdamW is linear in it)
    dout = (layers[-1]["dout"] * 1e-8).astype(np.float32)
    c = cfg_to_abi(lib, cfg)
    adam = adam_to_abi(lib, cfg)
    a, b = device_stack(lib, cfg, layers), device_stack(lib, cfg, layers)
    ws_s = lib.stack_workspace(c, 1, cfg.cache_len)
    ws_l = lib.workspace(c, 1, cfg.cache_len)
    dh_s = torch.from_numpy(dout).cuda()
    dh_l = dh_s.clone()
    ss_s = torch.zeros(2, dtype=torch.float64, device="cuda")
    ss_l = torch.zeros(2, dtype=torch.float64, device="cuda")
    dout_dev = torch.from_numpy(dout).cuda()
    for rep in range(2):      # a second pass starts from the updated adapters and moments
        dh_s.copy_(dout_dev)
        dh_l.copy_(dout_dev)
        lib.stack_backward(c, 1, cfg.cache_len, [d["w"] for d in a], [d["a"] for d in a],
                           [d["lq"] for d in a], [d["lv"] for d in a], adam, dh_s, ss_s, ws_s)
        for l in reversed(range(n_layers)):
            lib.layer_backward(c, 1, cfg.cache_len, b[l]["w"], b[l]["a"], b[l]["lq"], b[l]["lv"], adam, dh_l, ss_l,
                               ws_l)
    lib.workspace_status(ws_s)
    # d_in runs through no atomic sum whose order could change: bit for bit
    np.testing.assert_array_equal(host(dh_s), host(dh_l))
    # the adapter gradients sum the heads' shares with float atomics, in either order
    for l in range(n_layers):
        for k in ADAPTER_KEYS:
            check("layer %d %s" % (l, k), host(a[l]["L"][k]), host(b[l]["L"][k]), rel_l2=1e-6, max_abs=None)
    # sum dA^2 inherits those ~1e-7 differences of dA
    np.testing.assert_allclose(ss_s.cpu().numpy(), ss_l.cpu().numpy(), rtol=1e-6)


def test_sequence_stack_runs_layers_in_turn(lib):
    """Layers with S > 1 take the plain loop on the caller's stream."""
    import torch
    cfg = TINY.with_(name="tiny_stack", n_layers=3)
    layers = [layer_inputs(cfg, layer=l, seed=0, with_dout=(l == cfg.n_layers - 1)) for l in range(3)]
    dout = layers[-1]["dout"]
    ref = OL.stack_backward(cfg, layers, dout)
    c = cfg_to_abi(lib, cfg)
    adam = adam_to_abi(lib, cfg)
    devs = device_stack(lib, cfg, layers)
    ws = lib.stack_workspace(c, cfg.seq_len, cfg.cache_len)
    dh = torch.from_numpy(dout).cuda()
    ss = torch.zeros(2, dtype=torch.float64, device="cuda")
    lib.stack_backward(c, cfg.seq_len, cfg.cache_len, [d["w"] for d in devs], [d["a"] for d in devs],
                       [d["lq"] for d in devs], [d["lv"] for d in devs], adam, dh, ss, ws)
    check("stack d_in", host(dh), ref["d_in"])
    gnorm = float(np.sqrt(ss[0].item()))
    assert abs(gnorm - ref["gnorm"]) <= 1e-5 * ref["gnorm"]
    for l in range(3):
        for p in ("a_q", "b_q", "a_v", "b_v"):
            check("layer %d %s" % (l, p), host(devs[l]["L"][p]), ref["layers"][l][p])


@pytest.mark.parametrize("variant", ["residual", "prenorm"])
def test_sequence_tensor_core_stack(lib, variant):
    """bf16 layers with S > 1: each layer's first product takes the bf16 copy of d_in that
    the layer above left in the workspace (written by the [W_gate | W_up]^T epilogue, or,
    with the pre-norm, by the O-projection's conversion).  Against the oracle's stack, and
    bit for bit against the same layers called one at a time (which convert d_hidden
    themselves)."""
    import torch
    from synth import SEQ512
    n_layers = 3
    cfg = SEQ512.with_(name="seq_stack", dim=512, ffn_dim=1024, n_heads=8, n_kv_heads=2, head_dim=64, rank=8,
                       lora_alpha=16.0, seq_len=200, cache_len=200, n_layers=n_layers,
                       pre_norm=(variant == "prenorm"))
    layers = [layer_inputs(cfg, layer=l, seed=4, with_dout=(l == n_layers - 1)) for l in range(n_layers)]
    dout = layers[-1]["dout"]
    ref = OL.stack_backward(cfg, layers, dout)
    c = cfg_to_abi(lib, cfg)
    adam = adam_to_abi(lib, cfg)
    a, b = device_stack(lib, cfg, layers, with_grads=True), device_stack(lib, cfg, layers)
    S, L = cfg.seq_len, cfg.cache_len
    ws_s = lib.stack_workspace(c, S, L)
    ws_l = lib.workspace(c, S, L)
    dh_s = torch.from_numpy(dout).cuda()
    dh_l = dh_s.clone()
    ss_s = torch.zeros(2, dtype=torch.float64, device="cuda")
    ss_l = torch.zeros(2, dtype=torch.float64, device="cuda")
    n0 = lib.launch_count()
    lib.stack_backward(c, S, L, [d["w"] for d in a], [d["a"] for d in a], [d["lq"] for d in a],
                       [d["lv"] for d in a], adam, dh_s, ss_s, ws_s)
    names = lib.launch_names(n0)
    assert_route(cfg, names)
    assert names.count("attn_tc_dq") == n_layers, names
    for l in reversed(range(n_layers)):
        lib.layer_backward(c, S, L, b[l]["w"], b[l]["a"], b[l]["lq"], b[l]["lv"], adam, dh_l, ss_l, ws_l)
    lib.workspace_status(ws_s)
    lib.workspace_status(ws_l)
    np.testing.assert_array_equal(host(dh_s), host(dh_l))
    for l in range(n_layers):
        for k in ("a_q", "b_q", "a_v", "b_v"):
            np.testing.assert_array_equal(host(a[l]["L"][k]), host(b[l]["L"][k]))
    # the stated bf16 tensor-core bar on d_in and on every layer's adapter gradients
    rel = {"d_in": check("stack d_in", host(dh_s), ref["d_in"], BF16_REL_L2, None)[0]}
    for l in range(n_layers):
        for k in ("dA_q", "dB_q", "dA_v", "dB_v"):
            rel["layer %d %s" % (l, k)] = check("layer %d %s" % (l, k), host(a[l]["g"][k]), ref["layers"][l][k],
                                               BF16_REL_L2, None)[0]
    print("bf16 %d-layer stack (%s), relative L2:" % (n_layers, variant), {k: "%.2e" % v for k, v in rel.items()})
    # parameters: AdamW of the GPU's own gradients, to float32 accuracy
    for l in range(n_layers):
        for tag in ("q", "v"):
            for p, lr in (("a_" + tag, cfg.lr), ("b_" + tag, cfg.lr * cfg.lr_b_mult)):
                g = host(a[l]["g"]["d" + p[0].upper() + "_" + tag])
                d = layers[l]
                rp, _, _ = ops.adamw(d[p], g, d["m_" + p], d["v_" + p], lr, cfg.beta1, cfg.beta2, cfg.adam_eps,
                                     cfg.weight_decay, cfg.step)
                check("layer %d %s" % (l, p), host(a[l]["L"][p]), rp)
    gnorm = float(np.sqrt(ss_s[0].item()))
    assert abs(gnorm - ref["gnorm"]) <= BF16_REL_L2 * ref["gnorm"]


@pytest.mark.parametrize("name", ["decode", "bf16_seq"])
def test_exact_input_gradient_stack_against_oracle(lib, name):
    """The exact layer-input gradient through a stack: each layer's d_in (through Q, K, V,
    the LoRA A paths and the pre-norm) is the dOut of the layer below; single-token layers
    run one after another (the overlap would hand dR1 down too early)."""
    import torch
    from synth import SEQ512
    if name == "decode":
        cfg = DECODE.with_(name="decode_exact_stack", dim=256, ffn_dim=512, n_heads=8, n_kv_heads=2, head_dim=64,
                           rank=4, lora_alpha=8.0, cache_len=100, wtype="f32", weight_std=0.05, n_layers=3,
                           exact_din=True)
        tol = (1e-5, 1e-4)
    else:
        cfg = SEQ512.with_(name="seq_exact_stack", dim=512, ffn_dim=1024, n_heads=8, n_kv_heads=2, head_dim=64,
                           rank=8, lora_alpha=16.0, seq_len=128, cache_len=160, n_layers=3, pre_norm=True,
                           exact_din=True)
        tol = (BF16_REL_L2, None)
    n = cfg.n_layers
    layers = [layer_inputs(cfg, layer=l, seed=6, with_dout=(l == n - 1)) for l in range(n)]
    dout = layers[-1]["dout"]
    ref = OL.stack_backward(cfg, layers, dout)
    c = cfg_to_abi(lib, cfg)
    devs = device_stack(lib, cfg, layers, with_grads=True)
    ws = lib.stack_workspace(c, cfg.seq_len, cfg.cache_len)
    dh = torch.from_numpy(dout).cuda()
    ss = torch.zeros(2, dtype=torch.float64, device="cuda")
    lib.stack_backward(c, cfg.seq_len, cfg.cache_len, [d["w"] for d in devs], [d["a"] for d in devs],
                       [d["lq"] for d in devs], [d["lv"] for d in devs], adam_to_abi(lib, cfg), dh, ss, ws)
    lib.workspace_status(ws)
    rel = {"d_in": check("stack d_in", host(dh), ref["d_in"], *tol)[0]}
    for l in range(n):
        for k in ("dA_q", "dB_q", "dA_v", "dB_v"):
            rel["layer %d %s" % (l, k)] = check("layer %d %s" % (l, k), host(devs[l]["g"][k]), ref["layers"][l][k],
                                               *tol)[0]
    print("exact %s stack, relative L2:" % name, {k: "%.2e" % v for k, v in rel.items()})
