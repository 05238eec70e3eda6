"""Full-size sequence configuration (S = L = 2048, dim 2560, ffn 9728, 32/8 heads of 128,
SwiGLU, RoPE, residual, bf16 weights, LoRA rank 16): one layer against the float64
oracle, and the 36-layer stack through its linearity in dOut.

The gradient that leaves a layer (dR1) does not depend on the adapters (the pages stop
the backward at the Q / V projection outputs), so the stack's d_in is linear in the dOut
that enters it even though every layer's AdamW step moves the adapters between calls:
  stack(a u + b w) = a stack(u) + b stack(w).
That property holds at any size and checks the whole 36-layer chain of tcgen05 GEMMs,
tensor-core attention and tiled LoRA against itself at full scale.
"""
import numpy as np
import pytest

from oracle import layer as OL
from synth import STACK2048, layer_inputs
from tests.helpers import BF16_REL_L2, adam_to_abi, assert_route, cfg_to_abi, check, host, lora_dev, to_dev

pytestmark = pytest.mark.gpu

LAYER = STACK2048.with_(name="layer2048", n_layers=1)


@pytest.mark.parametrize("mode", ["truncated", "exact_din", "recompute"])
def test_full_size_layer_against_oracle(lib, mode):
    import torch
    exact = mode == "exact_din"
    cfg = {"truncated": LAYER, "exact_din": LAYER.with_(name="layer2048_exact", exact_din=True),
           "recompute": LAYER.with_(name="layer2048_recompute", recompute_p=True)}[mode]
    d = layer_inputs(cfg, layer=0, seed=0)
    ref = OL.layer_backward(cfg, d, d["dout"])
    t = to_dev(d, cfg.wtype)
    c = cfg_to_abi(lib, cfg)
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
    assert_route(cfg, lib.launch_names(n0))
    lib.workspace_status(ws)
    rel = {"d_in": check("d_in", host(dh), ref["d_in"], BF16_REL_L2, None)[0]}
    for k in ("dA_q", "dB_q", "dA_v", "dB_v"):
        rel[k] = check(k, host(grads[k]), ref[k], BF16_REL_L2, None)[0]
    print("full-size layer (%s): relative L2" % mode, {k: "%.2e" % v for k, v in rel.items()})
    s = ss.cpu().numpy()
    assert abs(s[0] - ref["sumsq_a"]) <= 2 * BF16_REL_L2 * ref["sumsq_a"]
    assert abs(s[1] - ref["sumsq_b"]) <= 2 * BF16_REL_L2 * ref["sumsq_b"]


def test_full_stack_is_linear_in_dout(lib):
    import torch
    from synth.device import device_layer
    cfg = STACK2048
    S, L, depth = cfg.seq_len, cfg.cache_len, cfg.n_layers
    c = cfg_to_abi(lib, cfg)
    adam = adam_to_abi(lib, cfg)
    layers = []
    for l in range(2):                      # two distinct layers, alternating through the stack
        t = device_layer(cfg, l, seed=11)
        # the dict keeps the tensors alive: the ABI structs hold raw device pointers
        layers.append(dict(t=t, w=lib.layer_weights(c, t), a=lib.layer_acts(c, t, cfg.kv_layout, L),
                           lq=lib.lora(t, "q"), lv=lib.lora(t, "v")))
    ws = lib.workspace(c, S, L)
    ss = torch.zeros(2, dtype=torch.float64, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    u = torch.randn(S, cfg.dim, device="cuda", generator=g)
    w = torch.randn(S, cfg.dim, device="cuda", generator=g)
    a_, b_ = 0.75, -1.25

    sws = lib.stack_workspace(c, S, L)
    sW, sA, sQ, sV = ([layers[j % 2][k] for j in range(depth)] for k in ("w", "a", "lq", "lv"))

    def stack(dout):
        dh = dout.clone()
        n0 = lib.launch_count()
        lib.stack_backward(c, S, L, sW, sA, sQ, sV, adam, dh, ss, sws)
        names = lib.launch_names(n0)
        assert_route(cfg, names)
        assert names.count("attn_tc_dq") == depth
        lib.workspace_status(sws)
        return host(dh)

    yu, yw, yc = stack(u), stack(w), stack(a_ * u + b_ * w)
    assert np.all(np.isfinite(yc)) and np.linalg.norm(yu) > 0
    # d_in runs through stream-K GEMMs whose shared tiles are summed in a fixed order and
    # through elementwise epilogues, none of which reads the adapters that AdamW moved in
    # between: a repeat is bit-identical
    np.testing.assert_array_equal(stack(u), yu)
    # every layer rounds its GEMM operands to bf16 afresh and the two sides round different
    # values, so their independent errors add in quadrature over the depth
    rel, _ = check("stack(a u + b w)", yc, a_ * yu + b_ * yw, BF16_REL_L2 * np.sqrt(depth), None)
    print("stack linearity: relative L2 %.3e" % rel)
