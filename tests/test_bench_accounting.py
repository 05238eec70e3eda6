"""The bench's algorithmic flop counts, the numerators of its tensor roofline fractions,
checked against the products of the layer backward written out one by one with their
shapes ([FFN] "Backward (reverse)", [ATT] "Gradient Flow", [RS] LoRA Q / V backward),
and against a brute-force count of the (query, key) pairs a causal row sees."""
import pytest

import bench
from synth import SEQ512, STACK2048


def visible_pairs(S, L):
    # query row i sits at position L - S + i and sees keys 0 .. L - S + i
    return sum(1 for i in range(S) for j in range(L) if j <= L - S + i)


def products(cfg):
    """(product, multiply-adds) of one layer backward on the sequence path."""
    S, L, H, I, r = cfg.seq_len, cfg.cache_len, cfg.dim, cfg.ffn_dim, cfg.rank
    P = visible_pairs(S, L)
    hd, nh = cfg.head_dim, cfg.n_heads
    out = [
        ("dF = dOut W_down^T           [S, H] x [H, I]", S * H * I),
        ("dN2 = [dG | dU] [W_g | W_u]^T [S, 2I] x [2I, H]", S * 2 * I * H),
        ("dSub = dR1 W_O^T             [S, H] x [H, q_dim]", S * H * cfg.q_dim),
        ("dAttn = dCtx V^T over visible pairs", P * hd * nh),
        ("dQ = dS K over visible pairs", P * hd * nh),
        ("dV = attn^T dCtx over visible pairs", P * hd * nh),
    ]
    for od in (cfg.q_dim, cfg.kv_dim):
        out += [("dB = G^T h   [od, S] x [S, r]", od * S * r),
                ("gh = G B_old [S, od] x [od, r]", S * od * r),
                ("dA = gh^T x  [r, S] x [S, H]", r * S * H)]
    return out


SMALL = SEQ512.with_(name="small_ragged", dim=96, ffn_dim=160, n_heads=6, n_kv_heads=2, head_dim=16,
                     rank=4, seq_len=7, cache_len=19)


@pytest.mark.parametrize("cfg", [SMALL, SEQ512.with_(name="small_square", seq_len=9, cache_len=9), SEQ512],
                         ids=lambda c: c.name)
def test_layer_flops_are_the_listed_products(cfg):
    assert bench.seq_layer_flops(cfg) == 2 * sum(m for _, m in products(cfg))


def test_per_kernel_flops_of_the_tensor_core_layer():
    cfg = SMALL
    P = visible_pairs(cfg.seq_len, cfg.cache_len)
    names = ["to_bf16", "tcgen05 gemm", "tcgen05 gemm", "tcgen05 gemm fixup", "tcgen05 gemm", "attn_tc_prep",
             "attn_tc_dq", "attn_tc_dv", "attn_tc_dv_sum"]
    got = bench.seq_kernel_flops(cfg, names)
    S, H, I = cfg.seq_len, cfg.dim, cfg.ffn_dim
    want = [0, 2 * S * H * I, 2 * S * 2 * I * H, 0, 2 * S * H * cfg.q_dim, 0,
            2 * 2 * P * cfg.head_dim * cfg.n_heads, 2 * P * cfg.head_dim * cfg.n_heads, 0]
    assert [f for f, _ in got] == want
    assert [k for _, k in got] == [None, "bf16", "bf16", None, "bf16", None, "tf32", "tf32", None]


def test_stack_step_is_36_layers():
    # the default line's step: the 36-layer S = L = 2048 stack; pairs in closed form there
    cfg = STACK2048
    S = cfg.seq_len
    assert visible_pairs(64, 64) == 64 * 65 // 2
    per_layer = 2 * sum(m for _, m in products(cfg.with_(seq_len=64, cache_len=64)))
    assert per_layer == bench.seq_layer_flops(cfg.with_(seq_len=64, cache_len=64))
    assert bench.seq_layer_flops(cfg) == (2 * S * cfg.dim * cfg.ffn_dim * 3 + 2 * S * cfg.dim * cfg.q_dim +
                                          3 * 2 * (S * (S + 1) // 2) * cfg.head_dim * cfg.n_heads +
                                          2 * 2 * S * cfg.rank * (cfg.q_dim + cfg.kv_dim) +
                                          2 * 2 * S * cfg.rank * cfg.dim)


def test_attention_kernel_bytes():
    cfg = SMALL
    S, L, qd, kvd = cfg.seq_len, cfg.cache_len, cfg.q_dim, cfg.kv_dim
    weights = 4 * cfg.n_heads * visible_pairs(S, L)
    got = bench.seq_kernel_bytes(cfg, ["tcgen05 gemm", "attn_tc_prep", "attn_tc_dq", "attn_tc_dv", "lora_tc_gpass"])
    assert got == [0, 0, weights + 4 * (S * qd + L * kvd + L * kvd + S * qd), weights + 4 * (S * qd + S * kvd), 0]


def test_per_kernel_entries_of_a_layer_line():
    # the kernels of one S = L = 2048 layer call and live times of the same order as the
    # bench line's; the weight products carry flops, the attention kernels flops and bytes
    cfg = STACK2048.with_(n_layers=1)
    names = ["to_bf16", "tcgen05 gemm", "tcgen05 gemm", "tcgen05 gemm fixup", "tcgen05 gemm", "attn_tc_prep",
             "attn_tc_dq", "attn_tc_dv", "attn_tc_dv_sum", "lora_tc_gpass", "lora_gh_sum", "lora_tc_xpass",
             "lora_seq_adamw"]
    ms = [0.0082, 0.0891, 0.1219, 0.0096, 0.0399, 0.0146, 0.1184, 0.0654, 0.0102, 0.0194, 0.0070, 0.0141, 0.0090]
    peak_of = {"bf16": 1750.0, "tf32": 921.0, "fp32": 80.0}
    fl = bench.seq_kernel_flops(cfg, names)
    kb = bench.seq_kernel_bytes(cfg, names)
    e = bench.kernel_entries(names, ms, fl, kb, peak_of, 6702.2)
    assert [x["kernel"] for x in e] == names
    assert [x.get("operands") for x in e] == [None, "bf16", "bf16", None, "bf16", None, "tf32", "tf32", None,
                                              None, None, None, None]
    gate_up = e[2]
    assert gate_up["flop"] == 2 * 2048 * 2560 * 2 * 9728
    assert gate_up["frac"] == pytest.approx(gate_up["flop"] / 0.1219e-3 / 1e12 / 1750.0)
    dq, dv = e[6], e[7]
    assert dq["bytes"] == 4 * 32 * (2048 * 2049 // 2) + 4 * (2 * 2048 * 4096 + 2 * 2048 * 1024)
    assert dq["hbm_frac"] == pytest.approx(dq["bytes"] / 0.1184e-3 / 1e9 / 6702.2)
    assert 0.4 < dq["hbm_frac"] < 0.5 and 0.3 < dq["frac"] < 0.35      # bound by its bytes, not its flops
    assert dv["bytes"] == 4 * 32 * (2048 * 2049 // 2) + 4 * (2048 * 4096 + 2048 * 1024)
    assert "bytes" not in e[1] and "flop" not in e[0]
