"""The seeded input generator against the recipe it states: shapes of the named
workloads, value sets and ranges, the masked softmax rows (and their logsumexp when the
weights are recomputed), and the caches formed from drawn values.  Host only."""
import numpy as np
import pytest

from synth import DECODE, SEQ512, STACK2048, TINY, layer_inputs
from synth import rng
from synth.inputs import pack_ternary2


def test_named_workload_shapes():
    assert (TINY.dim, TINY.ffn_dim, TINY.n_heads, TINY.n_kv_heads, TINY.head_dim) == (64, 256, 4, 2, 16)
    assert (TINY.seq_len, TINY.cache_len) == (32, 32)
    assert (DECODE.dim, DECODE.ffn_dim, DECODE.n_heads, DECODE.n_kv_heads, DECODE.head_dim) == (2560, 6912, 20, 5, 128)
    assert (DECODE.seq_len, DECODE.cache_len, DECODE.pos0) == (1, 1024, 1023)
    assert (SEQ512.dim, SEQ512.ffn_dim, SEQ512.n_heads, SEQ512.n_kv_heads, SEQ512.head_dim) == (2560, 9728, 32, 8, 128)
    assert SEQ512.seq_len == SEQ512.cache_len == 512 and SEQ512.wtype == "bf16" and SEQ512.rank == 16
    assert STACK2048.seq_len == STACK2048.cache_len == 2048 and STACK2048.n_layers == 36
    assert (STACK2048.dim, STACK2048.ffn_dim, STACK2048.q_dim, STACK2048.kv_dim) == (2560, 9728, 4096, 1024)


def test_streams_are_seeded_and_distinct():
    a = layer_inputs(TINY, layer=0, seed=3)
    b = layer_inputs(TINY, layer=0, seed=3)
    c = layer_inputs(TINY, layer=1, seed=3)
    for k in a:
        assert np.array_equal(a[k], b[k]), k
    assert not np.array_equal(a["gate"], c["gate"])
    assert not np.array_equal(a["gate"], a["up"])           # one stream per tensor


def test_normal_and_uniform_streams():
    z = rng.normal(rng.stream_key(0, "recipe", 0, "z"), 200_000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    u = rng.uniform(rng.stream_key(0, "recipe", 0, "u"), 200_000, 0.5, 1.5)
    assert u.min() >= 0.5 and u.max() < 1.5 and abs(u.mean() - 1.0) < 0.01


SMALL_DECODE = DECODE.with_(name="recipe_decode", dim=256, ffn_dim=384, n_heads=4, n_kv_heads=2, head_dim=64,
                            rank=4, lora_alpha=8.0, cache_len=96)
SMALL_SEQ = SEQ512.with_(name="recipe_seq", dim=128, ffn_dim=256, n_heads=4, n_kv_heads=2, head_dim=32,
                         rank=4, lora_alpha=8.0, seq_len=24, cache_len=40, use_silu_cache=True,
                         adam_state="warm", step=3)


def test_ternary_weights_and_packing():
    d = layer_inputs(SMALL_DECODE, seed=1)
    w = d["w_gate"]
    assert w.dtype == np.int8 and set(np.unique(w)) <= {-1, 0, 1}
    frac = [(w == v).mean() for v in (-1, 0, 1)]
    assert all(abs(f - 1 / 3) < 0.02 for f in frac), frac
    for s in ("s_down", "s_gate", "s_up", "s_o"):
        assert 0.5 <= d[s] < 2.0
    packed = pack_ternary2(w)
    codes = np.stack([(packed >> (2 * i)) & 3 for i in range(4)], axis=-1)
    assert codes.max() <= 2                                  # 3 is never a weight's code
    assert np.array_equal(codes.reshape(w.shape).astype(np.int16) - 1, w)


def test_bf16_weights_are_exact_bf16():
    d = layer_inputs(SMALL_SEQ, seed=2)
    for k in ("w_down", "w_gate", "w_up", "w_o"):
        bits = d[k].astype(np.float32).view(np.uint32)
        assert np.all(bits & 0xFFFF == 0), k
        assert abs(d[k].std() - SMALL_SEQ.weight_std) < 0.1 * SMALL_SEQ.weight_std


@pytest.mark.parametrize("cfg", [TINY, SMALL_DECODE, SMALL_SEQ], ids=lambda c: c.name)
def test_attention_rows_are_masked_softmax_rows(cfg):
    d = layer_inputs(cfg, seed=4)
    P = d["attn"].astype(np.float64)
    S, L = cfg.seq_len, cfg.cache_len
    assert P.shape == (cfg.n_heads, S, L)
    vis = np.arange(L)[None, :] <= (cfg.pos0 + np.arange(S))[:, None]
    assert np.all(P[:, ~vis] == 0.0)
    assert np.all(P[:, vis] > 0.0)
    assert np.allclose(P.sum(axis=-1), 1.0, atol=1e-5)


def test_recomputed_weights_follow_their_logsumexp():
    cfg = SMALL_SEQ.with_(name="recipe_rc", recompute_p=True)
    d = layer_inputs(cfg, seed=5)
    S, L, hd, g = cfg.seq_len, cfg.cache_len, cfg.head_dim, cfg.n_heads // cfg.n_kv_heads
    K = d["k"].astype(np.float64).reshape(L, cfg.n_kv_heads, hd)
    q = d["q"].astype(np.float64).reshape(S, cfg.n_heads, hd)
    vis = np.arange(L)[None, :] <= (cfg.pos0 + np.arange(S))[:, None]
    for h in range(cfg.n_heads):
        z = cfg.attn_scale * q[:, h, :] @ K[:, h // g, :].T
        e = np.where(vis, np.exp(z - d["lse"][h].astype(np.float64)[:, None]), 0.0)
        assert np.allclose(e.sum(axis=-1), 1.0, atol=1e-5)
        assert np.allclose(e, d["attn"][h], atol=1e-6)


def test_gains_moments_and_derived_caches():
    cfg = SMALL_SEQ.with_(name="recipe_norms", sub_norm=True, pre_norm=True, qk_norm=True)
    d = layer_inputs(cfg, seed=6)
    for k in ("g_sub_ffn", "g_sub_attn", "g_ffn", "g_q"):
        assert d[k].min() >= 0.5 and d[k].max() < 1.5, k
    for p in ("a_q", "b_q", "a_v", "b_v"):
        assert d["v_" + p].min() >= 0.0 and d["v_" + p].max() < 1e-4
        assert abs(d["m_" + p].std() - 1e-2) < 2e-3
    g = d["gate"].astype(np.float64)
    assert np.allclose(d["silu_gate"], g / (1.0 + np.exp(-g)), rtol=1e-6, atol=1e-7)
    x = d["x"].astype(np.float64)
    assert np.allclose(d["lora_q_h"], x @ d["a_q"].astype(np.float64).T, rtol=1e-5, atol=1e-6)
    assert np.allclose(d["lora_v_h"], x @ d["a_v"].astype(np.float64).T, rtol=1e-5, atol=1e-6)
    cold = layer_inputs(SMALL_SEQ.with_(name="recipe_cold", adam_state="zeros"), seed=6)
    assert not any(cold["m_" + p].any() or cold["v_" + p].any() for p in ("a_q", "b_q", "a_v", "b_v"))
