"""Failure detection on the device, in the forms that fault no GPU.

* TLB_CHECK_FINITE ([RS] backward_through_layers, contract C-WGPU-TRAIN-007: the
  grad_hidden that enters is finite): a NaN planted on the host in the dOut of a layer,
  or in a cached activation so that a layer's dR1 turns non-finite, is reported as
  TLB_ENONFINITE by tlb_workspace_status, and no adapter below that point takes its AdamW
  step.  With finite inputs the flag changes no result.
* The bounded waits: the test hook makes one block of the persistent single-token kernel
  skip its arrival at a global-memory grid barrier (a flag that nothing else sets), every
  block's wait runs out after about a second, the call reports TLB_ETIMEOUT, and the next
  call on the same workspace gives the oracle's result again.
"""
import numpy as np
import pytest

from oracle import layer as OL
from synth import DECODE, SEQ512, TINY, layer_inputs
from tests.helpers import BF16_REL_L2, adam_to_abi, check, host, lora_dev, to_dev

pytestmark = pytest.mark.gpu

ADAPTERS = ("a_q", "b_q", "a_v", "b_v", "m_a_q", "v_a_q", "m_b_q", "v_b_q", "m_a_v", "v_a_v", "m_b_v", "v_b_v")
DEC_SMALL = DECODE.with_(name="dec_small", dim=256, ffn_dim=512, n_heads=8, n_kv_heads=2, head_dim=64,
                         rank=4, lora_alpha=8.0, cache_len=100, wtype="f32", weight_std=0.05)
SEQ_SMALL = SEQ512.with_(name="seq_small", dim=512, ffn_dim=1024, n_heads=8, n_kv_heads=2, head_dim=64,
                         rank=8, lora_alpha=16.0, seq_len=200, cache_len=200)
CASES = {c.name: c for c in (TINY, DEC_SMALL, SEQ_SMALL)}


def run_layer(lib, cfg, d, check_finite, persistent=False, ws=None, dout=None):
    import torch
    t = to_dev(d, cfg.wtype)
    c = lib.layer_cfg_of(cfg, persistent=persistent, check_finite=check_finite)
    ws = lib.workspace(c, cfg.seq_len, cfg.cache_len) if ws is None else ws
    L = lora_dev(t)
    dh = (t["dout"] if dout is None else torch.from_numpy(dout).cuda()).clone()
    ss = torch.zeros(2, dtype=torch.float64, device="cuda")
    lib.layer_backward(c, cfg.seq_len, cfg.cache_len, lib.layer_weights(c, t),
                       lib.layer_acts(c, t, cfg.kv_layout, cfg.cache_len), lib.lora(L, "q"), lib.lora(L, "v"),
                       adam_to_abi(lib, cfg), dh, ss, ws)
    return dh, L, ss, ws


@pytest.mark.parametrize("name", sorted(CASES))
def test_check_finite_changes_nothing_on_finite_input(lib, name):
    cfg = CASES[name]
    d = layer_inputs(cfg, layer=0, seed=0)
    a = run_layer(lib, cfg, d, check_finite=False)
    b = run_layer(lib, cfg, d, check_finite=True)
    lib.workspace_status(a[3])
    lib.workspace_status(b[3])          # TLB_OK: raises otherwise
    # the same kernels (float atomics may sum in another order: the single-token chain
    # combines column ranges that way)
    check("d_in", host(b[0]), host(a[0]), rel_l2=1e-6, max_abs=None)
    for k in ADAPTERS:
        check(k, host(b[1][k]), host(a[1][k]), rel_l2=1e-6, max_abs=None)


@pytest.mark.parametrize("name", sorted(CASES))
def test_nan_in_dout_is_reported_and_skips_adamw(lib, name):
    cfg = CASES[name]
    d = layer_inputs(cfg, layer=0, seed=0)
    dout = d["dout"].copy()
    dout[cfg.seq_len // 2, 3] = np.nan
    dh, L, ss, ws = run_layer(lib, cfg, d, check_finite=True, dout=dout)
    with pytest.raises(lib.TlbError) as e:
        lib.workspace_status(ws)
    assert e.value.code == lib._abi.TLB_ENONFINITE
    assert "dOut" in str(e.value)
    for k in ADAPTERS:                  # adapters and moments untouched
        np.testing.assert_array_equal(host(L[k]), d[k].astype(np.float32).astype(np.float64), err_msg=k)
    lib.workspace_status(ws)            # the status was cleared by the read


def test_nan_inside_a_stack_stops_the_steps_below(lib):
    """A NaN in layer 1's cached up projection makes layer 1's dR1 non-finite (a NaN in
    the ReLU^2 gate would not: max(0, NaN) is 0 there): layers 3 and 2 (run before it)
    take their steps as in a clean run, layers 1 and 0 take none."""
    import torch
    n = 4
    cfg = DEC_SMALL.with_(name="dec_small_stack", n_layers=n)
    layers = [layer_inputs(cfg, layer=l, seed=2, with_dout=(l == n - 1)) for l in range(n)]
    bad = [dict(x) for x in layers]
    bad[1]["up"] = bad[1]["up"].copy()
    bad[1]["up"][0, 5] = np.nan

    def run(src, chk):
        c = lib.layer_cfg_of(cfg, check_finite=chk)
        devs = []
        for x in src:
            t = to_dev(x, cfg.wtype)
            L = lora_dev(t)
            devs.append(dict(t=t, L=L, w=lib.layer_weights(c, t), a=lib.layer_acts(c, t, cfg.kv_layout, cfg.cache_len),
                             lq=lib.lora(L, "q"), lv=lib.lora(L, "v")))
        ws = lib.stack_workspace(c, 1, cfg.cache_len)
        dh = torch.from_numpy(layers[-1]["dout"]).cuda()
        ss = torch.zeros(2, dtype=torch.float64, device="cuda")
        lib.stack_backward(c, 1, cfg.cache_len, [x["w"] for x in devs], [x["a"] for x in devs],
                           [x["lq"] for x in devs], [x["lv"] for x in devs], adam_to_abi(lib, cfg), dh, ss, ws)
        return devs, ws

    clean, ws_c = run(layers, True)
    lib.workspace_status(ws_c)
    dirty, ws_d = run(bad, True)
    with pytest.raises(lib.TlbError) as e:
        lib.workspace_status(ws_d)
    assert e.value.code == lib._abi.TLB_ENONFINITE and "dR1" in str(e.value)
    for l in (3, 2):
        for k in ADAPTERS:
            check("layer %d %s" % (l, k), host(dirty[l]["L"][k]), host(clean[l]["L"][k]), rel_l2=1e-6, max_abs=None)
    for l in (1, 0):
        for k in ADAPTERS:
            np.testing.assert_array_equal(host(dirty[l]["L"][k]), layers[l][k].astype(np.float32).astype(np.float64),
                                          err_msg="layer %d %s" % (l, k))


def test_bounded_wait_runs_out_and_the_workspace_stays_usable(lib):
    cfg = DEC_SMALL
    d = layer_inputs(cfg, layer=0, seed=0)
    ref = OL.layer_backward(cfg, d, d["dout"])
    lib.debug_skip_barrier_arrival(3)
    try:
        _, _, _, ws = run_layer(lib, cfg, d, check_finite=False, persistent=True)
    finally:
        lib.debug_skip_barrier_arrival(-1)
    with pytest.raises(lib.TlbError) as e:
        lib.workspace_status(ws)
    assert e.value.code == lib._abi.TLB_ETIMEOUT
    # the same workspace: the barrier counter was put back by the kernel that timed out
    dh, L, ss, ws = run_layer(lib, cfg, d, check_finite=False, persistent=True, ws=ws)
    lib.workspace_status(ws)
    check("d_in after a timeout", host(dh), ref["d_in"])
    for p in ("a_q", "b_q", "a_v", "b_v"):
        check(p, host(L[p]), ref[p])
