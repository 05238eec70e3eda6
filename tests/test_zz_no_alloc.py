"""The allocation-free LoRA gradient + AdamW entry point.

tlb_lora_grad_adamw_noalloc exists for callers that cannot allocate device memory
(and so cannot provide a workspace): its scratch is a fixed array inside the
library.  It must give what tlb_lora_grad_adamw gives.  This file is collected
last on purpose; it runs the two entry points on identical inputs twice in a row
(the second call sees the array holding the first call's rows) and compares
gradients, parameters and AdamW moments.
"""
import numpy as np
import pytest

from synth import SEQ512, layer_inputs
from tests.helpers import adam_to_abi, check, host, lora_dev, to_dev

pytestmark = pytest.mark.gpu

CFG = SEQ512.with_(name="noalloc", dim=512, ffn_dim=1024, n_heads=8, n_kv_heads=2, head_dim=64,
                   seq_len=300, cache_len=300, adam_state="warm", step=3)


def run_adapter(lib, use_noalloc, t, G, out_dim, tag, calls):
    import torch
    L = lora_dev(t)
    grads = {"dA_" + tag: torch.empty_like(L["a_" + tag]), "dB_" + tag: torch.empty_like(L["b_" + tag])}
    ss = torch.zeros(2, dtype=torch.float64, device="cuda")
    adam = adam_to_abi(lib, CFG)
    args = (CFG.seq_len, out_dim, CFG.dim, CFG.rank, CFG.lora_alpha, G, t["lora_%s_h" % tag], t["x"],
            lib.lora(L, tag, grads), adam, ss)
    outs = []
    for _ in range(calls):
        if use_noalloc:
            lib.lora_grad_adamw_noalloc(*args)
        else:
            ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
            lib.lora_grad_adamw(*args, ws)
        torch.cuda.synchronize()
        outs.append({k: host(v) for k, v in list(grads.items()) + [(p, L[p]) for p in L]})
    outs.append({"sumsq": ss.cpu().numpy()})
    return outs


@pytest.mark.parametrize("tag", ["q", "v"])
def test_noalloc_matches_workspace_entry_point(lib, tag):
    import torch
    d = layer_inputs(CFG)
    t = to_dev(d, CFG.wtype)
    out_dim = CFG.q_dim if tag == "q" else CFG.kv_dim
    G = torch.from_numpy(
        np.random.default_rng(5).normal(size=(CFG.seq_len, out_dim)).astype(np.float32)).cuda()
    ref = run_adapter(lib, False, t, G, out_dim, tag, calls=2)
    got = run_adapter(lib, True, t, G, out_dim, tag, calls=2)
    for call in range(2):
        for k in ref[call]:
            check("call %d %s" % (call, k), got[call][k], ref[call][k])
    assert np.allclose(got[2]["sumsq"], ref[2]["sumsq"], rtol=1e-5, atol=0)


def test_noalloc_rejects_oversized_calls(lib):
    import torch
    from transformer_layer_backward_gb300 import TlbError
    d = layer_inputs(CFG)
    t = to_dev(d, CFG.wtype)
    L = lora_dev(t)
    big_S = 65536 // CFG.rank + 1
    G = torch.zeros(big_S, CFG.q_dim, device="cuda")
    h = torch.zeros(big_S, CFG.rank, device="cuda")
    x = torch.zeros(big_S, CFG.dim, device="cuda")
    with pytest.raises(TlbError, match="exceeds the built-in scratch"):
        lib.lora_grad_adamw_noalloc(big_S, CFG.q_dim, CFG.dim, CFG.rank, CFG.lora_alpha, G, h, x,
                                    lib.lora(L, "q"), adam_to_abi(lib, CFG), None)
