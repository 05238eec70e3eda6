"""CPU-side checks of the C ABI library: it builds for sm_103a, loads, exports every
symbol the header declares, and rejects bad arguments on the host before any
device work (no GPU needed: these paths return before the first CUDA call)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from transformer_layer_backward_gb300 import build, _abi
    build.build()
    return _abi.load()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "tlb.h")).read()
    return sorted(set(re.findall(r"^\s*(?:const char \*|int |size_t |void |uint64_t )(tlb_\w+)\(", text, re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("tlb_layer_backward", "tlb_attn_backward", "tlb_ffn_backward", "tlb_rmsnorm_backward",
              "tlb_rope_backward", "tlb_lora_grad_adamw", "tlb_softmax_backward", "tlb_act_backward"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from transformer_layer_backward_gb300 import _abi
    for n in declared_functions():
        assert hasattr(lib, n), n
        assert n in _abi.SIGNATURES, "binding lacks " + n


def test_host_side_argument_errors(lib):
    from transformer_layer_backward_gb300 import _abi as A
    assert lib.tlb_softmax_backward(None, None, None, -1, 4, None) == A.TLB_EINVAL
    assert b"negative" in lib.tlb_last_error()
    assert lib.tlb_softmax_backward(None, None, None, 0, 0, None) == A.TLB_OK    # empty: no-op
    assert lib.tlb_softmax_backward(None, None, None, 3, 4, None) == A.TLB_EINVAL
    assert lib.tlb_act_backward(7, None, None, None, None, None, None, 4, None) == A.TLB_EINVAL
    assert lib.tlb_rope_backward(None, None, 2, 2, 5, 0, 1e4, None) == A.TLB_EINVAL     # odd head_dim
    assert lib.tlb_rope_backward(None, None, 2, 2, 512, 0, 1e4, None) == A.TLB_EUNSUPPORTED
    assert lib.tlb_rmsnorm_backward(C.c_void_p(16), C.c_void_p(16), C.c_void_p(32), C.c_void_p(32),
                                    1, 4, 1e-6, 1, None) == A.TLB_EINVAL                # alias + accumulate
    bad = A.LayerCfg(64, 256, 4, 3, 16, 4, 8.0, 1e4, 1e-6, 0.25, 0, 0, 0)         # 4 heads, 3 kv heads
    assert lib.tlb_workspace_bytes(C.byref(bad), 4, 4) > 0
    assert lib.tlb_layer_backward(C.byref(bad), 4, 4, None, None, None, None, None, None, None, None, 0,
                                  None) == A.TLB_EINVAL
    assert b"n_kv_heads" in lib.tlb_last_error()
    adam = A.AdamwCfg(1e-4, 0.9, 0.999, 1e-8, 0.0, 16.0, 0)
    assert lib.tlb_adamw(C.c_void_p(16), C.c_void_p(16), C.c_void_p(16), C.c_void_p(16), 4, C.byref(adam),
                         1.0, None, None) == A.TLB_EINVAL                               # step 0


def test_struct_layouts_match_the_header(tmp_path):
    """The binding passes these structs by pointer and, to tlb_stack_backward, as arrays:
    their sizes and field offsets must be the C compiler's."""
    import shutil
    import subprocess
    from transformer_layer_backward_gb300 import _abi as A
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    pairs = [("tlb_layer_cfg", A.LayerCfg), ("tlb_weight", A.Weight), ("tlb_layer_weights", A.LayerWeights),
             ("tlb_layer_acts", A.LayerActs), ("tlb_lora", A.Lora), ("tlb_adamw_cfg", A.AdamwCfg)]
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "tlb.h"', "int main(void) {"]
    for cname, py in pairs:
        lines.append('printf("%%s %%zu\\n", "%s", sizeof(%s));' % (cname, cname))
        for f in py._fields_:
            lines.append('printf("%%s.%%s %%zu\\n", "%s", "%s", offsetof(%s, %s));' % (cname, f[0], cname, f[0]))
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run([gcc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = dict(l.rsplit(" ", 1) for l in subprocess.run([str(exe)], check=True, capture_output=True,
                                                          text=True).stdout.split("\n") if l)
    for cname, py in pairs:
        assert int(got[cname]) == C.sizeof(py), cname
        for f in py._fields_:
            assert int(got["%s.%s" % (cname, f[0])]) == getattr(py, f[0]).offset, (cname, f[0])


def test_stack_host_side_errors(lib):
    from transformer_layer_backward_gb300 import _abi as A
    cfg = A.LayerCfg(64, 256, 4, 2, 16, 4, 8.0, 1e4, 1e-6, 0.25, 0, 0, 0)
    adam = A.AdamwCfg(1e-4, 0.9, 0.999, 1e-8, 0.0, 16.0, 1)
    assert lib.tlb_stack_workspace_bytes(C.byref(cfg), 1, 8) >= 2 * lib.tlb_workspace_bytes(C.byref(cfg), 1, 8)
    assert lib.tlb_stack_backward(C.byref(cfg), 1, 8, -1, None, None, None, None, C.byref(adam), None, None,
                                  None, 0, None) == A.TLB_EINVAL
    assert lib.tlb_stack_backward(C.byref(cfg), 1, 8, 0, None, None, None, None, C.byref(adam), None, None,
                                  None, 0, None) == A.TLB_OK                          # no layers: no-op
    assert lib.tlb_stack_backward(C.byref(cfg), 1, 8, 2, None, None, None, None, C.byref(adam), None, None,
                                  None, 0, None) == A.TLB_EINVAL
    assert b"NULL layer array" in lib.tlb_last_error()


def test_stack_workspace_sets(lib):
    """Single-token stacks rotate four layer workspaces; longer layers share one."""
    from transformer_layer_backward_gb300 import _abi as A
    cfg = A.LayerCfg(256, 512, 8, 2, 64, 4, 8.0, 1e4, 1e-6, 0.125, 1, 1, 4 | 8 | 32)
    one = lambda S, L: (lib.tlb_workspace_bytes(C.byref(cfg), S, L) + 255) // 256 * 256
    assert lib.tlb_stack_workspace_bytes(C.byref(cfg), 1, 40) == 4 * one(1, 40)
    assert lib.tlb_stack_workspace_bytes(C.byref(cfg), 64, 96) == one(64, 96)


def test_workspace_grows_with_rows(lib):
    from transformer_layer_backward_gb300 import _abi as A
    cfg = A.LayerCfg(2560, 9728, 32, 8, 128, 16, 32.0, 1e4, 1e-6, 128 ** -0.5, 1, 1, 4 | 8 | 32)
    sizes = [lib.tlb_workspace_bytes(C.byref(cfg), s, s) for s in (1, 64, 512)]
    assert sizes[0] < sizes[1] < sizes[2]
    assert all(s % 256 == 0 for s in sizes)


def test_qk_norm_needs_its_inputs(lib):
    """TLB_QK_NORM without q_raw or gamma_q is refused before any device work; with them
    the call gets past the input checks to the workspace check."""
    from transformer_layer_backward_gb300 import _abi as A
    cfg = A.LayerCfg(64, 256, 4, 2, 16, 4, 8.0, 1e4, 1e-6, 0.25, 0, 0, A.QK_NORM | A.CAUSAL)
    adam = A.AdamwCfg(1e-4, 0.9, 0.999, 1e-8, 0.0, 16.0, 1)
    fake = C.c_void_p(256)                       # never dereferenced: the checks fail first
    w = A.LayerWeights(A.Weight(fake, 1.0), A.Weight(fake, 1.0), A.Weight(fake, 1.0), A.Weight(fake, 1.0),
                       None, None, None, None)
    acts = A.LayerActs(fake, fake, fake, None, None, None, None, fake, fake, 16, 32, fake, fake, fake, None)
    lq = A.Lora(fake, fake, fake, fake, fake, fake, None, None)
    args = (C.byref(cfg), 8, 8, C.byref(w), C.byref(acts), C.byref(lq), C.byref(lq), C.byref(adam), fake, fake,
            None, 0, None)
    assert lib.tlb_layer_backward(*args) == A.TLB_EINVAL
    assert b"QK_NORM needs q_raw and gamma_q" in lib.tlb_last_error()
    w.gamma_q = fake
    acts.q_raw = fake
    assert lib.tlb_layer_backward(*args) == A.TLB_EINVAL
    assert b"workspace" in lib.tlb_last_error()


def test_linear_backward_host_side_errors(lib):
    """tlb_linear_backward refuses unknown weight types, packed-ternary rows that are not
    whole bytes, negative sizes, NULL operands and a short workspace before any device work."""
    from transformer_layer_backward_gb300 import _abi as A
    fake = C.c_void_p(256)                       # never dereferenced: the checks fail first

    def call(wtype, S, out_dim, in_dim, W=fake, dY=fake, dX=fake, ws=None, ws_bytes=0):
        return lib.tlb_linear_backward(wtype, W, 1.0, dY, S, out_dim, in_dim, dX, 0, ws, ws_bytes, None)

    assert call(9, 4, 8, 8) == A.TLB_EINVAL
    assert b"unknown weight type" in lib.tlb_last_error()
    assert call(A.W_TERNARY_2B, 4, 6, 8) == A.TLB_EINVAL                   # rows of 6 two-bit codes
    assert b"out_dim % 4" in lib.tlb_last_error()
    assert call(A.W_F32, -1, 8, 8) == A.TLB_EINVAL
    assert b"negative" in lib.tlb_last_error()
    assert call(A.W_F32, 0, 8, 8, W=None, dY=None, dX=None) == A.TLB_OK    # no rows: a no-op
    assert call(A.W_F32, 4, 8, 8, W=None) == A.TLB_EINVAL
    assert b"null pointer" in lib.tlb_last_error()
    assert lib.tlb_linear_workspace_bytes(A.W_F32, -1, 8, 8) == 0
    need = lib.tlb_linear_workspace_bytes(A.W_BF16, 256, 512, 256)
    assert need > lib.tlb_linear_workspace_bytes(A.W_F32, 256, 512, 256)   # bf16 copy of dY and partials
    assert call(A.W_BF16, 256, 512, 256, ws=fake, ws_bytes=need - 1) == A.TLB_EINVAL
    assert b"workspace" in lib.tlb_last_error()


def test_lora_grad_adamw_host_side_errors(lib):
    from transformer_layer_backward_gb300 import _abi as A
    fake = C.c_void_p(256)
    good = A.Lora(fake, fake, fake, fake, fake, fake, None, None)
    adam = A.AdamwCfg(1e-4, 0.9, 0.999, 1e-8, 0.0, 16.0, 1)

    def call(S, out_dim, in_dim, rank, lora=good, G=fake):
        return lib.tlb_lora_grad_adamw(S, out_dim, in_dim, rank, 2.0 * rank, G, fake, fake, C.byref(lora),
                                       C.byref(adam), None, None, 0, None)

    assert call(8, 0, 16, 4) == A.TLB_EINVAL
    assert b"bad sizes" in lib.tlb_last_error()
    for rank in (0, 65):
        assert call(8, 16, 16, rank) == A.TLB_EINVAL
        assert b"rank" in lib.tlb_last_error()
    assert call(8, 16, 16, 4, lora=A.Lora(fake, None, fake, fake, fake, fake, None, None)) == A.TLB_EINVAL
    assert b"NULL pointer" in lib.tlb_last_error()
    assert call(8, 16, 16, 4, G=None) == A.TLB_EINVAL
    assert b"NULL input" in lib.tlb_last_error()
    assert call(0, 16, 16, 4, G=None) == A.TLB_OK          # no tokens: no gradient and no step
    assert call(8, 16, 16, 4) == A.TLB_EINVAL
    assert b"workspace" in lib.tlb_last_error()


def test_attention_inputs_of_each_mode_are_checked(lib):
    """The exact input gradient, the recomputed attention and the cache bounds refuse
    missing inputs before any device work; with them the call reaches the workspace check."""
    from transformer_layer_backward_gb300 import _abi as A
    fake = C.c_void_p(256)
    adam = A.AdamwCfg(1e-4, 0.9, 0.999, 1e-8, 0.0, 16.0, 1)
    lq = A.Lora(fake, fake, fake, fake, fake, fake, None, None)

    def layer(flags, S=8, L=8, **fields):
        cfg = A.LayerCfg(64, 256, 4, 2, 16, 4, 8.0, 1e4, 1e-6, 0.25, 0, 0, A.CAUSAL | flags)
        w = A.LayerWeights(A.Weight(fake, 1.0), A.Weight(fake, 1.0), A.Weight(fake, 1.0), A.Weight(fake, 1.0))
        acts = A.LayerActs(fake, fake, fake, None, None, None, None, fake, fake, 16, 32, fake, fake, fake)
        for k, v in fields.items():
            setattr(w if hasattr(w, k) and k.startswith(("w_", "gamma")) else acts, k, v)
        return lib.tlb_layer_backward(C.byref(cfg), S, L, C.byref(w), C.byref(acts), C.byref(lq), C.byref(lq),
                                      C.byref(adam), fake, fake, None, 0, None)

    wqkv = dict(w_q=A.Weight(fake, 1.0), w_k=A.Weight(fake, 1.0), w_v=A.Weight(fake, 1.0))
    assert layer(A.EXACT_DIN) == A.TLB_EINVAL
    assert b"EXACT_DIN needs w_q, w_k and w_v" in lib.tlb_last_error()
    assert layer(A.EXACT_DIN, **wqkv) == A.TLB_EINVAL
    assert b"EXACT_DIN needs q" in lib.tlb_last_error()
    assert layer(A.EXACT_DIN, q=fake, **wqkv) == A.TLB_EINVAL
    assert b"workspace" in lib.tlb_last_error()
    assert layer(A.EXACT_DIN | A.PRE_NORM, q=fake, r1=fake, gamma_ffn=fake, **wqkv) == A.TLB_EINVAL
    assert b"EXACT_DIN with PRE_NORM needs x_in and gamma_attn" in lib.tlb_last_error()
    assert layer(A.EXACT_DIN | A.QK_NORM, q=fake, q_raw=fake, gamma_q=fake, **wqkv) == A.TLB_EINVAL
    assert b"EXACT_DIN with QK_NORM needs k_raw and gamma_k" in lib.tlb_last_error()

    assert layer(A.RECOMPUTE_P, attn=None) == A.TLB_EINVAL
    assert b"RECOMPUTE_P needs q and lse" in lib.tlb_last_error()
    assert layer(A.RECOMPUTE_P, attn=None, q=fake, lse=fake) == A.TLB_EINVAL
    assert b"workspace" in lib.tlb_last_error()
    assert layer(0, attn=None) == A.TLB_EINVAL
    assert b"attn pointer is NULL" in lib.tlb_last_error()

    assert layer(0, S=9, L=8) == A.TLB_EINVAL
    assert b"need 0 <= S <= L" in lib.tlb_last_error()
    assert layer(0, S=1, L=1 << 24) == A.TLB_EUNSUPPORTED
    assert layer(0, kv_stride_pos=8) == A.TLB_EINVAL
    assert b"strides smaller than head_dim" in lib.tlb_last_error()


def test_no_host_fallback_on_the_product_path(monkeypatch):
    """The binding never computes on the host: CPU tensors are refused before any library
    call, and a missing library is an error, not a fallback."""
    import torch
    from transformer_layer_backward_gb300 import _abi, api
    x = torch.zeros(2, 4)
    with pytest.raises(ValueError, match="CUDA"):
        api.softmax_backward(x, x)
    monkeypatch.setattr(_abi, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        _abi.load(os.path.join(ROOT, "no_such_dir", "libtlb.so"))
