"""GPU parity of the standalone steps against the float64 oracle (element by element),
including empty, ragged (length not a multiple of 4, misaligned) and long rows."""
import numpy as np
import pytest

from oracle import ops
from synth import rng
from synth.inputs import pack_ternary2
from tests.helpers import BF16_REL_L2, check, host

pytestmark = pytest.mark.gpu


def normal(name, shape, std=1.0):
    n = int(np.prod(shape))
    return rng.normal(rng.stream_key(0, "steps", name, *shape), n, 0.0, std).reshape(shape).astype(np.float32)


def softmax_rows(name, shape):
    z = normal(name, shape).astype(np.float64)
    e = np.exp(z - z.max(-1, keepdims=True))
    return (e / e.sum(-1, keepdims=True)).astype(np.float32)


def dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("rows,length", [(0, 5), (3, 0), (4, 7), (5, 128), (9, 1000), (3, 1001),
                                         (32, 4096), (2, 32768), (3, 20000), (64, 20)])
def test_softmax_backward(lib, rows, length):
    import torch
    a = softmax_rows("attn", (rows, length)) if rows and length else np.zeros((rows, length), np.float32)
    g = normal("dattn", (rows, length))
    out = lib.softmax_backward(dev(a), dev(g))
    torch.cuda.synchronize()
    check("dS", host(out), ops.softmax_backward(a, g))
    if rows and length:
        assert np.max(np.abs(host(out).sum(-1))) < 1e-5          # rows sum to zero


def test_softmax_backward_misaligned_view(lib):
    import torch
    a = softmax_rows("attn_mis", (4, 65))
    g = normal("dattn_mis", (4, 65))
    big_a = torch.zeros(4 * 65 + 1, device="cuda")
    big_a[1:] = dev(a).reshape(-1)
    big_g = torch.zeros(4 * 65 + 1, device="cuda")
    big_g[1:] = dev(g).reshape(-1)
    out = lib.softmax_backward(big_a[1:].view(4, 65), big_g[1:].view(4, 65))
    check("dS misaligned", host(out), ops.softmax_backward(a, g))


@pytest.mark.parametrize("act", ["relu2_mul", "silu_mul", "silu_mul_cache"])
@pytest.mark.parametrize("n", [0, 1, 7, 1024, 100003])
def test_act_backward(lib, act, n):
    gate, up, dh = normal("gate", (n,)), normal("up", (n,)), normal("dh", (n,))
    sg = None
    kind = "silu_mul" if act.startswith("silu") else act
    if act == "silu_mul_cache":
        sg = (gate / (1.0 + np.exp(-gate.astype(np.float64)))).astype(np.float32)
    dg, du = lib.act_backward(kind, dev(gate), dev(up), dev(dh), None if sg is None else dev(sg))
    if kind == "relu2_mul":
        rg, ru = ops.relu2_mul_backward(gate, up, dh)
    else:
        rg, ru = ops.silu_mul_backward(gate, up, dh, sg)
    check("dGate", host(dg), rg)
    check("dUp", host(du), ru)


@pytest.mark.parametrize("rows,n", [(1, 2560), (33, 2560), (5, 6912), (3, 7), (2, 20000), (0, 16), (17, 96)])
@pytest.mark.parametrize("accumulate", [False, True])
def test_rmsnorm_backward(lib, rows, n, accumulate):
    x, dy = normal("x", (rows, n)), normal("dy", (rows, n))
    gamma = rng.uniform(rng.stream_key(0, "steps", "gamma", n), n, 0.5, 1.5).astype(np.float32)
    base = normal("base", (rows, n))
    out = dev(base.copy())
    lib.rmsnorm_backward(dev(x), dev(gamma), dev(dy), 1e-6, out=out, accumulate=accumulate)
    ref = ops.rmsnorm_backward(x, gamma, dy, 1e-6) + (base if accumulate else 0.0)
    check("dx", host(out), ref)


@pytest.mark.parametrize("rows,nh,hd,pos0", [(1, 20, 128, 1023), (33, 3, 16, 0), (65, 4, 6, 2000),
                                             (7, 32, 128, 2041), (0, 2, 8, 0), (100, 5, 8, 60000),
                                             (20000, 2, 128, 5), (9, 7, 64, 300), (3000, 24, 128, 7)])
def test_rope_backward(lib, rows, nh, hd, pos0):
    dy = normal("dq", (rows, nh, hd))
    ref = ops.rope_backward(dy, pos0 + np.arange(rows), 10000.0)
    out = lib.rope_backward(dev(dy), pos0, 10000.0)
    check("dQpre", host(out), ref)
    inplace = dev(dy)
    lib.rope_backward(inplace, pos0, 10000.0, out=inplace)
    check("dQpre in place", host(inplace), ref)


@pytest.mark.parametrize("n", [1, 5, 4096, 100001])
@pytest.mark.parametrize("step", [1, 7])
def test_adamw(lib, n, step):
    import torch
    p, g = normal("p", (n,), 0.02), normal("g", (n,))
    if step == 1:
        m = np.zeros(n, np.float32)
        v = np.zeros(n, np.float32)
    else:
        m = normal("m", (n,), 1e-2)
        v = rng.uniform(rng.stream_key(0, "steps", "v", n), n, 0, 1e-4).astype(np.float32)
    cfg = lib.adamw_cfg(1e-3, 0.9, 0.999, 1e-8, 0.01, step)
    tp, tm, tv = dev(p.copy()), dev(m.copy()), dev(v.copy())
    ss = torch.zeros(1, dtype=torch.float64, device="cuda")
    lib.adamw(tp, dev(g), tm, tv, cfg, lr_mult=16.0, sumsq=ss)
    rp, rm, rv = ops.adamw(p, g, m, v, 16e-3, 0.9, 0.999, 1e-8, 0.01, step)
    check("p", host(tp), rp)
    check("m", host(tm), rm)
    check("v", host(tv), rv)
    assert abs(float(ss.item()) - float(np.sum(g.astype(np.float64) ** 2))) <= 1e-5 * float(np.sum(g.astype(np.float64) ** 2))


@pytest.mark.parametrize("wtype", ["f32", "bf16", "ternary", "ternary2"])
@pytest.mark.parametrize("S,in_dim,out_dim", [(1, 640, 2560), (1, 37, 50), (3, 100, 64), (130, 96, 272),
                                              (1, 6912, 2560), (256, 768, 1024), (130, 272, 4096),
                                              (77, 640, 2560), (512, 2560, 9728), (512, 9728, 2560),
                                              (300, 600, 1024), (2048, 2560, 9728)])
@pytest.mark.parametrize("accumulate", [False, True])
def test_linear_backward(lib, wtype, S, in_dim, out_dim, accumulate):
    import torch
    shape = (in_dim, out_dim)
    if wtype == "ternary2" and out_dim % 4:
        pytest.skip("packed ternary rows hold whole bytes")
    if wtype in ("ternary", "ternary2"):
        W = rng.ternary(rng.stream_key(0, "steps", "wt", *shape), in_dim * out_dim).reshape(shape)
        Wt = torch.from_numpy(pack_ternary2(W) if wtype == "ternary2" else W).cuda()
    else:
        W = normal("w", shape, 0.05)
        if wtype == "bf16":
            W = rng.round_to_bf16(W)
            Wt = torch.from_numpy(W).cuda().to(torch.bfloat16)
        else:
            Wt = torch.from_numpy(W).cuda()
    dY = normal("dy_lin", (S, out_dim))
    base = normal("base_lin", (S, in_dim))
    out = dev(base.copy())
    lib.linear_backward(wtype, Wt, dev(dY), scale=1.25, out=out, accumulate=accumulate)
    ref = ops.linear_backward(dY, W, 1.25) + (base if accumulate else 0.0)
    if wtype == "bf16" and S > 1 and out_dim % 8 == 0 and in_dim % 4 == 0:
        # tcgen05 path: dY rounded to bf16, fp32 accumulation
        check("dX (tensor cores)", host(out), ref, BF16_REL_L2, None)
    else:
        check("dX", host(out), ref)
