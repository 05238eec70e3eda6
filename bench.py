"""Throughput of the LoRA layer backward on one GB300 (or N independent replicas).

Default workload (stack2048): the 36-layer stack backward at S = L = 2048 (dim 2560,
ffn 9728, 32/8 heads x 128, SwiGLU FFN, RoPE, residual, bf16 weights, LoRA rank 16 on Q
and V, AdamW + LoRA+).  One step = one tlb_stack_backward call: grad_hidden [2048, 2560]
through 36 distinct layers (weights, caches and adapters of their own, ~1 GB each), in
reverse, every layer's adapters updated.  tokens/s = 2048 / step time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl tlb|reference]
                  [--workload stack2048|seq2048|seq512|decode|sweep]

--impl reference times the float64 CPU oracle (the only other implementation of this
path available here) on the same workload: each step one 512-row causal slice of an
S = L = 2048 layer (the four slices in turn hold the layer's whole work), extrapolated
to the 36 layers of a step.  Under torchrun every rank runs its own replica (the path
has no exchange step); rank 0 prints one JSON line.

Other workloads: seq512 / seq2048 time one sequence layer backward of S tokens per
step; decode the single-token layer backward (dim 2560, ffn 6912, 20 / 5 heads of 128,
cache 1024, ternary int8 weights, ReLU^2 x Mul with sub-norms and pre-norm); sweep the
standalone fp32 kernels (softmax, RMSNorm, RoPE, gated activations, AdamW) over their
size ranges, per-case GB/s, the headline the lowest among the cases above 4 x L2.
The sequence inputs are drawn on the device with torch's seeded generator, with the
shapes and distributions of the parity inputs.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "LoRA layer-backward tokens/s"
UNIT = "tokens/s"


def parse(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None, help="timed steps (default: decode 20000, stack2048 30, others 200)")
    p.add_argument("--warmup", type=int, default=None, help="untimed steps (default: decode 2000, others 5)")
    p.add_argument("--impl", default="tlb", choices=["tlb", "reference"])
    p.add_argument("--layers", type=int, default=None,
                   help="distinct layers (weights, caches, adapters) cycled: decode 8, stack the depth, layers 2")
    p.add_argument("--e2e-steps", type=int, default=2000)
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--no-graph", action="store_true")
    p.add_argument("--stack-layers", type=int, default=36,
                   help="decode: also time the layer inside a stack of this many layers (0: skip)")
    p.add_argument("--cases", default=None,
                   help="sweep: run only the cases whose 'kernel shape' label matches this regex")
    p.add_argument("--workload", default="stack2048", choices=["decode", "seq512", "seq2048", "stack2048", "sweep", "tf32peak", "h2dpeak"])
    p.add_argument("--qk-norm", action="store_true",
                   help="layers with the per-head QK-norm on q (decode and sequence workloads)")
    p.add_argument("--recompute-p", action="store_true",
                   help="sequence workloads: attention weights recomputed from q, K and each row's logsumexp "
                        "(not read from the cached [nh, S, L] weights)")
    p.add_argument("--wtype", default="ternary", choices=["ternary", "ternary2"],
                   help="decode: int8 ternary weights, or the same values packed four 2-bit codes to a byte")
    p.add_argument("--exact-din", action="store_true",
                   help="sequence workloads: the exact layer-input gradient (through W_Q, W_K, W_V, the "
                        "LoRA A paths and the attention pre-norm) instead of the pages' truncated one")
    a = p.parse_args(argv)
    if a.steps is None:
        a.steps = {"decode": 20000, "stack2048": 30}.get(a.workload, 200)
    if a.warmup is None:
        a.warmup = 2000 if a.workload == "decode" else 5
    return a


def wbytes(cfg) -> float:
    """Bytes per stored weight: int8 ternary 1, packed ternary 1/4."""
    return 0.25 if cfg.wtype == "ternary2" else 1.0


def decode_bytes(cfg) -> int:
    """Algorithmic HBM bytes of one decode layer backward (each input read once)."""
    H, I, qd, kvd, r, L = cfg.dim, cfg.ffn_dim, cfg.q_dim, cfg.kv_dim, cfg.rank, cfg.cache_len
    weights = int((I * H + 2 * H * I + qd * H) * wbytes(cfg))       # ternary int8 or packed
    kv = 2 * kvd * L * 4
    attn = cfg.n_heads * L * 4
    lora = (2 * r * H + qd * r + kvd * r) * 24                      # p, m, v read + write
    vectors = (H * 2 + I * 3 + H + qd + I + H + qd + 2 * r + H) * 4  # dOut,x,gate,up,hid,r1,ctx,gammas,h,d_in
    return weights + kv + attn + lora + vectors


# The kernels of one decode layer backward (multi-kernel schedule, launch order) and the
# bytes each must move at least once (algorithmic traffic; int8 ternary weights).
def decode_kernel_bytes(cfg):
    H, I, qd, kvd, r, L, nh = cfg.dim, cfg.ffn_dim, cfg.q_dim, cfg.kv_dim, cfg.rank, cfg.cache_len, cfg.n_heads
    lora = (2 * r * H + qd * r + kvd * r) * 24 + 2 * H * 4 + 2 * r * 4
    wb = wbytes(cfg)
    return [
        ("dec_k1 dF = W_down dOut", int(I * H * wb) + (H + I + 2 * I) * 4),
        ("dec_k2 dN2 = W_gate dG + W_up dU", int(2 * H * I * wb) + (5 * I + 3 * H) * 4),
        ("dec_k3 dSub = W_O dR1", int(qd * H * wb) + (4 * H + qd + 2 * qd) * 4),
        ("dec_k4 attention over K, V", 2 * kvd * L * 4 + nh * L * 4 + 3 * qd * 4),
        ("dec_k6 dQpre, gh_q", 2 * qd * 4 * (L // 64) + qd * r * 4),
        ("dec_k7 LoRA grads + AdamW", lora),
    ]


def slowest_rank_ms(ms, dist, device="cuda"):
    """The job's time: the slowest rank's, the same on every rank (a max all-reduce)."""
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return None


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(index), "--query-gpu=" + self.Q,
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return None
        self.p.terminate()
        self.p.wait()
        rows = [l.split(", ") for l in open(self.f.name).read().strip().splitlines() if l.count(",") >= 8]
        os.unlink(self.f.name)
        if not rows:
            return None
        mhz = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def oracle_step_time(cfg, seconds):
    """Seconds per decode layer backward of the float64 oracle on the host cores."""
    from oracle import layer as OL
    from synth import layer_inputs
    d = layer_inputs(cfg, layer=0, seed=0)
    n, t0 = 0, time.perf_counter()
    while True:
        OL.layer_backward(cfg, d, d["dout"])
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds or n >= 1000:
            return el / n, n


def host_threads():
    try:
        from threadpoolctl import threadpool_info
        t = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if t:
            return max(t)
    except Exception:
        pass
    return os.cpu_count()


def run_reference(args, rank, world):
    if rank != 0:
        return
    if args.workload == "sweep":
        per = max(args.cpu_seconds / 8, 0.5)
        big = {}
        for kind, shape, bpe in sweep_cases():       # the largest case of each kernel
            big[kind] = (shape, bpe)
        res = {k: sweep_oracle_gbs(k, shp, bpe, per) for k, (shp, bpe) in big.items()}
        worst = min(res, key=lambda k: res[k][0])
        v = res[worst][0]
        line = {"impl": "reference", "metric": SWEEP_METRIC, "value": v, "unit": "GB/s", "n_gpus": world,
                "steps": len(res), "warmup": 0, "ms_per_step": per * 1e3, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": {"workload": "standalone kernel sweep sample: the float64 oracle on up to 2^22 "
                                       "elements of the largest case of each kernel",
                           "parallelism": "replicas"},
                "sweep": [{"kernel": k, "GB/s": r[0], "sample": r[1]} for k, r in res.items()],
                "cpu_baseline": {"value": v, "unit": "GB/s", "cores": host_threads(), "kind": "oracle",
                                 "sample": "%s: %s" % (worst, res[worst][1])},
                "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    if args.workload != "decode":
        # one step = one row slice of the full-size layer (the slices in turn cover the
        # layer's work), extrapolated to the step's depth
        cfg, depth = seq_config(args.workload)
        if args.qk_norm:
            cfg = cfg.with_(qk_norm=True)
        if args.exact_din:
            cfg = cfg.with_(exact_din=True)
        if args.recompute_p:
            cfg = cfg.with_(recompute_p=True)
        slices = seq_cpu_sample(cfg)
        for k in range(min(args.warmup, 1)):
            seq_cpu_time(slices[k])
        times = [seq_cpu_time(slices[k % SLICES]) for k in range(args.steps)]
        tok = cfg.seq_len // SLICES
        v = args.steps * tok / (sum(times) * depth)
        line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": sum(times) * depth / args.steps * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic (host generator)", "config": seq_workload_config(cfg, depth, world),
                "cpu_baseline": {"value": v, "unit": UNIT, "cores": host_threads(), "kind": "oracle",
                                 "sample": "each step: the float64 numpy oracle on one %d-row causal slice of an "
                                           "S = L = %d layer (slices 0..%d in turn, together the layer's whole "
                                           "work), x %d layers" % (tok, cfg.seq_len, SLICES - 1, depth)},
                "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    from synth import DECODE
    cfg = DECODE.with_(qk_norm=True) if args.qk_norm else DECODE
    if args.wtype == "ternary2":
        cfg = cfg.with_(name="decode_t2", wtype="ternary2")
    per = max(args.cpu_seconds / max(args.steps, 1), 0.0)
    times = []
    for _ in range(args.warmup if args.warmup < 3 else 1):
        oracle_step_time(cfg, 0.0)
    for _ in range(args.steps):
        t, _ = oracle_step_time(cfg, per)
        times.append(t)
    t = statistics.mean(times)
    v = 1.0 / t
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "decode layer backward: dim 2560, ffn 6912, 20/5 heads x 128, "
                                   "cache 1024, ternary, " + ("QK-norm on q, " if cfg.qk_norm else "") +
                                   "LoRA r16", "global_batch": 1, "seq_len": 1,
                       "parallelism": "replicas"},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": host_threads(), "kind": "oracle",
                             "sample": "one decode layer backward per step, float64 numpy oracle"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- sequence workloads

def seq_config(workload):
    from synth import SEQ512
    if workload == "seq512":
        return SEQ512, 1
    return SEQ512.with_(name=workload, seq_len=2048, cache_len=2048), (36 if workload == "stack2048" else 1)


def seq_kernel_flops(cfg, names):
    """Algorithmic flops of each kernel of one sequence layer, by launch order: the
    three tcgen05 GEMMs are W_down^T, [W_gate | W_up]^T and W_O^T; the attention counts
    the visible (query, key) pairs of the contractions the method needs (dAttn and dQ in
    the dQ kernel, dV in the dV kernel), not the extra P K product of its U - D W split;
    'tf32' marks the attention contractions."""
    S, L, H, I, qd = cfg.seq_len, cfg.cache_len, cfg.dim, cfg.ffn_dim, cfg.q_dim
    pairs = S * (L - S) + S * (S + 1) // 2
    kvd = cfg.kv_dim
    gemm = [2 * S * I * H, 2 * S * H * 2 * I, 2 * S * qd * H, 2 * S * H * (qd + 2 * kvd)]
    out, gi = [], 0
    for nm in names:
        if nm == "tcgen05 gemm":
            out.append((gemm[gi] if gi < 4 else 0, "bf16"))
            gi += 1
        elif nm == "attn_tc_dq":            # dAttn = dCtx V^T and dQ = dS K
            out.append((2 * 2 * pairs * cfg.head_dim * cfg.n_heads, "tf32"))
        elif nm == "attn_tc_dv":
            out.append((2 * pairs * cfg.head_dim * cfg.n_heads, "tf32"))
        elif nm == "attn_dq_tiled":       # dAttn, dQ (+ the recomputed scores)
            out.append(((3 if cfg.recompute_p else 2) * 2 * pairs * cfg.head_dim * cfg.n_heads, "fp32"))
        elif nm == "attn_dv_tiled":
            out.append(((2 if cfg.recompute_p else 1) * 2 * pairs * cfg.head_dim * cfg.n_heads, "fp32"))
        elif nm in ("attn_dk_tiled", "attn_dk_tc"):     # dAttn recomputed and dK = dS^T q
            out.append((2 * 2 * pairs * cfg.head_dim * cfg.n_heads, "fp32" if nm == "attn_dk_tiled" else "tf32"))
        else:
            out.append((0, None))
    return out


def seq_kernel_bytes(cfg, names):
    """Algorithmic HBM bytes of the tensor-core attention kernels of one sequence layer,
    by launch order (0 for the other kernels): what each must read and write once.  dQ
    reads the weights of the visible (query, key) pairs, dCtx, K and V and writes dQpre;
    dV reads the weights and dCtx and writes dV.  Both are bound by these bytes rather than
    by their tf32 flops."""
    S, L, qd, kvd = cfg.seq_len, cfg.cache_len, cfg.q_dim, cfg.kv_dim
    pairs = S * (L - S) + S * (S + 1) // 2
    P = 4 * cfg.n_heads * pairs
    out = []
    for nm in names:
        if nm == "attn_tc_dq":
            out.append(P + 4 * (S * qd + 2 * L * kvd + S * qd))
        elif nm == "attn_tc_dv":
            out.append(P + 4 * (S * qd + S * kvd))
        else:
            out.append(0)
    return out


def kernel_entries(names, ktime_ms, flops, nbytes, peak_of, hbm_gbs):
    """The bench line's per-kernel entries: live time, and where known the algorithmic
    flops against the peak of the operand type and the algorithmic bytes against HBM."""
    out = []
    for nm, t, (f, kind), b in zip(names, ktime_ms, flops, nbytes):
        e = {"kernel": nm, "us": t * 1e3}
        if f:
            e.update({"flop": f, "TFLOP/s": f / (t / 1e3) / 1e12, "operands": kind,
                      "frac": f / (t / 1e3) / 1e12 / peak_of[kind]})
        if b:
            e.update({"bytes": b, "GB/s": b / (t / 1e3) / 1e9, "hbm_frac": b / (t / 1e3) / 1e9 / hbm_gbs})
        out.append(e)
    return out


def seq_workload_config(cfg, depth, world):
    """The config dict of a sequence workload: the same for both arms."""
    name = ("%d-layer stack backward, S = L = %d" % (depth, cfg.seq_len) if depth > 1 else
            "sequence layer backward, S = L = %d" % cfg.seq_len)
    return {"workload": name + ": dim 2560, ffn 9728, 32/8 heads x 128, SwiGLU, RoPE, residual, " +
                        ("QK-norm on q, " if cfg.qk_norm else "") +
                        ("exact layer-input gradient, " if cfg.exact_din else "") +
                        ("attention recomputed from q, K and the logsumexp, " if cfg.recompute_p else "") +
                        "bf16 weights, LoRA r16 Q/V, AdamW+LoRA+",
            "global_batch": world, "seq_len": cfg.seq_len, "layers_per_step": depth,
            "parallelism": "replicas" if world > 1 else "single",
            "l2": "inputs > L2 (each layer: weights 170 MB, attn %.0f MB)" % (cfg.n_heads * cfg.seq_len * cfg.cache_len * 4 / 1e6)}


def tf32_peak(bf16_sustained):
    """(TF/s, source) of the dense tf32 peak: the committed measurement of a cuBLAS tf32
    GEMM (the method of the bf16 figures), else the bf16 figure x the nominal 1.1/2.25."""
    prof = os.path.join(ROOT, "profiles", "tf32_peak.json")
    if os.path.exists(prof):
        m = json.load(open(prof))
        return m["tf32_tflops_sustained"], "profiles/tf32_peak.json tf32_tflops_sustained (of measured)"
    return bf16_sustained * 1.1 / 2.25, "bf16 sustained x nominal 1.1/2.25 (derived)"


def seq_main(args, rank, world, local, dist):
    import torch
    import transformer_layer_backward_gb300 as tlb
    from synth.device import device_layer

    torch.cuda.set_device(local)
    tlb.load()
    cfg, depth = seq_config(args.workload)
    if args.qk_norm:
        cfg = cfg.with_(qk_norm=True)
    if args.exact_din:
        cfg = cfg.with_(exact_din=True)
    if args.recompute_p:
        cfg = cfg.with_(recompute_p=True)
    S, L = cfg.seq_len, cfg.cache_len
    NL = args.layers or (depth if depth > 1 else 2)     # distinct layers (weights, caches, adapters)
    c = tlb.layer_cfg_of(cfg)
    adam = tlb.adamw_cfg_of(cfg)
    layers = []
    for l in range(NL):
        t = device_layer(cfg, l, seed=rank)
        layers.append(dict(t=t, w=tlb.layer_weights(c, t), a=tlb.layer_acts(c, t, cfg.kv_layout, L),
                           lq=tlb.lora(t, "q"), lv=tlb.lora(t, "v")))
    ws = tlb.workspace(c, S, L)
    dh = torch.empty(S, cfg.dim, device="cuda")
    ss = torch.zeros(2, dtype=torch.float64, device="cuda")
    stream = torch.cuda.current_stream()

    def layer_call(j):
        ly = layers[j % NL]
        tlb.layer_backward(c, S, L, ly["w"], ly["a"], ly["lq"], ly["lv"], adam, dh, ss, ws)

    if depth > 1:
        # the stack entry point; layer l of the stack is distinct layer l % NL
        sws = tlb.stack_workspace(c, S, L)
        sW, sA, sQ, sV = ([layers[l % NL][k] for l in range(depth)] for k in ("w", "a", "lq", "lv"))
    ng = 1 if depth > 1 else NL             # graphs: one per distinct step

    def step(i):
        dh.copy_(layers[(i * depth + depth - 1) % NL]["t"]["dout"])
        if depth > 1:
            tlb.stack_backward(c, S, L, sW, sA, sQ, sV, adam, dh, ss, sws)
        else:
            layer_call(i)

    graphs = None
    if not args.no_graph:
        for i in range(ng):
            step(i)
        torch.cuda.synchronize()
        graphs = []
        for i in range(ng):
            gph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gph):
                step(i)
            graphs.append(gph)
        torch.cuda.synchronize()

    def run(i):
        if graphs is not None:
            graphs[i % ng].replay()
        else:
            step(i)

    n0 = tlb.launch_count()
    step(0)
    launches_per_step = tlb.launch_count() - n0
    for i in range(max(args.warmup, 3)):
        run(i)
    tlb.workspace_status(sws if depth > 1 else ws)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = Clocks(local)
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        run(i)
    e1.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    tlb.workspace_status(sws if depth > 1 else ws)
    ms_max = slowest_rank_ms(ms, dist)
    value = args.steps * S * world / (ms_max / 1e3)

    # per-kernel times of one layer, live, inside a CUDA graph of nk layer calls; the
    # library records an event before the first and after every kernel of each call
    nk, ne = 8, 64
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(ne)] for _ in range(nk)]
    for row in evs:
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    keep = []
    pg = torch.cuda.CUDAGraph()
    with torch.cuda.graph(pg):
        for i in range(nk):
            dh.copy_(layers[i % NL]["t"]["dout"])
            keep.append(tlb.profile_events(evs[i]))
            layer_call(i)
        lib = tlb._abi.load()
        names = []
        while True:
            nm = lib.tlb_profile_kernel_name(len(names))
            if nm is None:
                break
            names.append(nm.decode())
        tlb.profile_events(None)
    pg.replay()
    torch.cuda.synchronize()
    nkern = min(len(names), ne - 1)
    ktime = [sum(evs[i][k].elapsed_time(evs[i][k + 1]) for i in range(nk)) / nk for k in range(nkern)]
    del keep
    fl = seq_kernel_flops(cfg, names[:nkern])
    pk = peaks()
    bf16_peak = pk["bf16_tflops_sustained"] if pk else 1700.0
    tf32, tf32_src = tf32_peak(bf16_peak)
    # CUDA-core fp32 kernels: FMA peak from the unit counts (128 fp32 lanes per SM, 2 flops
    # per FMA) at the maximum SM clock
    sms = torch.cuda.get_device_properties(local).multi_processor_count
    fp32_peak = sms * 128 * 2 * (pk["sm_max_mhz"] if pk else 2070.0) * 1e6 / 1e12
    peak_of = {"bf16": bf16_peak, "tf32": tf32, "fp32": fp32_peak}
    per_kernel = kernel_entries(names, ktime, fl, seq_kernel_bytes(cfg, names[:nkern]), peak_of,
                                pk["hbm_gbs"] if pk else 6800.0)
    dom = max((k for k in range(nkern) if fl[k][0]), key=lambda k: ktime[k])
    achieved = fl[dom][0] / (ktime[dom] / 1e3) / 1e12
    peak = peak_of[fl[dom][1]]
    # DRAM bytes of the dominant kernel from the committed ncu capture of the S = 2048 layer
    # (per launch; the stack runs the same launches per layer)
    traffic = None
    prof = os.path.join(ROOT, "profiles", "seq2048_dram_bytes.json")
    if S == 2048 and os.path.exists(prof):
        key = names[dom] if names[dom] != "tcgen05 gemm" else "tcgen05 gemm #%d" % (names[:dom + 1].count("tcgen05 gemm"))
        traffic = json.load(open(prof)).get(key)
    layer_flop = seq_layer_flops(cfg)
    step_s = ms_max / args.steps / 1e3
    step_roofline = {"bound": "tensor", "flop_per_step": layer_flop * depth,
                     "achieved": layer_flop * depth / step_s / 1e12, "peak": bf16_peak, "unit": "TFLOP/s",
                     "frac": layer_flop * depth / step_s / 1e12 / bf16_peak,
                     "note": "all algorithmic flops of a step (weight products bf16, attention tf32, "
                             "LoRA fp32) against the sustained bf16 peak"}

    # end to end through the public API: every layer's activations and caches copied from
    # pinned host memory on a copy stream (the next layer's copy overlapping this layer's
    # kernels), one tlb_layer_backward call per layer from the top of the stack down, and
    # d_in and the gradient sums read back at the end of each step
    acts = ("x", "gate", "up", "silu_gate", "k", "v", "lora_q_h", "lora_v_h") + \
        (("lse", "q") if cfg.recompute_p else ("attn",)) + (("q_raw",) if cfg.qk_norm else ()) + \
        (("q",) if cfg.exact_din and not cfg.recompute_p else ()) + \
        (("k_raw",) if cfg.exact_din and cfg.qk_norm else ())
    NP = min(NL, 2)
    pinned = [{k: layers[l]["t"][k].cpu().pin_memory() for k in acts} for l in range(NP)]
    dout_h = layers[0]["t"]["dout"].cpu().pin_memory()
    h2d = sum(pinned[0][k].numel() * 4 for k in acts) * depth + dout_h.numel() * 4
    res_h = torch.empty(S, cfg.dim, pin_memory=True)
    ss_h = torch.empty(2, dtype=torch.float64, pin_memory=True)
    d2h = res_h.numel() * 4 + 16
    n_e2e = max(2, min(args.steps, 5 if depth > 1 else 20))
    cs = torch.cuda.Stream()
    copied = [torch.cuda.Event() for _ in range(NL)]
    used = [torch.cuda.Event() for _ in range(NL)]
    for ev in used:
        ev.record(stream)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(n_e2e):
        for j in reversed(range(depth)):
            li = (i * depth + j) % NL
            ly = layers[li]
            with torch.cuda.stream(cs):
                cs.wait_event(used[li])                  # the previous user of these buffers is done
                for k in acts:
                    ly["t"][k].copy_(pinned[li % NP][k], non_blocking=True)
                copied[li].record(cs)
            stream.wait_event(copied[li])
            if j == depth - 1:
                dh.copy_(dout_h, non_blocking=True)
            tlb.layer_backward(c, S, L, ly["w"], ly["a"], ly["lq"], ly["lv"], adam, dh, ss, ws)
            used[li].record(stream)
        res_h.copy_(dh, non_blocking=True)
        ss_h.copy_(ss, non_blocking=True)
    torch.cuda.synchronize()
    e2e_s = time.perf_counter() - t0
    e2e = {"value": n_e2e * S * world / e2e_s, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "steps": n_e2e, "h2d_gbs": h2d * n_e2e / e2e_s / 1e9,
           "note": "copy-bound: the host link moves about 210 GB/s host to device on this machine "
                   "(bench.py --workload h2dpeak, profiles/h2d_link.md)"}

    cpu = None
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        cpu = seq_cpu_baseline(cfg, depth)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (device generator)",
                "config": seq_workload_config(cfg, depth, world),
                "harness": {"layers_distinct": NL, "cuda_graph": graphs is not None,
                            "step": ("one tlb_stack_backward call over %d layers" % depth) if depth > 1 else
                                    "one tlb_layer_backward call"},
                "layer_tokens_per_s": value * depth,
                "roofline": {"bound": "alu" if fl[dom][1] == "fp32" else "tensor", "kernel": names[dom],
                             "achieved": achieved, "peak": peak,
                             "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                             "algorithmic_flop": fl[dom][0],
                             "peak_source": {"bf16": ("MEASURED_PEAKS.json bf16_tflops_sustained (of measured)" if pk
                                                      else "fallback"),
                                             "tf32": tf32_src,
                                             "fp32": "SMs x 128 fp32 lanes x 2 flops x max SM clock (derived)"}[
                                                 fl[dom][1]]},
                "step_roofline": step_roofline,
                "per_kernel": per_kernel, "per_kernel_timing": "graph",
                "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches_per_step * args.steps, "clocks": clk}
        print(json.dumps(line), flush=True)


def seq_layer_flops(cfg):
    """Algorithmic flops of one sequence layer backward: the three weight products, the
    attention's dAttn, dQ and dV contractions over the visible (query, key) pairs, and the
    LoRA products (dB, gh, dA of both adapters)."""
    S, L, H, I, qd, kvd, r = cfg.seq_len, cfg.cache_len, cfg.dim, cfg.ffn_dim, cfg.q_dim, cfg.kv_dim, cfg.rank
    pairs = S * (L - S) + S * (S + 1) // 2
    gemm = 2 * S * I * H + 2 * S * H * 2 * I + 2 * S * qd * H
    attn = 3 * 2 * pairs * cfg.head_dim * cfg.n_heads
    lora = sum(2 * 2 * S * od * r for od in (qd, kvd)) + 2 * 2 * S * r * H   # dB, gh per adapter; dA
    if cfg.exact_din:       # dK = dS^T q, the [dQpre | dK | dV] W^T product, the LoRA A paths
        gemm += 2 * S * H * (qd + 2 * kvd)
        attn += 2 * pairs * cfg.head_dim * cfg.n_heads
        lora += 2 * 2 * S * r * H
    return gemm + attn + lora


SLICES = 4


def seq_cpu_sample(cfg, seed=0):
    """The host problem of one S = L layer and its SLICES row slices (S / SLICES rows each
    over the keys they may see): together the slices hold exactly the layer's work."""
    from synth import layer_inputs_sample, row_slice
    d = layer_inputs_sample(cfg, seed)
    n = cfg.seq_len // SLICES
    return [row_slice(cfg, d, k * n, (k + 1) * n) for k in range(SLICES)]


def seq_cpu_time(sl):
    """Seconds of one float64 oracle layer backward of a slice."""
    from oracle import layer as OL
    sub, d = sl
    t0 = time.perf_counter()
    OL.layer_backward(sub, d, d["dout"])
    return time.perf_counter() - t0


def seq_cpu_baseline(cfg, depth):
    """The float64 oracle on every row slice of one full-size layer (its whole work),
    extrapolated to the depth of the step, tokens/s."""
    slices = seq_cpu_sample(cfg)
    t = sum(seq_cpu_time(sl) for sl in slices)
    return {"value": cfg.seq_len / (t * depth), "unit": UNIT, "cores": host_threads(), "kind": "oracle",
            "sample": "the float64 numpy oracle on one S = L = %d layer, run as its %d causal row slices of "
                      "%d rows (%.1f s), x %d layers" % (cfg.seq_len, SLICES, cfg.seq_len // SLICES, t, depth)}


# ---------------------------------------------------------------- bandwidth sweep

SWEEP_METRIC = "standalone-kernel HBM bandwidth (lowest over the kernels)"


def sweep_cases():
    """The standalone fp32 kernels over the stated size ranges: (kernel, shape, bytes per
    element that must cross HBM once).  Softmax rows [32, len] as stated plus [rows, len]
    with rows * len = 2^27 (1.6 GB, far above L2); RMSNorm rows of 2560; RoPE [rows, 32,
    128]; gated activations 2^16 .. 2^28 elements; AdamW 2^12 .. 2^26 parameters."""
    c = []
    for n in (128, 512, 2048, 8192, 32768):
        c.append(("softmax_backward", (32, n), 12))
        c.append(("softmax_backward", (2 ** 27 // n, n), 12))
    for rows in (1, 16, 256, 4096, 65536):
        c.append(("rmsnorm_backward", (rows, 2560), 12))
    c.append(("rmsnorm_backward +=", (65536, 2560), 16))
    for rows in (1, 16, 256, 4096, 65536):
        c.append(("rope_backward", (rows, 32, 128), 8))
    for e in (16, 20, 24, 28):
        c.append(("act_backward relu2_mul", (2 ** e,), 20))
        c.append(("act_backward silu_mul cached", (2 ** e,), 24))
    c.append(("act_backward silu_mul", (2 ** 24,), 20))
    c.append(("act_backward silu_mul", (2 ** 28,), 20))
    for e in (12, 16, 20, 24, 26):
        c.append(("adamw", (2 ** e,), 28))
    return c


def sweep_setup(tlb, kind, shape, g):
    """Device inputs of one case (N(0, 1); softmax rows normalised; gammas U(0.5, 1.5))
    and the call that runs it through the binding."""
    import torch
    n = lambda: torch.randn(*shape, device="cuda", generator=g)
    if kind == "softmax_backward":
        a, d = torch.softmax(n(), dim=-1), n()
        o = torch.empty_like(a)
        return (lambda: tlb.softmax_backward(a, d, out=o)), {"attn": a, "dattn": d}, o
    if kind.startswith("rmsnorm_backward"):
        x, dy, o = n(), n(), n()
        gam = torch.rand(shape[-1], device="cuda", generator=g) + 0.5
        acc = kind.endswith("+=")
        return (lambda: tlb.rmsnorm_backward(x, gam, dy, out=o, accumulate=acc)), {"x": x, "dy": dy}, o
    if kind == "rope_backward":
        dy = n()
        o = torch.empty_like(dy)
        return (lambda: tlb.rope_backward(dy, 0, out=o)), {"dy": dy}, o
    if kind.startswith("act_backward"):
        gate, up, dh = n(), n(), n()
        dg, du = torch.empty_like(gate), torch.empty_like(gate)
        act = "relu2_mul" if "relu2" in kind else "silu_mul"
        sg = torch.nn.functional.silu(gate) if kind.endswith("cached") else None
        ins = {"gate": gate, "up": up, "dh": dh}
        if sg is not None:
            ins["silu_gate"] = sg
        return (lambda: tlb.act_backward(act, gate, up, dh, silu_gate=sg, dgate=dg, dup=du)), ins, dg
    if kind == "adamw":
        p, gr = n(), n()
        m, v = torch.zeros_like(p), torch.zeros_like(p)
        cfg = tlb.adamw_cfg(1e-4)
        return (lambda: tlb.adamw(p, gr, m, v, cfg)), {"g": gr}, p
    raise ValueError(kind)


def sweep_oracle_gbs(kind, shape, bpe, seconds):
    """Algorithmic GB/s of the float64 oracle on a sample of one case (at most 2^22
    elements of it), on the host cores."""
    from oracle import ops
    rng = np.random.default_rng(0)
    size = int(np.prod(shape))
    if len(shape) > 1:
        rows = max(1, min(shape[0], (2 ** 22) // (size // shape[0])))
        shp = (rows,) + tuple(shape[1:])
    else:
        shp = (min(size, 2 ** 22),)
    a = rng.standard_normal(shp)
    b = rng.standard_normal(shp)
    c = rng.standard_normal(shp)
    if kind == "softmax_backward":
        e = np.exp(a - a.max(axis=-1, keepdims=True))
        p = e / e.sum(axis=-1, keepdims=True)
        fn = lambda: ops.softmax_backward(p, b)
    elif kind.startswith("rmsnorm_backward"):
        gam = rng.uniform(0.5, 1.5, shp[-1])
        fn = lambda: ops.rmsnorm_backward(a, gam, b, 1e-6)
    elif kind == "rope_backward":
        pos = np.arange(shp[0])
        fn = lambda: ops.rope_backward(a, pos, 10000.0)
    elif kind.startswith("act_backward"):
        fn = (lambda: ops.relu2_mul_backward(a, b, c)) if "relu2" in kind else (lambda: ops.silu_mul_backward(a, b, c))
    else:
        z = np.zeros(shp)
        fn = lambda: ops.adamw(a.copy(), b, z.copy(), z.copy(), 1e-4, 0.9, 0.999, 1e-8, 0.01, 1)
    n, t0 = 0, time.perf_counter()
    while True:
        fn()
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds or n >= 1000:
            break
    return n * int(np.prod(shp)) * bpe / el / 1e9, "%d oracle calls on %s" % (n, "x".join(map(str, shp)))


def sweep_main(args, rank, world, local, dist):
    """Each case: W untimed launches, then K launches each timed alone with CUDA events on
    the launching stream (median); L2 is flushed (a 2 x L2 buffer cleared) before every
    timed launch whose working set is under 4 x L2.  Those small cases are reported but
    not counted in the lowest-bandwidth figure."""
    import torch
    import transformer_layer_backward_gb300 as tlb
    torch.cuda.set_device(local)
    tlb.load()
    props = torch.cuda.get_device_properties(local)
    l2 = getattr(props, "L2_cache_size", 0) or 126 * 2 ** 20
    flush = torch.empty(2 * l2 // 4, device="cuda")
    pk = peaks()
    hbm = pk["hbm_gbs"] if pk else 6800.0
    K, W = max(1, min(args.steps, 20)), max(3, min(args.warmup, 5))
    g = torch.Generator(device="cuda")
    g.manual_seed(1234 + rank)
    stream = torch.cuda.current_stream()
    rows, launches = [], 0
    if dist is not None:
        dist.barrier()
    clocks = Clocks(local)
    t_start = time.perf_counter()
    cases = [c for c in sweep_cases()
             if args.cases is None or re.search(args.cases, "%s %s" % (c[0], "x".join(map(str, c[1]))))]
    for kind, shape, bpe in cases:
        fn, ins, out = sweep_setup(tlb, kind, shape, g)
        elems = int(np.prod(shape))
        nbytes = elems * bpe
        small = nbytes < 4 * l2
        for _ in range(W):
            fn()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        c0 = tlb.launch_count()
        for e0, e1 in ev:
            if small:
                flush.zero_()
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize()
        launches += tlb.launch_count() - c0
        us = statistics.median(e0.elapsed_time(e1) for e0, e1 in ev) * 1e3
        gbs = nbytes / (us * 1e-6) / 1e9
        rows.append({"kernel": kind, "shape": list(shape), "bytes": nbytes, "us": us, "GB/s": gbs,
                     "frac": gbs / hbm, "set": "small (< 4 x L2, flushed)" if small else "hbm"})
        print("%-30s %-18s %10.1f MB %9.2f us %8.0f GB/s %5.1f %%%s" % (
            kind, "x".join(map(str, shape)), nbytes / 1e6, us, gbs, 100 * gbs / hbm,
            "  (small)" if small else ""), file=sys.stderr, flush=True)
        del fn, ins, out
        torch.cuda.empty_cache()
    wall = time.perf_counter() - t_start
    clk = clocks.stop()
    if dist is not None:
        dist.barrier()
    big = [r for r in rows if r["set"] == "hbm"] or rows
    worst = min(big, key=lambda r: r["GB/s"])
    value = worst["GB/s"]

    # end to end through the binding for the lowest case: its inputs from pinned host
    # memory, the call, its output read back
    fn, ins, out = sweep_setup(tlb, worst["kernel"], tuple(worst["shape"]), g)
    pinned = {k: v.cpu().pin_memory() for k, v in ins.items()}
    out_h = torch.empty(out.shape, pin_memory=True)
    h2d = sum(v.numel() * 4 for v in pinned.values())
    d2h = out_h.numel() * 4
    torch.cuda.synchronize()
    n_e2e = 3
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        for k, v in pinned.items():
            ins[k].copy_(v, non_blocking=True)
        fn()
        out_h.copy_(out, non_blocking=True)
    torch.cuda.synchronize()
    e2e_s = (time.perf_counter() - t0) / n_e2e
    e2e = {"value": worst["bytes"] / e2e_s / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "case": worst["kernel"]}
    del fn, ins, out

    # DRAM bytes per algorithmic byte of the kernel from the committed ncu capture (one
    # case of 0.3 - 2 GB per kernel; a streaming kernel's traffic grows in proportion to
    # its elements), times this case's algorithmic bytes
    traffic = None
    prof = os.path.join(ROOT, "profiles", "sweep_dram_bytes.json")
    if os.path.exists(prof):
        caps = json.load(open(prof))
        r = caps.get("%s %s" % (worst["kernel"], "x".join(map(str, worst["shape"]))))
        r = r or next((v for v in caps.values() if v["kernel"] == worst["kernel"]), None)
        traffic = None if r is None else r["traffic_per_algorithmic_byte"] * worst["bytes"]
    cpu = None
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        v, sample = sweep_oracle_gbs(worst["kernel"], tuple(worst["shape"]), worst["bytes"] // int(np.prod(worst["shape"])),
                                     min(args.cpu_seconds, 10.0))
        cpu = {"value": v, "unit": "GB/s", "cores": host_threads(), "kind": "oracle", "sample": sample}
    if rank == 0:
        line = {"metric": SWEEP_METRIC, "value": value * world, "unit": "GB/s", "n_gpus": world, "steps": K,
                "warmup": W, "ms_per_step": wall * 1e3 / len(rows), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic (device generator)",
                "config": {"workload": "standalone fp32 kernel sweep: softmax, RMSNorm, RoPE, gated "
                                       "activations, AdamW over the stated sizes",
                           "cases": len(rows), "l2": "flushed before each timed launch below 4 x L2",
                           "timing": "median of K launches, each timed alone"},
                "roofline": {"bound": "hbm", "kernel": "%s %s" % (worst["kernel"], "x".join(map(str, worst["shape"]))),
                             "achieved": value, "peak": hbm, "unit": "GB/s", "frac": value / hbm,
                             "traffic": traffic, "algorithmic_bytes": worst["bytes"],
                             "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)" if pk else "fallback"},
                "sweep": rows, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clk}
        print(json.dumps(line), flush=True)


def tf32peak_main(args, local):
    """Dense tf32 tensor-core peak, measured like the bf16 figures of the peaks file: a
    cuBLAS tf32 GEMM of 8192^3 (2 N^3 flops), best of 10 (burst) and back to back for
    4 s (sustained), CUDA events on the launching stream, clocks sampled meanwhile."""
    import torch
    torch.cuda.set_device(local)
    torch.backends.cuda.matmul.allow_tf32 = True
    n = 8192
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    a = torch.randn(n, n, device="cuda", generator=g)
    b = torch.randn(n, n, device="cuda", generator=g)
    c = torch.empty(n, n, device="cuda")
    for _ in range(5):
        torch.matmul(a, b, out=c)
    torch.cuda.synchronize()
    clocks = Clocks(local)
    best = 1e30
    for _ in range(10):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        torch.matmul(a, b, out=c)
        e1.record()
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1))
    reps, t0 = 0, time.perf_counter()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    while time.perf_counter() - t0 < 4.0:
        for _ in range(20):
            torch.matmul(a, b, out=c)
        reps += 20
        torch.cuda.synchronize()
    e1.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    flop = 2.0 * n ** 3
    print(json.dumps({"tf32_tflops": flop / (best / 1e3) / 1e12,
                      "tf32_tflops_sustained": flop * reps / (e0.elapsed_time(e1) / 1e3) / 1e12,
                      "how": "torch.matmul fp32 with allow_tf32 (cuBLAS) %d^3, 2 N^3 flops: best of 10 (burst) and "
                             "%d back to back (sustained), CUDA events" % (n, reps),
                      "gpu": torch.cuda.get_device_name(local), "torch": torch.__version__, "clocks": clk}), flush=True)


def h2dpeak_main(args, local):
    """Host -> device bandwidth of this machine's link, the ceiling of every e2e figure: 1 GiB
    from pinned host memory into device memory, split over 1, 2 and 4 copy streams, best of 4
    each, CUDA events around the copies."""
    import torch
    torch.cuda.set_device(local)
    n = 1 << 28                                   # floats: 1 GiB
    h = torch.empty(n, pin_memory=True)
    h.fill_(1.0)
    d = torch.empty(n, device="cuda")
    main = torch.cuda.current_stream()
    out = {}
    for ns in (1, 2, 4):
        streams = [torch.cuda.Stream() for _ in range(ns)]
        chunk = n // ns
        best = 1e30
        for _ in range(4):
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(main)
            for k, st in enumerate(streams):
                st.wait_event(e0)
                with torch.cuda.stream(st):
                    d[k * chunk:(k + 1) * chunk].copy_(h[k * chunk:(k + 1) * chunk], non_blocking=True)
            for st in streams:
                main.wait_stream(st)
            e1.record(main)
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        out["%d stream%s" % (ns, "" if ns == 1 else "s")] = n * 4 / (best / 1e3) / 1e9
    print(json.dumps({"h2d_gbs": max(out.values()), "by_streams": out,
                      "how": "torch copy_ of 1 GiB from pinned host memory, non_blocking, split over the copy "
                             "streams, best of 4, CUDA events", "gpu": torch.cuda.get_device_name(local),
                      "torch": torch.__version__}), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    import torch
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    if args.impl == "reference":
        run_reference(args, rank, world)
        if dist is not None:
            dist.destroy_process_group()
        return

    if args.workload == "h2dpeak":
        h2dpeak_main(args, local)
        return
    if args.workload == "tf32peak":
        tf32peak_main(args, local)
        return
    if args.workload == "sweep":
        sweep_main(args, rank, world, local, dist)
        if dist is not None:
            dist.destroy_process_group()
        return
    if args.workload != "decode":
        seq_main(args, rank, world, local, dist)
        if dist is not None:
            dist.destroy_process_group()
        return

    import transformer_layer_backward_gb300 as tlb
    from synth import DECODE, layer_inputs
    from synth.device import lora_dev, to_dev

    torch.cuda.set_device(local)
    tlb.load()
    cfg = DECODE.with_(qk_norm=True) if args.qk_norm else DECODE
    if args.wtype == "ternary2":
        cfg = cfg.with_(name="decode_t2", wtype="ternary2")
    NL = args.layers or 8
    c = tlb.layer_cfg_of(cfg)
    adam = tlb.adamw_cfg_of(cfg)
    layers, host_layers = [], []
    for l in range(NL):
        d = layer_inputs(cfg, layer=l, seed=0)
        t = to_dev(d, cfg.wtype)
        L = lora_dev(t)
        layers.append(dict(t=t, L=L, w=tlb.layer_weights(c, t),
                           a=tlb.layer_acts(c, t, cfg.kv_layout, cfg.cache_len),
                           lq=tlb.lora(L, "q"), lv=tlb.lora(L, "v")))
        host_layers.append(d)
    ws = tlb.workspace(c, 1, cfg.cache_len)
    dh = torch.empty(1, cfg.dim, device="cuda")
    ss = torch.zeros(2, dtype=torch.float64, device="cuda")
    stream = torch.cuda.current_stream()

    def step(i):
        ly = layers[i % NL]
        dh.copy_(ly["t"]["dout"])
        tlb.layer_backward(c, 1, cfg.cache_len, ly["w"], ly["a"], ly["lq"], ly["lv"], adam, dh, ss, ws)

    # CUDA graphs: one per layer, and one for a whole cycle of the NL layers (the same
    # calls back to back, so a graph boundary comes once per NL steps)
    graphs = cycle = None
    if not args.no_graph:
        for i in range(NL):
            step(i)
        torch.cuda.synchronize()
        graphs = []
        for i in range(NL):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step(i)
            graphs.append(g)
        cycle = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cycle):
            for i in range(NL):
                step(i)
        torch.cuda.synchronize()

    def run_steps(n):
        """n steps, starting at layer 0: whole cycles through the cycle graph, the rest
        one layer graph each."""
        if cycle is None:
            for i in range(n):
                step(i)
            return
        for _ in range(n // NL):
            cycle.replay()
        for i in range(n % NL):
            graphs[i].replay()

    launches_per_step = None
    n0 = tlb.launch_count()
    step(0)
    launches_per_step = tlb.launch_count() - n0
    run_steps(max(args.warmup, 3, NL))        # every graph replayed before the timed region
    tlb.workspace_status(ws)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = Clocks(local)
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run_steps(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()
    ms = e0.elapsed_time(e1)
    tlb.workspace_status(ws)
    ms_max = slowest_rank_ms(ms, dist)
    tokens = args.steps * world
    value = tokens / (ms_max / 1e3)

    # per-kernel times, live, on this stream: the library records an event before the first
    # and after every kernel of the step; the steps are captured in one CUDA graph like the
    # timed loop (stream launches would add host dispatch gaps to the intervals)
    kern = decode_kernel_bytes(cfg)
    nk = 64
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(kern) + 1)] for _ in range(nk)]
    for row in evs:
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()

    def profiled_steps():
        keep = []
        for i in range(nk):
            ly = layers[i % NL]
            dh.copy_(ly["t"]["dout"])
            keep.append(tlb.profile_events(evs[i]))
            tlb.layer_backward(c, 1, cfg.cache_len, ly["w"], ly["a"], ly["lq"], ly["lv"], adam, dh, ss, ws)
        tlb.profile_events(None)
        return keep

    try:
        pg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(pg):
            keep = profiled_steps()
        pg.replay()
        torch.cuda.synchronize()
        ktime = [sum(evs[i][k].elapsed_time(evs[i][k + 1]) for i in range(nk)) / nk for k in range(len(kern))]
        ktiming = "graph"
    except Exception:
        torch.cuda.synchronize()
        torch.cuda._sleep(200_000_000)      # queue the steps so they run back to back
        keep = profiled_steps()
        torch.cuda.synchronize()
        ktime = [sum(evs[i][k].elapsed_time(evs[i][k + 1]) for i in range(nk)) / nk for k in range(len(kern))]
        ktiming = "stream"
    del keep
    pk = peaks()
    hbm = pk["hbm_gbs"] if pk else 6800.0
    per_kernel = [{"kernel": n, "us": t * 1e3, "bytes": b, "GB/s": b / (t / 1e3) / 1e9}
                  for (n, b), t in zip(kern, ktime)]
    dom = max(range(len(kern)), key=lambda k: ktime[k])
    achieved = per_kernel[dom]["GB/s"]
    traffic = None
    prof = os.path.join(ROOT, "profiles", "decode_dram_bytes.json")
    if os.path.exists(prof) and cfg.wtype == "ternary":          # captured with int8 weights
        traffic = json.load(open(prof)).get(kern[dom][0].split()[0])

    # end to end through the public API: per-step activations from pinned host memory,
    # d_in and the gradient norm read back every step
    e2e = None
    if args.e2e_steps > 0:
        acts = ("x", "gate", "up", "hidden", "r1", "ctx", "k", "v", "attn", "lora_q_h", "lora_v_h", "dout")
        pinned = [{k: torch.from_numpy(np.ascontiguousarray(host_layers[l][k])).pin_memory() for k in acts}
                  for l in range(NL)]
        h2d = sum(pinned[0][k].numel() * 4 for k in acts)
        res_h = torch.empty(1, cfg.dim, pin_memory=True)
        ss_h = torch.empty(2, dtype=torch.float64, pin_memory=True)
        d2h = res_h.numel() * 4 + 16
        ne = min(args.e2e_steps, max(args.steps, 10))
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(ne):
            ly = layers[i % NL]
            for k in acts:
                ly["t"][k].copy_(pinned[i % NL][k], non_blocking=True)
            dh.copy_(ly["t"]["dout"])
            tlb.layer_backward(c, 1, cfg.cache_len, ly["w"], ly["a"], ly["lq"], ly["lv"], adam, dh, ss, ws)
            res_h.copy_(dh, non_blocking=True)
            ss_h.copy_(ss, non_blocking=True)
        torch.cuda.synchronize()
        e2e_s = time.perf_counter() - t0
        e2e = {"value": ne * world / e2e_s, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h}

    # the same layer inside a stack ([RS] backward_through_layers): args.stack_layers layer
    # calls (weights and caches cycling the NL sets, adapters of their own) through
    # tlb_stack_backward, which overlaps each layer's attention / LoRA half with the next
    # layer's GEMV chain; reported per layer
    stack = None
    if args.stack_layers > 0:
        NS = args.stack_layers
        sl = []
        for l in range(NS):
            src = layers[l % NL]
            L = lora_dev(src["L"])
            sl.append(dict(L=L, w=src["w"], a=src["a"], lq=tlb.lora(L, "q"), lv=tlb.lora(L, "v")))
        sws = tlb.stack_workspace(c, 1, cfg.cache_len)
        # d_in grows about 5e3 times per synthetic ternary layer, through two weight
        # products (W_down^T, then [W_gate | W_up]^T): the stack's layers take those three
        # BitLinear scales times 1 / sqrt(5e3), so that every layer of the stack runs on
        # finite values throughout the stack (checked below)
        damp = 1.0 / math.sqrt(5e3)
        sW = []
        for d in sl:
            w = type(d["w"]).from_buffer_copy(d["w"])          # the struct's bytes: same weights
            for k in ("w_down", "w_gate", "w_up"):
                wk = getattr(w, k)
                setattr(w, k, type(wk)(wk.w, wk.scale * damp))
            sW.append(w)
        sA = [d["a"] for d in sl]
        sQ, sV = [d["lq"] for d in sl], [d["lv"] for d in sl]
        sd = layers[0]["t"]["dout"].contiguous()

        def sstep():
            dh.copy_(sd)
            tlb.stack_backward(c, 1, cfg.cache_len, sW, sA, sQ, sV, adam, dh, ss, sws)

        sstep()                      # creates the library's second stream outside any capture
        torch.cuda.synchronize()
        sg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(sg):
            sstep()
        for _ in range(3):
            sg.replay()
        ns = max(3, min(200, args.steps // NS))
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(ns):
            sg.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        sms = e0.elapsed_time(e1) / ns
        tlb.workspace_status(sws)
        stack_finite = bool(torch.isfinite(dh).all().item())
        stack_rms = float(dh.float().pow(2).mean().sqrt().item())
        stack = {"value": NS * world / (sms / 1e3), "unit": "layer tokens/s", "layers": NS,
                 "ms_per_stack": sms, "us_per_layer": sms * 1e3 / NS, "steps": ns,
                 "d_in_finite": stack_finite, "d_in_rms": stack_rms,
                 "note": "one token through %d decode layers per step (tlb_stack_backward, one CUDA graph); "
                         "W_down, W_gate, W_up scales x 1/sqrt(5e3) so d_in stays finite (it grows about 2x "
                         "per layer instead of 5e3x)" % NS}
        del sl, sws

    cpu = None
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        t_or, n_or = oracle_step_time(cfg, args.cpu_seconds)
        cpu = {"value": 1.0 / t_or, "unit": UNIT, "cores": host_threads(), "kind": "oracle",
               "sample": "%d decode layer backwards of layer 0 (float64 numpy oracle)" % n_or}

    if rank == 0:
        step_bytes = decode_bytes(cfg)
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": {"workload": "decode layer backward: dim 2560, ffn 6912, 20/5 heads "
                                       "x 128, cache 1024, pos 1023, " +
                                       ("packed 2-bit" if cfg.wtype == "ternary2" else "int8") +
                                       " ternary weights, ReLU^2xMul, "
                                       "sub-norms, " + ("QK-norm on q, " if cfg.qk_norm else "") +
                                       "LoRA r16 Q/V, AdamW+LoRA+",
                           "global_batch": world, "seq_len": 1, "parallelism": "replicas" if world > 1 else "single",
                           "layers_cycled": NL, "l2": "inputs > L2: %d distinct layers x %.1f MB" % (NL, step_bytes / 1e6),
                           "cuda_graph": "one graph per cycle of %d layer calls" % NL if cycle is not None else False},
                "roofline": {"bound": "hbm", "kernel": kern[dom][0], "achieved": achieved, "peak": hbm,
                             "unit": "GB/s", "frac": achieved / hbm, "traffic": traffic,
                             "algorithmic_bytes": kern[dom][1],
                             "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)" if pk else "fallback"},
                "per_kernel": per_kernel, "per_kernel_timing": ktiming,
                "per_kernel_note": "events recorded between the kernels serialise the programmatic launches, so "
                                   "each kernel's time here includes the wait for its predecessor and its first "
                                   "round of loads (about its time alone); in the live chain k2 spans about 11 us "
                                   "(per-block globaltimer timeline, profiles/decode_kernels.md)",
                "step_roofline": {"bytes_per_step": step_bytes, "achieved": step_bytes / (ms_max / args.steps / 1e3) / 1e9,
                                  "peak": hbm, "unit": "GB/s",
                                  "frac": step_bytes / (ms_max / args.steps / 1e3) / 1e9 / hbm},
                "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
                "clocks": clk, "in_stack": stack}
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
