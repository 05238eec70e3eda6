// Composition of the layer backward and the layer-level extern "C" entry points:
// FFN backward ([FFN] "Backward (reverse)", executeFFNBackward; [RS] FFN part of
// backward_through_layers), attention backward ([ATT] "Gradient Flow"; [RS]
// attention block), LoRA Q/V gradients with AdamW ([RS] LoRA blocks, cpu_adamw).
#include "common.cuh"
#include "kernels.cuh"
#include "decode.cuh"

#include <algorithm>
#include <map>
#include <mutex>

namespace tlb {

namespace {

struct LayerWs {
    size_t dF, dG, dU, dN2, dSub, dqpre, dv, lora_q, lora_v;   // lora_*: tiled LoRA partial sums
    size_t abf, gbf, ubf, part;               // tensor-core path: bf16 A operands, split-K partials
    size_t atc;                               // tensor-core attention: tf32 operand copies
    size_t dR1, Upart, Wpart, Dpart, gh2, part1, part2, part3, gbar, pp;   // single-token path
    size_t dk, dkpart, Dh, dn1, dctx, xbf, dkx;   // exact layer-input gradient (TLB_EXACT_DIN)
    size_t total;
};

// The sequence FFN / O-projection products run on tcgen05 when the weights are bf16.
bool tc_route(const tlb_layer_cfg &c, int64_t S) {
    const int64_t I = c.ffn_dim, H = c.dim, qd = int64_t(c.n_heads) * c.head_dim;
    return c.wtype == TLB_W_BF16 && S > 1 && tc_supported(S, I, H) && tc_supported(S, H, 2 * I) &&
           tc_supported(S, qd, H) && I % 8 == 0;
}

// With bf16 weights the sequence attention contractions run on tcgen05 too (tf32
// operands); fp32 and ternary layers keep the fp32 CUDA-core kernels.
bool attn_tc_route(const tlb_layer_cfg &c, int64_t S, int64_t L) {
    return c.wtype == TLB_W_BF16 && !(c.flags & TLB_RECOMPUTE_P) &&
           attn_tc_supported(S, L, c.n_heads, c.n_kv_heads, c.head_dim);
}

// The recomputed attention (TLB_RECOMPUTE_P) runs its flash-style tcgen05 kernels on the
// same layers; with the exact input gradient it keeps the CUDA-core kernels, whose key
// gradient recomputes too.
bool attn_tc_rc_route(const tlb_layer_cfg &c, int64_t S, int64_t L) {
    return c.wtype == TLB_W_BF16 && (c.flags & TLB_RECOMPUTE_P) && !(c.flags & TLB_EXACT_DIN) &&
           attn_tc_supported(S, L, c.n_heads, c.n_kv_heads, c.head_dim);
}

LayerWs plan(const tlb_layer_cfg &c, int64_t S, int64_t L) {
    WsPlan p;
    LayerWs w;
    const int64_t I = c.ffn_dim, H = c.dim, qd = int64_t(c.n_heads) * c.head_dim;
    const int64_t kvd = int64_t(c.n_kv_heads) * c.head_dim;
    const bool exact = (c.flags & TLB_EXACT_DIN) != 0;
    if (tc_route(c, S)) {
        w.abf = p.take(S * H * 2);            // dOut, later dR1, in bf16
        w.gbf = p.take(S * I * 2);            // dG in bf16
        w.ubf = p.take(S * I * 2);            // dU in bf16
        size_t part = std::max({tc_partial_bytes(S, I, H), tc_partial_bytes(S, H, 2 * I),
                                tc_partial_bytes(S, qd, H), size_t(256)});
        if (exact) part = std::max({part, tc_partial_bytes(S, H, qd + 2 * kvd), tc_partial_bytes(S, H, qd),
                                    tc_partial_bytes(S, H, kvd)});
        w.part = p.take(part);
    } else {
        w.abf = w.gbf = w.ubf = w.part = 0;
    }
    w.atc = attn_tc_route(c, S, L)      ? p.take(attn_tc_bytes(S, L, c.n_heads, c.n_kv_heads, c.head_dim))
            : attn_tc_rc_route(c, S, L) ? p.take(attn_tc_rc_bytes(S, L, c.n_heads, c.n_kv_heads, c.head_dim))
                                        : 0;
    w.dF = p.take(S * I * 4);
    w.dG = p.take(S * I * 4);
    w.dU = p.take(S * I * 4);
    w.dN2 = p.take(S * H * 4);
    w.dSub = p.take(S * qd * 4);
    w.dqpre = p.take(S * qd * 4);
    w.dv = p.take(S * kvd * 4);
    w.lora_q = p.take(lora_seq_bytes(S, int(qd), int(H), c.rank));
    w.lora_v = p.take(lora_seq_bytes(S, int(kvd), int(H), c.rank));
    if (S == 1) {
        const int64_t nchunks = ceil_div(L, int64_t(std::min(32, kDecodeChunk)));   // the finer chunking
        w.dR1 = p.take(H * 4);
        w.Upart = p.take(nchunks * qd * 4);
        w.Wpart = p.take(nchunks * qd * 4);
        w.Dpart = p.take(nchunks * c.n_heads * 4);
        w.gh2 = p.take(2 * int64_t(c.rank) * 4);
        w.part1 = p.take(ceil_div(I, 8) * 8);   // one float2 per block of >= 8 rows
        w.part2 = p.take(ceil_div(H, 8) * 8);
        w.part3 = p.take(ceil_div(qd, 8) * 8);
        w.gbar = p.take(256);
        w.pp = p.take(3 * int64_t(kMaxPersistentBlocks) * 8);
    } else {
        w.dR1 = w.Upart = w.Wpart = w.Dpart = w.gh2 = w.part1 = w.part2 = w.part3 = w.gbar = w.pp = 0;
    }
    if (exact) {
        w.dk = p.take(S * kvd * 4);
        w.dkpart = p.take(std::max(attn_dk_bytes(S, c.n_heads, c.n_kv_heads, c.head_dim), size_t(256)));
        w.Dh = p.take(int64_t(c.n_heads) * S * 4);
        w.dn1 = p.take(S * H * 4);
        w.dctx = p.take(S * qd * 4);
        // [dQpre | dK | dV] in bf16, the A operands of the three-segment tcgen05 product
        // (q_dim, kv_dim multiples of 8: every operand 16-byte aligned, whole float4 groups)
        const bool tcx = tc_route(c, S) && qd % 8 == 0 && kvd % 8 == 0 && tc_supported(S, H, qd) &&
                         tc_supported(S, H, kvd);
        w.xbf = tcx ? p.take(S * (qd + 2 * kvd) * 2) : 0;
        // the tcgen05 key gradient: tf32 copies of dCtx and of q transposed
        w.dkx = attn_tc_route(c, S, L) ? p.take(attn_tc_dk_bytes(S, c.n_heads, c.head_dim)) : 0;
    } else {
        w.dk = w.dkpart = w.Dh = w.dn1 = w.dctx = w.xbf = w.dkx = 0;
    }
    w.total = p.off;
    return w;
}

int validate_cfg(const tlb_layer_cfg *c) {
    TLB_REQUIRE(c != nullptr, TLB_EINVAL, "layer cfg is NULL");
    TLB_REQUIRE(c->dim > 0 && c->ffn_dim > 0 && c->n_heads > 0 && c->n_kv_heads > 0 && c->head_dim > 0,
                TLB_EINVAL, "layer cfg: dimensions must be positive");
    TLB_REQUIRE(c->n_heads % c->n_kv_heads == 0, TLB_EINVAL,
                "layer cfg: n_heads (%d) not a multiple of n_kv_heads (%d)", c->n_heads, c->n_kv_heads);
    TLB_REQUIRE(c->head_dim % 2 == 0, TLB_EINVAL, "layer cfg: head_dim must be even");
    TLB_REQUIRE(c->head_dim <= 256, TLB_EUNSUPPORTED, "layer cfg: head_dim > 256");
    TLB_REQUIRE(c->rank >= 1 && c->rank <= 64, TLB_EINVAL, "layer cfg: rank must be in 1..64");
    TLB_REQUIRE(c->act == TLB_ACT_RELU2_MUL || c->act == TLB_ACT_SILU_MUL, TLB_EINVAL,
                "layer cfg: unknown activation %d", c->act);
    TLB_REQUIRE(c->wtype == TLB_W_F32 || c->wtype == TLB_W_BF16 || c->wtype == TLB_W_TERNARY_I8 ||
                    c->wtype == TLB_W_TERNARY_2B, TLB_EINVAL, "layer cfg: unknown weight type %d", c->wtype);
    if (c->wtype == TLB_W_TERNARY_2B)   // every weight row (out weights) a whole number of bytes
        TLB_REQUIRE(c->dim % 4 == 0 && c->ffn_dim % 4 == 0 && (c->n_heads * c->head_dim) % 4 == 0 &&
                        (c->n_kv_heads * c->head_dim) % 4 == 0,
                    TLB_EINVAL, "layer cfg: packed ternary weights need dim, ffn_dim, q_dim, kv_dim % 4 == 0");
    return TLB_OK;
}

int validate_ws(const tlb_layer_cfg *c, int64_t S, int64_t L, void *ws, size_t ws_bytes) {
    const size_t need = plan(*c, S, L).total;
    TLB_REQUIRE(ws != nullptr && ws_bytes >= need, TLB_EINVAL,
                "workspace of %zu bytes is smaller than the %zu bytes needed", ws_bytes, need);
    TLB_REQUIRE((reinterpret_cast<uintptr_t>(ws) & 255u) == 0, TLB_EINVAL, "workspace not 256-byte aligned");
    return TLB_OK;
}

// abf_dout: the workspace's bf16 operand buffer already holds dOut in bf16 (a stack's layer
// above left it there).  *abf_dres (optional) is set when the buffer ends up holding the
// finished d_res in bf16, the A operand of the O-projection product.
int ffn_impl(const tlb_layer_cfg &c, int64_t S, const float *d_out, const tlb_layer_weights &w,
             const tlb_layer_acts &a, float *d_res, void *ws, cudaStream_t st, bool abf_dout = false,
             bool *abf_dres = nullptr) {
    if (abf_dres != nullptr) *abf_dres = false;
    const LayerWs p = plan(c, S, S);   // the FFN regions do not depend on L
    const int64_t I = c.ffn_dim, H = c.dim;
    float *dF = ws_at<float>(ws, p.dF), *dG = ws_at<float>(ws, p.dG), *dU = ws_at<float>(ws, p.dU);
    if (tc_route(c, S) && w.w_gate.scale == w.w_up.scale) {
        uint32_t *status = ws_at<uint32_t>(ws, 0);
        float *part = ws_at<float>(ws, p.part);
        void *abf = ws_at<void>(ws, p.abf), *gbf = ws_at<void>(ws, p.gbf), *ubf = ws_at<void>(ws, p.ubf);
        // dF = dOut W_down^T on the tensor cores (dOut rounded to bf16); dG, dU in bf16 are
        // the A operands of [W_gate | W_up]^T
        if (!abf_dout) TLB_TRY(tc_convert_bf16(d_out, abf, S * H, st));
        const TcOperand down{abf, w.w_down.w, H};
        const float *sg = (c.act == TLB_ACT_SILU_MUL && (c.flags & TLB_USE_SILU_CACHE)) ? a.silu_gate : nullptr;
        const bool fuse = !(c.flags & TLB_SUB_NORM) && aligned16(a.gate) && aligned16(a.up) &&
                          (sg == nullptr || aligned16(sg));
        if (!fuse) {
            TLB_TRY(tc_gemm(&down, 1, S, I, w.w_down.scale, dF, false, part, status, st));
            if (c.flags & TLB_SUB_NORM)
                TLB_TRY(rmsnorm_backward_launch(a.hidden, w.gamma_sub_ffn, dF, dF, S, I, c.norm_eps, 0, st));
            TLB_TRY(act_backward_bf16_launch(c.act, a.gate, a.up, sg, dF, gbf, ubf, S * I, st));
        } else {
            // the activation backward runs in the product's epilogue: dF never reaches memory.
            // The epilogue is bound by its loads, so it recomputes silu(gate) from the gate
            // value it reads rather than loading the cache (a third of its reads)
            const TcActEpilogue ae{c.act, a.gate, a.up, gbf, ubf};
            TLB_TRY(tc_gemm(&down, 1, S, I, w.w_down.scale, nullptr, false, part, status, st, &ae));
        }
        const TcOperand gu[2] = {{gbf, w.w_gate.w, I}, {ubf, w.w_up.w, I}};
        const bool resid = (c.flags & TLB_RESIDUAL) != 0;
        if (c.flags & TLB_PRE_NORM) {
            float *dN2 = ws_at<float>(ws, p.dN2);
            TLB_TRY(tc_gemm(gu, 2, S, H, w.w_gate.scale, dN2, false, part, status, st));
            if (resid && d_res != d_out)
                TLB_CUDA(cudaMemcpyAsync(d_res, d_out, size_t(S * H) * 4, cudaMemcpyDeviceToDevice, st));
            return rmsnorm_backward_launch(a.r1, w.gamma_ffn, dN2, d_res, S, H, c.norm_eps, resid ? 1 : 0, st);
        }
        if (resid && d_res != d_out)
            TLB_CUDA(cudaMemcpyAsync(d_res, d_out, size_t(S * H) * 4, cudaMemcpyDeviceToDevice, st));
        // the epilogue also leaves d_res in bf16 where dOut was (the W_down^T product is done with it)
        TLB_TRY(tc_gemm(gu, 2, S, H, w.w_gate.scale, d_res, resid, part, status, st, nullptr, abf));
        if (abf_dres != nullptr) *abf_dres = true;
        return TLB_OK;
    }
    // dF = dOut W_down^T
    TLB_TRY(linear_t_launch(c.wtype, w.w_down.w, w.w_down.scale, d_out, S, H, I, dF, false, st));
    // dh = RMSNorm_bwd(hidden, gamma, dF) (sub-norm), in place
    if (c.flags & TLB_SUB_NORM)
        TLB_TRY(rmsnorm_backward_launch(a.hidden, w.gamma_sub_ffn, dF, dF, S, I, c.norm_eps, 0, st));
    // dG, dU = activation backward
    const float *sg = (c.act == TLB_ACT_SILU_MUL && (c.flags & TLB_USE_SILU_CACHE)) ? a.silu_gate : nullptr;
    TLB_TRY(act_backward_launch(c.act, a.gate, a.up, sg, dF, dG, dU, S * I, st));
    const bool resid = (c.flags & TLB_RESIDUAL) != 0;
    if (resid && d_res != d_out)
        TLB_CUDA(cudaMemcpyAsync(d_res, d_out, size_t(S * H) * 4, cudaMemcpyDeviceToDevice, st));
    if (c.flags & TLB_PRE_NORM) {
        float *dN2 = ws_at<float>(ws, p.dN2);
        TLB_TRY(linear_t_launch(c.wtype, w.w_gate.w, w.w_gate.scale, dG, S, I, H, dN2, false, st));
        TLB_TRY(linear_t_launch(c.wtype, w.w_up.w, w.w_up.scale, dU, S, I, H, dN2, true, st));
        // dResidual (+)= RMSNorm_bwd(r1, gamma_ffn, dN2)
        TLB_TRY(rmsnorm_backward_launch(a.r1, w.gamma_ffn, dN2, d_res, S, H, c.norm_eps, resid ? 1 : 0, st));
    } else {
        TLB_TRY(linear_t_launch(c.wtype, w.w_gate.w, w.w_gate.scale, dG, S, I, H, d_res, resid, st));
        TLB_TRY(linear_t_launch(c.wtype, w.w_up.w, w.w_up.scale, dU, S, I, H, d_res, true, st));
    }
    return TLB_OK;
}

AttnArgs attn_args(const tlb_layer_cfg &c, int64_t S, int64_t L, const float *dctx, const tlb_layer_acts &a,
                   float *d_qpre, float *d_v) {
    AttnArgs g;
    g.dctx = dctx;
    g.k = a.k;
    g.v = a.v;
    g.sh = a.kv_stride_head;
    g.sp = a.kv_stride_pos;
    g.attn = a.attn;
    g.dq = d_qpre;
    g.dv = d_v;
    g.S = int(S);
    g.L = int(L);
    g.nh = c.n_heads;
    g.nkv = c.n_kv_heads;
    g.hd = c.head_dim;
    g.pos0 = int(L - S);
    g.causal = (c.flags & TLB_CAUSAL) ? 1 : 0;
    g.rope = (c.flags & TLB_ROPE) ? 1 : 0;
    g.scale = c.attn_scale;
    g.D = nullptr;
    g.q = a.q;
    g.lse = (c.flags & TLB_RECOMPUTE_P) ? a.lse : nullptr;
    return g;
}

// abf_dr1: the workspace's bf16 operand buffer already holds dR1 in bf16.  D (optional):
// receives the attention's row sums D[h, i].
int attn_impl(const tlb_layer_cfg &c, int64_t S, int64_t L, const float *dR1, const tlb_layer_weights &w,
              const tlb_layer_acts &a, float *d_qpre, float *d_v, void *ws, cudaStream_t st, bool abf_dr1 = false,
              float *D = nullptr) {
    const LayerWs p = plan(c, S, L);
    const int64_t qd = int64_t(c.n_heads) * c.head_dim;
    float *dSub = ws_at<float>(ws, p.dSub);
    const bool tc_attn = (attn_tc_route(c, S, L) && aligned16(d_qpre) && aligned16(d_v) && aligned16(a.attn)) ||
                         (attn_tc_rc_route(c, S, L) && aligned16(d_qpre) && aligned16(d_v) && aligned16(a.q));
    // without the sub-norm dSub is dCtx, and the product also writes the attention kernels'
    // tf32 dCtx^T (the start of their scratch, rows of S rounded up to 4)
    const bool dct = tc_attn && tc_route(c, S) && !(c.flags & TLB_SUB_NORM);
    // and on the stored-weight path without the exact input gradient nothing else reads dCtx
    // by rows: the product writes only the transposed copy
    const bool dct_only = dct && !(c.flags & TLB_RECOMPUTE_P) && !(c.flags & TLB_EXACT_DIN);
    // dSub = dR1 W_O^T
    if (tc_route(c, S)) {
        void *abf = ws_at<void>(ws, p.abf);
        if (!abf_dr1) TLB_TRY(tc_convert_bf16(dR1, abf, S * c.dim, st));
        const TcOperand o{abf, w.w_o.w, c.dim};
        TLB_TRY(tc_gemm(&o, 1, S, qd, w.w_o.scale, dct_only ? nullptr : dSub, false, ws_at<float>(ws, p.part),
                        ws_at<uint32_t>(ws, 0), st, nullptr, nullptr, dct ? ws_at<float>(ws, p.atc) : nullptr,
                        (S + 3) & ~int64_t(3)));
    } else {
        TLB_TRY(linear_t_launch(c.wtype, w.w_o.w, w.w_o.scale, dR1, S, c.dim, qd, dSub, false, st));
    }
    // dCtx = RMSNorm_bwd(ctx, gamma_sub_attn, dSub) (sub-norm), in place
    if (c.flags & TLB_SUB_NORM)
        TLB_TRY(rmsnorm_backward_launch(a.ctx, w.gamma_sub_attn, dSub, dSub, S, qd, c.norm_eps, 0, st));
    AttnArgs g = attn_args(c, S, L, dSub, a, d_qpre, d_v);
    g.D = D;
    g.dct_ready = dct ? 1 : 0;
    if (dct_only) g.dctx = nullptr;
    if (tc_attn)
        TLB_TRY(attn_tc_launch(g, c.rope_base, ws_at<void>(ws, p.atc), ws_at<uint32_t>(ws, 0), st));
    else
        TLB_TRY(attn_core_launch(g, c.rope_base, st));
    // QK-norm: dQpre of each (row, head) back through the per-head RMSNorm, in place
    if (c.flags & TLB_QK_NORM)
        return rmsnorm_backward_launch(a.q_raw, w.gamma_q, d_qpre, d_qpre, S * c.n_heads, c.head_dim, c.norm_eps,
                                       0, st);
    return TLB_OK;
}

// Where exact_din_impl left the projections' input gradient (the LoRA A paths go there too).
float *exact_dst(const tlb_layer_cfg &c, float *d_hidden, void *ws, const LayerWs &p) {
    return (c.flags & TLB_PRE_NORM) ? ws_at<float>(ws, p.dn1) : d_hidden;
}

// TLB_EXACT_DIN (first part): the gradient of the layer input x_in beyond the pages' truncation
// (they stop at the Q / V projection outputs), the plain derivative of the stated forward
// with n1 = [RMSNorm(x_in; gamma_attn)] feeding the Q, K and V projections and both LoRA
// A products:
//   dK    = scale sum_group dS^T q on the S new cache rows, then RoPE backward and, with the
//           QK-norm, the per-head RMSNorm backward with gamma_k;
//   dn1   = s_q dQpre W_Q^T + s_k dK W_K^T + s_v dV W_V^T + s (dQpre B_q) A_q + s (dV B_v) A_v
//           (the last two, with A and B from before their AdamW step, are added by the LoRA
//           kernels, which form gh = s G B anyway);
//   d_in  = [dR1] + [RMSNorm_bwd(x_in, gamma_attn, dn1)]   (residual, pre-norm: exact_din_finish).
// d_hidden holds dR1 on entry (already consumed by the O-projection product); without the
// pre-norm dn1 is formed on d_hidden itself.  dctx: the attention's dCtx; D: its row sums.
int exact_din_impl(const tlb_layer_cfg &c, int64_t S, int64_t L, const tlb_layer_weights &w,
                   const tlb_layer_acts &a, const float *dqpre, const float *dv, const float *dctx, const float *D,
                   float *d_hidden, void *ws, const LayerWs &p, cudaStream_t st) {
    const int64_t H = c.dim, qd = int64_t(c.n_heads) * c.head_dim, kvd = int64_t(c.n_kv_heads) * c.head_dim;
    float *dk = ws_at<float>(ws, p.dk);
    const AttnArgs g = attn_args(c, S, L, dctx, a, nullptr, nullptr);
    if (p.dkx != 0 && aligned16(a.attn) && aligned16(a.q))   // the attention ran on tcgen05 too
        TLB_TRY(attn_tc_dk_launch(g, a.q, D, dk, ws_at<void>(ws, p.atc), ws_at<void>(ws, p.dkx),
                                  ws_at<uint32_t>(ws, 0), st));
    else
        TLB_TRY(attn_dk_launch(g, a.q, D, dk, ws_at<float>(ws, p.dkpart), st));
    if (c.flags & TLB_ROPE)
        TLB_TRY(rope_backward_launch(dk, dk, S, c.n_kv_heads, c.head_dim, L - S, c.rope_base, st));
    if (c.flags & TLB_QK_NORM)
        TLB_TRY(rmsnorm_backward_launch(a.k_raw, w.gamma_k, dk, dk, S * c.n_kv_heads, c.head_dim, c.norm_eps, 0, st));
    const bool pre = (c.flags & TLB_PRE_NORM) != 0, resid = (c.flags & TLB_RESIDUAL) != 0;
    // the projections' input gradient goes to dn1 (the pre-norm backward then adds it into
    // d_hidden) or, without the pre-norm, straight onto d_hidden (added to dR1 with the
    // residual, over it without)
    float *dst = exact_dst(c, d_hidden, ws, p);
    const bool acc0 = !pre && resid;
    if (p.xbf != 0) {
        uint32_t *status = ws_at<uint32_t>(ws, 0);
        float *part = ws_at<float>(ws, p.part);
        char *xb = ws_at<char>(ws, p.xbf);
        void *qb = xb, *kb = xb + S * qd * 2, *vb = xb + S * (qd + kvd) * 2;
        TLB_TRY(tc_convert_bf16(dqpre, qb, S * qd, st));
        TLB_TRY(tc_convert_bf16(dk, kb, S * kvd, st));
        TLB_TRY(tc_convert_bf16(dv, vb, S * kvd, st));
        const TcOperand seg[3] = {{qb, w.w_q.w, qd}, {kb, w.w_k.w, kvd}, {vb, w.w_v.w, kvd}};
        if (w.w_q.scale == w.w_k.scale && w.w_q.scale == w.w_v.scale) {
            TLB_TRY(tc_gemm(seg, 3, S, H, w.w_q.scale, dst, acc0, part, status, st));
        } else {
            TLB_TRY(tc_gemm(&seg[0], 1, S, H, w.w_q.scale, dst, acc0, part, status, st));
            TLB_TRY(tc_gemm(&seg[1], 1, S, H, w.w_k.scale, dst, true, part, status, st));
            TLB_TRY(tc_gemm(&seg[2], 1, S, H, w.w_v.scale, dst, true, part, status, st));
        }
    } else {
        TLB_TRY(linear_t_launch(c.wtype, w.w_q.w, w.w_q.scale, dqpre, S, qd, H, dst, acc0, st));
        TLB_TRY(linear_t_launch(c.wtype, w.w_k.w, w.w_k.scale, dk, S, kvd, H, dst, true, st));
        TLB_TRY(linear_t_launch(c.wtype, w.w_v.w, w.w_v.scale, dv, S, kvd, H, dst, true, st));
    }
    return TLB_OK;
}

// The last step of the exact input gradient, after the LoRA A paths were added into dn1.
int exact_din_finish(const tlb_layer_cfg &c, int64_t S, const tlb_layer_weights &w, const tlb_layer_acts &a,
                     float *d_hidden, void *ws, const LayerWs &p, cudaStream_t st) {
    if (!(c.flags & TLB_PRE_NORM)) return TLB_OK;
    return rmsnorm_backward_launch(a.x_in, w.gamma_attn, ws_at<float>(ws, p.dn1), d_hidden, S, c.dim, c.norm_eps,
                                   (c.flags & TLB_RESIDUAL) ? 1 : 0, st);
}

int check_acts_exact(const tlb_layer_cfg &c, const tlb_layer_weights *w, const tlb_layer_acts *a) {
    if (!(c.flags & TLB_EXACT_DIN)) return TLB_OK;
    TLB_REQUIRE(w->w_q.w && w->w_k.w && w->w_v.w, TLB_EINVAL, "EXACT_DIN needs w_q, w_k and w_v");
    TLB_REQUIRE(a->q, TLB_EINVAL, "EXACT_DIN needs q (the cached queries after RoPE)");
    if (c.flags & TLB_PRE_NORM)
        TLB_REQUIRE(a->x_in && w->gamma_attn, TLB_EINVAL, "EXACT_DIN with PRE_NORM needs x_in and gamma_attn");
    if (c.flags & TLB_QK_NORM)
        TLB_REQUIRE(a->k_raw && w->gamma_k, TLB_EINVAL, "EXACT_DIN with QK_NORM needs k_raw and gamma_k");
    return TLB_OK;
}

int check_acts_ffn(const tlb_layer_cfg &c, const tlb_layer_weights *w, const tlb_layer_acts *a) {
    TLB_REQUIRE(w && a, TLB_EINVAL, "weights / activations struct is NULL");
    TLB_REQUIRE(w->w_down.w && w->w_gate.w && w->w_up.w, TLB_EINVAL, "FFN weight pointer is NULL");
    TLB_REQUIRE(a->gate && a->up, TLB_EINVAL, "gate / up activation is NULL");
    if (c.flags & TLB_SUB_NORM)
        TLB_REQUIRE(a->hidden && w->gamma_sub_ffn, TLB_EINVAL, "SUB_NORM needs hidden and gamma_sub_ffn");
    if (c.flags & TLB_PRE_NORM)
        TLB_REQUIRE(a->r1 && w->gamma_ffn, TLB_EINVAL, "PRE_NORM needs r1 and gamma_ffn");
    if (c.act == TLB_ACT_SILU_MUL && (c.flags & TLB_USE_SILU_CACHE))
        TLB_REQUIRE(a->silu_gate, TLB_EINVAL, "USE_SILU_CACHE needs silu_gate");
    return TLB_OK;
}

int check_acts_attn(const tlb_layer_cfg &c, int64_t S, int64_t L, const tlb_layer_weights *w,
                    const tlb_layer_acts *a) {
    TLB_REQUIRE(w && a, TLB_EINVAL, "weights / activations struct is NULL");
    TLB_REQUIRE(L >= S && S >= 0, TLB_EINVAL, "need 0 <= S <= L (S=%lld, L=%lld)", (long long)S, (long long)L);
    TLB_REQUIRE(L < (int64_t(1) << 24), TLB_EUNSUPPORTED, "cache length >= 2^24");
    TLB_REQUIRE(w->w_o.w && a->k && a->v, TLB_EINVAL, "W_O / K / V pointer is NULL");
    if (c.flags & TLB_RECOMPUTE_P)
        TLB_REQUIRE(a->q && a->lse, TLB_EINVAL, "RECOMPUTE_P needs q and lse");
    else
        TLB_REQUIRE(a->attn, TLB_EINVAL, "attn pointer is NULL");
    TLB_REQUIRE(a->kv_stride_pos >= c.head_dim && a->kv_stride_head >= c.head_dim, TLB_EINVAL,
                "K/V strides smaller than head_dim");
    if (c.flags & TLB_SUB_NORM)
        TLB_REQUIRE(a->ctx && w->gamma_sub_attn, TLB_EINVAL, "SUB_NORM needs ctx and gamma_sub_attn");
    if (c.flags & TLB_QK_NORM)
        TLB_REQUIRE(a->q_raw && w->gamma_q, TLB_EINVAL, "QK_NORM needs q_raw and gamma_q");
    return TLB_OK;
}

int check_lora(const tlb_lora *l, const char *tag) {
    TLB_REQUIRE(l && l->a && l->b && l->m_a && l->v_a && l->m_b && l->v_b, TLB_EINVAL,
                "LoRA %s adapter: NULL pointer", tag);
    return TLB_OK;
}

int check_adam(const tlb_adamw_cfg *a) {
    TLB_REQUIRE(a != nullptr, TLB_EINVAL, "adamw cfg is NULL");
    TLB_REQUIRE(a->step >= 1, TLB_EINVAL, "adamw step must be >= 1");
    return TLB_OK;
}

// The single-token kernels read every vector with 16-byte loads.
bool decode_route(const tlb_layer_cfg &c, int64_t S, int64_t L, const tlb_layer_weights *w,
                  const tlb_layer_acts *acts, const float *d_hidden) {
    // the single-token kernels read the cached attention row
    if (!decode_supported(c, S, L) || (c.flags & TLB_RECOMPUTE_P)) return false;
    for (const void *ptr : {(const void *)w->w_down.w, (const void *)w->w_gate.w, (const void *)w->w_up.w,
                            (const void *)w->w_o.w, (const void *)w->gamma_sub_ffn, (const void *)w->gamma_ffn,
                            (const void *)w->gamma_sub_attn, (const void *)acts->gate, (const void *)acts->up,
                            (const void *)acts->silu_gate, (const void *)acts->hidden, (const void *)acts->r1,
                            (const void *)acts->ctx, (const void *)d_hidden})
        if (ptr != nullptr && !aligned16(ptr)) return false;
    return true;
}

// Arguments of the single-token kernels for one layer; dOut is read from and dR1
// copied to d_hidden (a stack overrides both).
void decode_args(const tlb_layer_cfg &c, int64_t L, const tlb_layer_weights *w, const tlb_layer_acts *acts,
                 const tlb_lora *lora_q, const tlb_lora *lora_v, const tlb_adamw_cfg *adam, float *d_hidden,
                 double *sumsq, void *ws, const LayerWs &p, DecodeArgs &d) {
    const int qd = c.n_heads * c.head_dim, kvd = c.n_kv_heads * c.head_dim;
    float *dqpre = ws_at<float>(ws, p.dqpre), *dv = ws_at<float>(ws, p.dv);
    d.H = c.dim;
    d.I = c.ffn_dim;
    d.qd = qd;
    d.kvd = kvd;
    d.nh = c.n_heads;
    d.nkv = c.n_kv_heads;
    d.hd = c.head_dim;
    d.L = int(L);
    d.rank = c.rank;
    d.flags = c.flags;
    d.act = c.act;
    d.pos = int(L - 1);
    d.chunk = kDecodeChunk;
    d.nchunks = int(ceil_div(L, kDecodeChunk));
    d.eps = c.norm_eps;
    d.scale = c.attn_scale;
    d.lora_scaling = c.lora_alpha / float(c.rank);
    d.rope_base = c.rope_base;
    d.w_down = w->w_down.w;
    d.w_gate = w->w_gate.w;
    d.w_up = w->w_up.w;
    d.w_o = w->w_o.w;
    d.s_down = w->w_down.scale;
    d.s_gate = w->w_gate.scale;
    d.s_up = w->w_up.scale;
    d.s_o = w->w_o.scale;
    d.g_sub_ffn = w->gamma_sub_ffn;
    d.g_ffn = w->gamma_ffn;
    d.g_sub_attn = w->gamma_sub_attn;
    d.x = acts->x;
    d.gate = acts->gate;
    d.up = acts->up;
    d.silu_gate = acts->silu_gate;
    d.hidden = acts->hidden;
    d.r1 = acts->r1;
    d.ctx = acts->ctx;
    d.k = acts->k;
    d.v = acts->v;
    d.attn = acts->attn;
    d.hq = acts->lora_q_h;
    d.hv = acts->lora_v_h;
    d.q_raw = acts->q_raw;
    d.g_q = w->gamma_q;
    d.sh = acts->kv_stride_head;
    d.sp = acts->kv_stride_pos;
    d.d_hidden = d_hidden;
    d.dF = ws_at<float>(ws, p.dF);
    d.dN2 = ws_at<float>(ws, p.dN2);
    d.dR1 = ws_at<float>(ws, p.dR1);
    d.dSub = ws_at<float>(ws, p.dSub);
    d.Upart = ws_at<float>(ws, p.Upart);
    d.Wpart = ws_at<float>(ws, p.Wpart);
    d.Dpart = ws_at<float>(ws, p.Dpart);
    d.dqpre = dqpre;
    d.dv = dv;
    d.gh = ws_at<float>(ws, p.gh2);    // [gh_q | gh_v], 2 * rank floats
    d.lq = *lora_q;
    d.lv = *lora_v;
    d.ka = adam_coef(*adam, 1.0f);
    d.kb = adam_coef(*adam, float(adam->lr_b_mult));
    d.sumsq = sumsq;
    d.status = nullptr;
    d.Dout = nullptr;
    const int rpb = decode_rows_per_block();
    d.n1 = int(ceil_div(c.ffn_dim, rpb));
    d.n2 = int(ceil_div(c.dim, rpb));
    d.n3 = int(ceil_div(qd, rpb));
    // column ranges: more blocks in flight for the two GEMVs with few rows (whole 16-byte
    // weight chunks per range, ranges a multiple of 4 floats), as long as k2 stays one
    // wave of three blocks per SM
    const int E = c.wtype == TLB_W_F32 ? 4 : (c.wtype == TLB_W_BF16 ? 8 : (c.wtype == TLB_W_TERNARY_I8 ? 16 : 64));
    d.ns2 = 1;
    for (int n : {4, 2})
        if (c.ffn_dim % (n * E) == 0 && (c.ffn_dim / n) % 4 == 0 && int64_t(d.n2) * n <= 3 * num_sms()) {
            d.ns2 = n;
            break;
        }
    d.ns3 = 1;
    if (c.dim % (2 * E) == 0 && (c.dim / 2) % 4 == 0) d.ns3 = 2;
    d.part1 = ws_at<float2>(ws, p.part1);
    d.part2 = ws_at<float2>(ws, p.part2);
    d.part3 = ws_at<float2>(ws, p.part3);
    d.dout = d_hidden;
    d.dhid_out = d_hidden;
}

// Sites of the finiteness checks, recorded beside kDevNonFinite in the status block.
constexpr uint32_t kSiteDOut = 1;   // the gradient entering a layer call (or the top of a stack)
constexpr uint32_t kSiteDR1 = 2;    // a layer's dR1: the gradient it hands to the layer below

// Workspace sets of a single-token stack: layer l uses set l % kStackSets.
constexpr int kStackSets = 4;

// The second stream of a single-token stack: one per device, at the lowest priority, so
// that the blocks of the next layer's GEMV chain go first; with its events: e3 after a
// layer's k1 .. k3, e7[l % kStackSets] after layer l's k4 .. k7.  Created on first use,
// which must not be inside a stream capture.
struct SideStream {
    std::mutex mu;
    cudaStream_t s = nullptr;
    cudaEvent_t e3 = nullptr, e7[kStackSets] = {};
};

int side_stream(SideStream *&out) {
    static std::mutex mu;
    static std::map<int, SideStream *> all;
    int dev = 0;
    TLB_CUDA(cudaGetDevice(&dev));
    std::lock_guard<std::mutex> lock(mu);
    SideStream *&ss = all[dev];
    if (ss == nullptr) {
        auto *n = new SideStream();
        int least = 0, greatest = 0;
        TLB_CUDA(cudaDeviceGetStreamPriorityRange(&least, &greatest));
        TLB_CUDA(cudaStreamCreateWithPriority(&n->s, cudaStreamNonBlocking, least));
        TLB_CUDA(cudaEventCreateWithFlags(&n->e3, cudaEventDisableTiming));
        for (int i = 0; i < kStackSets; ++i) TLB_CUDA(cudaEventCreateWithFlags(&n->e7[i], cudaEventDisableTiming));
        ss = n;
    }
    out = ss;
    return TLB_OK;
}

size_t stack_half(const tlb_layer_cfg &c, int64_t S, int64_t L) {
    return (plan(c, S, L).total + 255) / 256 * 256;
}

}  // namespace
}  // namespace tlb

using namespace tlb;

// One layer.  abf_dout: the workspace's bf16 operand buffer already holds d_hidden in bf16
// (the stack's layer above ran with the same workspace and ended with its dR1 = d_in there).
static int layer_backward_impl(const tlb_layer_cfg *cfg, int64_t S, int64_t L, const tlb_layer_weights *w,
                               const tlb_layer_acts *acts, const tlb_lora *lora_q, const tlb_lora *lora_v,
                               const tlb_adamw_cfg *adam, float *d_hidden, double *sumsq, void *ws,
                               size_t ws_bytes, void *stream, bool abf_dout) {
    clear_error();
    TLB_TRY(validate_cfg(cfg));
    TLB_TRY(check_acts_ffn(*cfg, w, acts));
    TLB_TRY(check_acts_attn(*cfg, S, L, w, acts));
    TLB_TRY(check_acts_exact(*cfg, w, acts));
    TLB_TRY(check_lora(lora_q, "Q"));
    TLB_TRY(check_lora(lora_v, "V"));
    TLB_TRY(check_adam(adam));
    if (S == 0) return TLB_OK;
    TLB_REQUIRE(d_hidden && acts->x && acts->lora_q_h && acts->lora_v_h, TLB_EINVAL,
                "layer_backward: NULL d_hidden / x / lora_q_h / lora_v_h");
    TLB_TRY(validate_ws(cfg, S, L, ws, ws_bytes));
    cudaStream_t st = as_stream(stream);
    const tlb_layer_cfg &c = *cfg;
    const LayerWs p = plan(c, S, L);
    const int qd = c.n_heads * c.head_dim, kvd = c.n_kv_heads * c.head_dim;
    ProfileScope prof(st);
    float *dqpre = ws_at<float>(ws, p.dqpre), *dv = ws_at<float>(ws, p.dv);
    // TLB_CHECK_FINITE ([RS] contract of backward_through_layers: grad_hidden finite): the
    // dOut that enters and the dR1 that leaves the FFN half are checked before any adapter
    // gradient is formed from them; a non-finite value is recorded in the status block,
    // whose AdamW kernels then leave the adapters and their moments unchanged
    const bool chk = (c.flags & TLB_CHECK_FINITE) != 0;
    uint32_t *status = ws_at<uint32_t>(ws, 0);
    if (chk) TLB_TRY(finite_check_launch(d_hidden, S * c.dim, status, kSiteDOut, st));
    const bool exact = (c.flags & TLB_EXACT_DIN) != 0;
    float *Dh = exact ? ws_at<float>(ws, p.Dh) : nullptr;
    if (decode_route(c, S, L, w, acts, d_hidden)) {
        DecodeArgs d;
        decode_args(c, L, w, acts, lora_q, lora_v, adam, d_hidden, sumsq, ws, p, d);
        if (chk || exact) {
            if (chk) d.status = status;
            d.Dout = Dh;
            TLB_TRY(decode_ffn_launch(d, c.wtype, st, false));
            if (chk) {
                TLB_TRY(finite_check_launch(d.dR1, c.dim, status, kSiteDR1, st));
                TLB_TRY(finite_gate_launch(status, status, st));
            }
            if (!exact) return decode_attn_launch(d, st);
            // the exact input gradient needs A and B before k7's AdamW step
            TLB_TRY(decode_attn_launch(d, st, false));
            const float *dctx = d.dSub;
            if (c.flags & TLB_SUB_NORM) {
                float *t = ws_at<float>(ws, p.dctx);
                TLB_TRY(rmsnorm_backward_launch(acts->ctx, w->gamma_sub_attn, d.dSub, t, 1, qd, c.norm_eps, 0, st));
                dctx = t;
            }
            TLB_TRY(exact_din_impl(c, S, L, *w, *acts, dqpre, dv, dctx, Dh, d_hidden, ws, p, st));
            // gh = [gh_q | gh_v] from k4 / k6 (B before k7's step)
            const float *gh[2] = {d.gh, d.gh + c.rank};
            const float *A[2] = {lora_q->a, lora_v->a};
            TLB_TRY(lora_din_launch(1, c.dim, c.rank, gh, A, 2, exact_dst(c, d_hidden, ws, p), st));
            TLB_TRY(exact_din_finish(c, S, *w, *acts, d_hidden, ws, p, st));
            return decode_lora_launch(d, st);
        }
        if ((c.flags & TLB_PERSISTENT) && persistent_supported(c, S, L))
            return decode_persistent_launch(d, c, L, ws, p.gbar, p.pp, st);
        return decode_layer_launch(d, c.wtype, st);
    }
    bool abf_dr1 = false;
    TLB_TRY(ffn_impl(c, S, d_hidden, *w, *acts, d_hidden, ws, st, abf_dout && tc_route(c, S), &abf_dr1));
    if (chk) {
        TLB_TRY(finite_check_launch(d_hidden, S * c.dim, status, kSiteDR1, st));
        TLB_TRY(finite_gate_launch(status, status, st));
    }
    TLB_TRY(attn_impl(c, S, L, d_hidden, *w, *acts, dqpre, dv, ws, st, abf_dr1, Dh));
    if (exact)   // attn_impl left dCtx in the dSub region
        TLB_TRY(exact_din_impl(c, S, L, *w, *acts, dqpre, dv, ws_at<float>(ws, p.dSub), Dh, d_hidden, ws, p, st));
    const LoraJob jobs[2] = {{dqpre, acts->lora_q_h, qd, *lora_q, ws_at<void>(ws, p.lora_q)},
                             {dv, acts->lora_v_h, kvd, *lora_v, ws_at<void>(ws, p.lora_v)}};
    // on the tensor cores where the attention backward ran there (the same tf32 class)
    TLB_TRY(lora_seq_launch(S, c.dim, c.rank, c.lora_alpha, acts->x, jobs, 2, *adam, sumsq, st,
                            chk ? status : nullptr, exact ? exact_dst(c, d_hidden, ws, p) : nullptr,
                            (attn_tc_route(c, S, L) || attn_tc_rc_route(c, S, L)) ? status : nullptr));
    return exact ? exact_din_finish(c, S, *w, *acts, d_hidden, ws, p, st) : TLB_OK;
}

extern "C" {

size_t tlb_workspace_bytes(const tlb_layer_cfg *cfg, int64_t S, int64_t L) {
    if (cfg == nullptr || S < 0) return 0;
    return plan(*cfg, S, L < S ? S : L).total;
}

int tlb_ffn_backward(const tlb_layer_cfg *cfg, int64_t S, const float *d_out, const tlb_layer_weights *w,
                     const tlb_layer_acts *acts, float *d_residual, void *ws, size_t ws_bytes, void *stream) {
    clear_error();
    TLB_TRY(validate_cfg(cfg));
    TLB_REQUIRE(S >= 0, TLB_EINVAL, "ffn_backward: negative S");
    if (S == 0) return TLB_OK;
    TLB_REQUIRE(d_out && d_residual, TLB_EINVAL, "ffn_backward: NULL gradient pointer");
    TLB_TRY(check_acts_ffn(*cfg, w, acts));
    TLB_TRY(validate_ws(cfg, S, S, ws, ws_bytes));
    return ffn_impl(*cfg, S, d_out, *w, *acts, d_residual, ws, as_stream(stream));
}

int tlb_attn_backward(const tlb_layer_cfg *cfg, int64_t S, int64_t L, const float *d_attn_out,
                      const tlb_layer_weights *w, const tlb_layer_acts *acts, float *d_qpre, float *d_v,
                      void *ws, size_t ws_bytes, void *stream) {
    clear_error();
    TLB_TRY(validate_cfg(cfg));
    TLB_TRY(check_acts_attn(*cfg, S, L, w, acts));
    if (S == 0) return TLB_OK;
    TLB_REQUIRE(d_attn_out && d_qpre && d_v, TLB_EINVAL, "attn_backward: NULL gradient pointer");
    TLB_TRY(validate_ws(cfg, S, L, ws, ws_bytes));
    return attn_impl(*cfg, S, L, d_attn_out, *w, *acts, d_qpre, d_v, ws, as_stream(stream));
}

int tlb_lora_grad_adamw(int64_t S, int32_t out_dim, int32_t in_dim, int32_t rank, float alpha, const float *G,
                        const float *h, const float *x, const tlb_lora *lora, const tlb_adamw_cfg *adam,
                        double *sumsq, void *ws, size_t ws_bytes, void *stream) {
    clear_error();
    TLB_REQUIRE(S >= 0 && out_dim > 0 && in_dim > 0, TLB_EINVAL, "lora_grad_adamw: bad sizes");
    TLB_REQUIRE(rank >= 1 && rank <= 64, TLB_EINVAL, "lora_grad_adamw: rank must be in 1..64");
    TLB_TRY(check_lora(lora, "(lora_grad_adamw)"));
    TLB_TRY(check_adam(adam));
    TLB_REQUIRE(S == 0 || (G && h && x), TLB_EINVAL, "lora_grad_adamw: NULL input");
    if (S == 0) return TLB_OK;   // no tokens: no gradient and no step, as in tlb_layer_backward
    const size_t need = kStatusBytes + lora_seq_bytes(S, out_dim, in_dim, rank);
    TLB_REQUIRE(ws && ws_bytes >= need, TLB_EINVAL, "lora_grad_adamw: workspace smaller than %zu bytes", need);
    TLB_REQUIRE((reinterpret_cast<uintptr_t>(ws) & 255u) == 0, TLB_EINVAL, "workspace not 256-byte aligned");
    const LoraJob job{G, h, out_dim, *lora, ws_at<void>(ws, kStatusBytes)};
    return lora_seq_launch(S, in_dim, rank, alpha, x, &job, 1, *adam, sumsq, as_stream(stream));
}

int tlb_layer_backward(const tlb_layer_cfg *cfg, int64_t S, int64_t L, const tlb_layer_weights *w,
                       const tlb_layer_acts *acts, const tlb_lora *lora_q, const tlb_lora *lora_v,
                       const tlb_adamw_cfg *adam, float *d_hidden, double *sumsq, void *ws, size_t ws_bytes,
                       void *stream) {
    return layer_backward_impl(cfg, S, L, w, acts, lora_q, lora_v, adam, d_hidden, sumsq, ws, ws_bytes, stream,
                               false);
}

size_t tlb_stack_workspace_bytes(const tlb_layer_cfg *cfg, int64_t S, int64_t L) {
    if (cfg == nullptr || S < 0) return 0;
    // single-token layers rotate over kStackSets workspace sets; longer ones share one
    return (S == 1 ? kStackSets : 1) * stack_half(*cfg, S, L < S ? S : L);
}

int tlb_stack_backward(const tlb_layer_cfg *cfg, int64_t S, int64_t L, int32_t n_layers,
                       const tlb_layer_weights *w, const tlb_layer_acts *acts, const tlb_lora *lora_q,
                       const tlb_lora *lora_v, const tlb_adamw_cfg *adam, float *d_hidden, double *sumsq,
                       void *ws, size_t ws_bytes, void *stream) {
    clear_error();
    TLB_TRY(validate_cfg(cfg));
    TLB_REQUIRE(n_layers >= 0 && S >= 0, TLB_EINVAL, "stack_backward: negative n_layers or S");
    if (n_layers == 0 || S == 0) return TLB_OK;
    TLB_REQUIRE(w && acts && lora_q && lora_v, TLB_EINVAL, "stack_backward: NULL layer array");
    TLB_REQUIRE(d_hidden, TLB_EINVAL, "stack_backward: NULL d_hidden");
    TLB_TRY(check_adam(adam));
    const tlb_layer_cfg &c = *cfg;
    const size_t half = stack_half(c, S, L), need = (S == 1 ? kStackSets : 1) * half;
    TLB_REQUIRE(ws != nullptr && ws_bytes >= need, TLB_EINVAL,
                "stack workspace of %zu bytes is smaller than the %zu bytes needed", ws_bytes, need);
    TLB_REQUIRE((reinterpret_cast<uintptr_t>(ws) & 255u) == 0, TLB_EINVAL, "workspace not 256-byte aligned");
    // the overlap of a single-token stack hands dR1 down before the layer's attention half
    // has run, which the exact input gradient needs
    const bool exact = (c.flags & TLB_EXACT_DIN) != 0;
    bool pipelined = S == 1 && !(c.flags & TLB_PERSISTENT) && !exact;
    const bool chk = (c.flags & TLB_CHECK_FINITE) != 0;
    for (int l = 0; l < n_layers; ++l) {
        TLB_TRY(check_acts_ffn(c, &w[l], &acts[l]));
        TLB_TRY(check_acts_attn(c, S, L, &w[l], &acts[l]));
        TLB_TRY(check_acts_exact(c, &w[l], &acts[l]));
        TLB_TRY(check_lora(&lora_q[l], "Q"));
        TLB_TRY(check_lora(&lora_v[l], "V"));
        TLB_REQUIRE(acts[l].x && acts[l].lora_q_h && acts[l].lora_v_h, TLB_EINVAL,
                    "stack_backward: layer %d: NULL x / lora_q_h / lora_v_h", l);
        pipelined = pipelined && decode_route(c, S, L, &w[l], &acts[l], d_hidden);
    }
    if (!pipelined) {
        // the layers one after another on the caller's stream ([RS] backward_through_layers),
        // all in the first workspace set: on the tensor-core route each layer leaves its d_in
        // in bf16 in the set's operand buffer, where the next layer's first product reads it
        for (int l = n_layers - 1; l >= 0; --l)
            TLB_TRY(layer_backward_impl(cfg, S, L, &w[l], &acts[l], &lora_q[l], &lora_v[l], adam, d_hidden, sumsq,
                                        ws, half, stream, l < n_layers - 1 && !exact));
        return TLB_OK;
    }
    // Single-token layers: layer l's k1 .. k3 (its dR1, the next layer's dOut) on the
    // caller's stream, its k4 .. k7 on the side stream, so that the attention and LoRA
    // half of layer l runs beside the GEMV chain of layer l - 1.  Layer l uses workspace
    // set l % 4, last used by layer l + 4.  Before the first kernel of each even layer l
    // the caller's stream waits for layer l + 2's side work; the side stream is in order,
    // so that also covers every layer above, and with it layer l + 4 for layers l and
    // l - 1.  The k1 of the other layers starts as a programmatic dependent of the k3
    // before it.
    cudaStream_t st = as_stream(stream);
    SideStream *side = nullptr;
    TLB_TRY(side_stream(side));
    std::lock_guard<std::mutex> lock(side->mu);
    const LayerWs p = plan(c, S, L);
    auto set = [&](int l) { return static_cast<void *>(static_cast<char *>(ws) + size_t(l % kStackSets) * half); };
    // with TLB_CHECK_FINITE every check reports into the first set's status block, the
    // one tlb_workspace_status reads: the top dOut, then each layer's dR1 (the next layer's
    // dOut) before the layer's attention and LoRA half is released to the side stream
    uint32_t *status = ws_at<uint32_t>(ws, 0);
    if (chk) TLB_TRY(finite_check_launch(d_hidden, c.dim, status, kSiteDOut, st));
    for (int l = n_layers - 1; l >= 0; --l) {
        const bool wait = (l % 2 == 0) && l + 2 <= n_layers - 1;
        if (wait) TLB_CUDA(cudaStreamWaitEvent(st, side->e7[(l + 2) % kStackSets], 0));
        DecodeArgs d;
        decode_args(c, L, &w[l], &acts[l], &lora_q[l], &lora_v[l], adam, d_hidden, sumsq, set(l), p, d);
        d.dout = l == n_layers - 1 ? d_hidden : ws_at<float>(set(l + 1), p.dR1);
        d.dhid_out = l == 0 ? d_hidden : nullptr;
        // layer l's AdamW (k7, on the side stream) reads the step gate of its own set,
        // written after its dR1 check: it sees exactly the checks of layers n-1 .. l
        if (chk) d.status = ws_at<uint32_t>(set(l), 0);
        TLB_TRY(decode_ffn_launch(d, c.wtype, st, !chk && !wait && l < n_layers - 1));
        if (chk) {
            TLB_TRY(finite_check_launch(d.dR1, c.dim, status, kSiteDR1, st));
            TLB_TRY(finite_gate_launch(status, ws_at<uint32_t>(set(l), 0), st));
        }
        TLB_CUDA(cudaEventRecord(side->e3, st));
        TLB_CUDA(cudaStreamWaitEvent(side->s, side->e3, 0));
        TLB_TRY(decode_attn_launch(d, side->s));
        TLB_CUDA(cudaEventRecord(side->e7[l % kStackSets], side->s));
    }
    TLB_CUDA(cudaStreamWaitEvent(st, side->e7[0], 0));   // layer 0 ends the side stream's work
    return TLB_OK;
}

}  // extern "C"
