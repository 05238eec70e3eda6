// Host-side launchers of the kernels, shared between translation units.  Every
// launcher enqueues on `st`, returns TLB_OK or an error code, and allocates nothing.
#pragma once

#include "common.cuh"

namespace tlb {

int softmax_backward_launch(const float *attn, const float *dattn, float *ds, int64_t rows,
                            int64_t len, cudaStream_t st);
int rmsnorm_backward_launch(const float *x, const float *gamma, const float *dy, float *dx,
                            int64_t rows, int64_t n, float eps, int accumulate, cudaStream_t st);
int act_backward_launch(int act, const float *gate, const float *up, const float *silu_gate,
                        const float *dh, float *dgate, float *dup, int64_t n, cudaStream_t st);
int rope_backward_launch(const float *dy, float *dx, int64_t rows, int n_heads, int head_dim,
                         int64_t pos0, float base, cudaStream_t st);
int adamw_launch(float *p, const float *g, float *m, float *v, int64_t n, const tlb_adamw_cfg &cfg,
                 float lr_mult, double *sumsq, cudaStream_t st);
// Records kDevNonFinite with `site` in the status block if any of x[0, n) is not finite.
int finite_check_launch(const float *x, int64_t n, uint32_t *status, uint32_t site, cudaStream_t st);
// gate_block[kStatusGate] = (a non-finite value is recorded in status): the step gate the
// AdamW kernels that come after it read.
int finite_gate_launch(const uint32_t *status, uint32_t *gate_block, cudaStream_t st);

}  // namespace tlb

namespace tlb {

// dX[S, in] (+)= scale * dY[S, out] . W[in, out]^T  (linear.cu)
// With a workspace of linear_ws_bytes() (status block first), bf16 weights and S > 1 take
// the tcgen05 path; otherwise (ws == nullptr allowed) the CUDA-core GEMM / GEMV.
int linear_t_launch(int wtype, const void *W, float scale, const float *dY, int64_t S, int64_t out_dim,
                    int64_t in_dim, float *dX, bool accumulate, cudaStream_t st, void *ws = nullptr,
                    size_t ws_bytes = 0);
size_t linear_ws_bytes(int wtype, int64_t S, int64_t out_dim, int64_t in_dim);
// tcgen05 GEMM (gemm_tc.cu): out[M, N] (+)= alpha * sum_seg A_seg[M, K_seg] . B_seg[N, K_seg]^T,
// A and B bf16 row-major (K-major), 16-byte aligned, K_seg % 8 == 0.
struct TcOperand {
    const void *a;   // bf16 [M, K]
    const void *b;   // bf16 [N, K]
    int64_t K;
};
struct TcPlan {
    int bn, ctas;    // tile width, persistent CTAs (CTA pairs when paired)
    int dp;          // whole tiles per CTA before the stream-K part
    int shared;      // CTA boundaries that fall inside a stream-K tile (0: no fixup)
    int pair;        // 1: clusters of two CTAs on 256 x 256 super-tiles (cta_group::2 MMA)
};
TcPlan tc_plan(int64_t M, int64_t N, int64_t K);
bool tc_supported(int64_t M, int64_t N, int64_t K);
size_t tc_partial_bytes(int64_t M, int64_t N, int64_t K);   // stream-K partial tiles for (M, N, K)
int tc_convert_bf16(const float *x, void *y, int64_t n, cudaStream_t st);
// Optional epilogue of tc_gemm: alpha * acc is dh, and the gated-activation backward
// writes dG, dU in bf16 (the A operands of the [W_gate | W_up]^T product) instead of out.
struct TcActEpilogue {
    int act;                              // TLB_ACT_*
    const float *gate, *up;               // [M, N] fp32; silu(gate) is recomputed
    void *dgate, *dup;                    // [M, N] bf16
};
// out_bf16 (optional, no activation epilogue): [M, N] bf16 copy of every value stored to out.
// out_t (optional, no activation epilogue, not accumulating): tf32-rounded transposed copy,
// out_t[c * ld_t + r] = tf32(out[r, c]) (the tensor-core attention's dCtx^T operand); with
// out_t, out may be null (only the copy is written).
int tc_gemm(const TcOperand *seg, int nseg, int64_t M, int64_t N, float alpha, float *out, bool accumulate,
            float *partial, uint32_t *status, cudaStream_t st, const TcActEpilogue *act = nullptr,
            void *out_bf16 = nullptr, float *out_t = nullptr, int64_t ld_t = 0);
// gated-activation backward writing bf16 dG, dU (rowwise.cu)
int act_backward_bf16_launch(int act, const float *gate, const float *up, const float *silu_gate, const float *dh,
                             void *dgate, void *dup, int64_t n, cudaStream_t st);

// Attention backward from dCtx to dQ(pre) and dV (attention.cu).
struct AttnArgs {
    const float *dctx;       // [S, q_dim]
    const float *k, *v;      // caches, element (kvh, j, d) at kvh*sh + j*sp + d
    int64_t sh, sp;
    const float *attn;       // [nh, S, L]
    float *dq;               // [S, q_dim]: dQpre when rope, else dQ
    float *dv;               // [S, kv_dim]: rows of keys L - S .. L - 1
    int S, L, nh, nkv, hd, pos0, causal, rope;
    float scale;
    float *D = nullptr;      // [nh, S] (optional): D[h, i] = sum_j attn[h,i,j] dAttn[h,i,j]
    // Recomputed attention (lse != NULL; attn unused): attn[h,i,j] = exp(scale <q[i,h,:],
    // k[j,kvh,:]> - lse[h,i]) on the visible keys, q [S, q_dim] the queries after RoPE.
    const float *q = nullptr;
    const float *lse = nullptr;   // [nh, S] logsumexp of each query row's scaled logits
    // tensor-core kernels: the scratch already holds the tf32 dCtx^T ([q_dim][S rounded up to
    // 4], at its start) that the O-projection product wrote (beside dctx; with dct_ready and
    // the stored weights, dctx may be null and the kernels read only the transposed copy)
    int dct_ready = 0;
};
int attn_core_launch(const AttnArgs &a, float rope_base, cudaStream_t st);
// Key gradient of the S newest cache rows (the keys of the call's own tokens), for the
// exact layer-input gradient:
//   dK[jj, kvh, :] = scale sum_{h in group} sum_i attn[h,i,j] (dCtx[i,h,:] . V[j,kvh,:] - D[h,i]) q[i,h,:]
// with j = L - S + jj, q [S, q_dim] the cached queries (after RoPE), D from the attention
// kernels; dk [S, kv_dim] (before RoPE backward).
// part: attn_dk_bytes(...) bytes of scratch (per-head partials; may be NULL when that is 0).
size_t attn_dk_bytes(int64_t S, int nh, int nkv, int hd);
int attn_dk_launch(const AttnArgs &a, const float *q, const float *D, float *dk, float *part, cudaStream_t st);

// Tensor-core (tf32) attention backward (attn_tc.cu): S > 1, head_dim 64 or 128, L and
// L - S multiples of 4; attn, dq and dv 16-byte aligned.  scratch: attn_tc_bytes(...) bytes, 256-byte aligned.
bool attn_tc_supported(int64_t S, int64_t L, int nh, int nkv, int hd);
size_t attn_tc_bytes(int64_t S, int64_t L, int nh, int nkv, int hd);
// With a.lse set (recomputed attention) the same entry runs the flash-style kernels (q 16-byte
// aligned instead of attn; attn unused); scratch: attn_tc_rc_bytes(...) bytes.
int attn_tc_launch(const AttnArgs &a, float rope_base, void *scratch, uint32_t *status, cudaStream_t st);
size_t attn_tc_rc_bytes(int64_t S, int64_t L, int nh, int nkv, int hd);
// Key gradient of the S newest keys on tcgen05 (the exact input gradient), after
// attn_tc_launch on the same scratch (its tf32 V copy and per-head partial buffer are
// reused); extra: attn_tc_dk_bytes(...) bytes, 16-byte aligned.  dk as attn_dk_launch.
size_t attn_tc_dk_bytes(int64_t S, int nh, int hd);
int attn_tc_dk_launch(const AttnArgs &a, const float *q, const float *D, float *dk, void *scratch, void *extra,
                      uint32_t *status, cudaStream_t st);

// LoRA gradients + AdamW of one adapter (lora.cu); gh: [S, rank] scratch.
int lora_launch(int64_t S, int out_dim, int in_dim, int rank, float alpha, const float *G, const float *h,
                const float *x, const tlb_lora &l, const tlb_adamw_cfg &adam, double *sumsq, float *gh,
                cudaStream_t st);

// Tiled LoRA gradients + AdamW (lora.cu) for one or two adapters that share x [S, in_dim].
// scratch: lora_seq_bytes(S, out_dim, in_dim, rank) bytes per adapter, 256-byte aligned.
struct LoraJob {
    const float *G, *h;     // [S, out_dim], [S, rank]
    int out_dim;
    tlb_lora l;
    void *scratch;
};
size_t lora_seq_bytes(int64_t S, int out_dim, int in_dim, int rank);
// The LoRA-A paths of the exact layer-input gradient: dn1[S, in_dim] += sum over the
// adapters of gh A, gh [S, rank] = s G B and A [rank, in_dim] both from before the update.
int lora_din_launch(int64_t S, int in_dim, int rank, const float *const *gh, const float *const *A, int njobs,
                    float *dn1, cudaStream_t st);
// The same passes on the tensor cores (lora_tc.cu, kind::tf32, rank 16): per adapter
// G [S, out_dim], h [S, 16], B [out_dim, 16] (before its update), gh [S, 16] (written
// between the passes) and the partial sums part_gh [n_ot][S][16], part_b [chunks][out][16],
// part_a [chunks][16][in_dim] of the CUDA-core passes, over chunks of 128-token tiles.
struct LoraTcJob {
    const float *G, *h, *b, *gh;
    float *part_gh, *part_b, *part_a;
    int out_dim;
};
bool lora_tc_supported(int64_t S, int in_dim, int rank, const float *x, const LoraTcJob *jobs, int njobs);
// Chunks of 128-token tiles for a pass over n_ct column tiles (about one CTA per SM).
int lora_tc_chunks(int64_t S, int n_ct, int &tiles_per_chunk);
int lora_tc_gpass_launch(int64_t S, const LoraTcJob *jobs, int njobs, int tiles_per_chunk, uint32_t *status,
                         cudaStream_t st);
int lora_tc_xpass_launch(int64_t S, int in_dim, const float *x, const LoraTcJob *jobs, int njobs,
                         int tiles_per_chunk, uint32_t *status, cudaStream_t st);
// tc (optional): run the passes on the tensor cores when lora_tc_supported holds, with
// bounded waits that run out recorded in this status block.
// status (optional): a status block whose step gate (kStatusGate) is 1 skips the AdamW
// steps (the gradients are still written and summed).
// din (optional): dn1 of the exact input gradient; gh A of every adapter is added into it
// between the gh sums and AdamW.
int lora_seq_launch(int64_t S, int in_dim, int rank, float alpha, const float *x, const LoraJob *jobs, int njobs,
                    const tlb_adamw_cfg &adam, double *sumsq, cudaStream_t st, const uint32_t *status = nullptr,
                    float *din = nullptr, uint32_t *tc = nullptr);

}  // namespace tlb
