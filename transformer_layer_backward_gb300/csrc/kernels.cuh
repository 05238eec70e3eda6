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

}  // namespace tlb

namespace tlb {

// dX[S, in] (+)= scale * dY[S, out] . W[in, out]^T  (linear.cu)
int linear_t_launch(int wtype, const void *W, float scale, const float *dY, int64_t S, int64_t out_dim,
                    int64_t in_dim, float *dX, bool accumulate, cudaStream_t st);
// Tensor-core path of the same product for bf16 weights; TLB_EUNSUPPORTED when the
// shape or alignment does not fit it (the caller then uses the CUDA-core GEMM).
int gemm_tc_try(const void *W, float scale, const float *dY, int64_t S, int64_t out_dim, int64_t in_dim,
                float *dX, bool accumulate, cudaStream_t st);

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
};
int attn_core_launch(const AttnArgs &a, float rope_base, cudaStream_t st);

// LoRA gradients + AdamW of one adapter (lora.cu); gh: [S, rank] scratch.
int lora_launch(int64_t S, int out_dim, int in_dim, int rank, float alpha, const float *G, const float *h,
                const float *x, const tlb_lora &l, const tlb_adamw_cfg &adam, double *sumsq, float *gh,
                cudaStream_t st);

}  // namespace tlb
