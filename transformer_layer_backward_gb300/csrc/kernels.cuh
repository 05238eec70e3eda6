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
