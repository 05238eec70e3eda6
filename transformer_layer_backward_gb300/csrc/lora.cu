// LoRA adapter gradients and their AdamW step ([RS] "LoRA Q backward" and
// "LoRA V backward", cpu_adamw, LoRA+ rate on B), s = alpha / rank:
//   gh[i, r] = s sum_o G[i, o] B[o, r]     (B before its update)
//   dB[o, r] = s sum_i G[i, o] h[i, r]     -> AdamW on B with lr * lr_b_mult
//   dA[r, c] = sum_i gh[i, r] x[i, c]      -> AdamW on A with lr
// The gradients stay in registers between their reduction and the update;
// sum dA^2 and sum dB^2 are added to sumsq[0] and sumsq[1].
#include "common.cuh"
#include "kernels.cuh"

namespace tlb {

template <int RB>
__global__ void __launch_bounds__(256)
lora_gh_kernel(const float *__restrict__ G, const float *__restrict__ B, float *__restrict__ gh,
               int out_dim, int rank, float scaling) {
    __shared__ float red[RB][8];
    const int i = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float acc[RB];
#pragma unroll
    for (int r = 0; r < RB; ++r) acc[r] = 0.f;
    const float *g = G + int64_t(i) * out_dim;
    for (int o = threadIdx.x; o < out_dim; o += blockDim.x) {
        const float gv = g[o];
        const float *b = B + int64_t(o) * rank;
#pragma unroll
        for (int r = 0; r < RB; ++r)
            if (r < rank) acc[r] = fmaf(gv, b[r], acc[r]);
    }
#pragma unroll
    for (int r = 0; r < RB; ++r) {
        const float v = warp_sum(acc[r]);
        if (lane == 0) red[r][warp] = v;
    }
    __syncthreads();
    if (threadIdx.x < rank) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) s += red[threadIdx.x][w];
        gh[int64_t(i) * rank + threadIdx.x] = scaling * s;
    }
}

__global__ void __launch_bounds__(256)
lora_db_adamw_kernel(const float *__restrict__ G, const float *__restrict__ h, int S, int out_dim, int rank,
                     float scaling, float *B, float *mB, float *vB, float *gradB, AdamCoef k,
                     double *sumsq) {
    __shared__ float red[32];
    const int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const bool valid = e < int64_t(out_dim) * rank;
    float db = 0.f;
    if (valid) {
        const int o = int(e / rank), r = int(e % rank);
        float acc = 0.f;
        for (int i = 0; i < S; ++i) acc = fmaf(G[int64_t(i) * out_dim + o], h[int64_t(i) * rank + r], acc);
        db = scaling * acc;
        if (gradB) gradB[e] = db;
        float m = mB[e], v = vB[e];
        B[e] = adam_elem(B[e], db, m, v, k);
        mB[e] = m;
        vB[e] = v;
    }
    if (sumsq) {
        const float ss = block_sum(db * db, red);
        if (threadIdx.x == 0) atomicAdd(sumsq + 1, double(ss));
    }
}

__global__ void __launch_bounds__(256)
lora_da_adamw_kernel(const float *__restrict__ gh, const float *__restrict__ x, int S, int in_dim, int rank,
                     float *A, float *mA, float *vA, float *gradA, AdamCoef k, double *sumsq) {
    __shared__ float red[32];
    const int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const bool valid = e < int64_t(rank) * in_dim;
    float da = 0.f;
    if (valid) {
        const int r = int(e / in_dim), c = int(e % in_dim);
        float acc = 0.f;
        for (int i = 0; i < S; ++i) acc = fmaf(gh[int64_t(i) * rank + r], x[int64_t(i) * in_dim + c], acc);
        da = acc;
        if (gradA) gradA[e] = da;
        float m = mA[e], v = vA[e];
        A[e] = adam_elem(A[e], da, m, v, k);
        mA[e] = m;
        vA[e] = v;
    }
    if (sumsq) {
        const float ss = block_sum(da * da, red);
        if (threadIdx.x == 0) atomicAdd(sumsq, double(ss));
    }
}

int lora_launch(int64_t S, int out_dim, int in_dim, int rank, float alpha, const float *G, const float *h,
                const float *x, const tlb_lora &l, const tlb_adamw_cfg &adam, double *sumsq, float *gh,
                cudaStream_t st) {
    if (S == 0) return TLB_OK;
    const float scaling = alpha / float(rank);
    if (rank <= 4) lora_gh_kernel<4><<<unsigned(S), 256, 0, st>>>(G, l.b, gh, out_dim, rank, scaling);
    else if (rank <= 8) lora_gh_kernel<8><<<unsigned(S), 256, 0, st>>>(G, l.b, gh, out_dim, rank, scaling);
    else if (rank <= 16) lora_gh_kernel<16><<<unsigned(S), 256, 0, st>>>(G, l.b, gh, out_dim, rank, scaling);
    else if (rank <= 32) lora_gh_kernel<32><<<unsigned(S), 256, 0, st>>>(G, l.b, gh, out_dim, rank, scaling);
    else lora_gh_kernel<64><<<unsigned(S), 256, 0, st>>>(G, l.b, gh, out_dim, rank, scaling);
    TLB_TRY(check_launch("lora_gh"));
    const AdamCoef kb = adam_coef(adam, adam.lr_b_mult);
    const AdamCoef ka = adam_coef(adam, 1.0f);
    lora_db_adamw_kernel<<<unsigned(ceil_div(int64_t(out_dim) * rank, 256)), 256, 0, st>>>(
        G, h, int(S), out_dim, rank, scaling, l.b, l.m_b, l.v_b, l.grad_b, kb, sumsq);
    TLB_TRY(check_launch("lora_db_adamw"));
    lora_da_adamw_kernel<<<unsigned(ceil_div(int64_t(rank) * in_dim, 256)), 256, 0, st>>>(
        gh, x, int(S), in_dim, rank, l.a, l.m_a, l.v_a, l.grad_a, ka, sumsq);
    return check_launch("lora_da_adamw");
}

}  // namespace tlb
