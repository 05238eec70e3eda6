// Attention backward over cached K/V with GQA, from dCtx down to dQpre and dV
// ([ATT] "Gradient Flow", apply / softmax / score / RoPE backward; [RS]
// backward_through_layers, attention block).
//
// General kernels (any S, L, strides):
//   attn_rows_kernel  one block per (query row i, head h):
//       dAttn[j] = dCtx[i,h,:] . V[kvh, j, :]                (apply backward)
//       D        = sum_j attn[h,i,j] dAttn[j]
//       dS[j]    = scale * attn[h,i,j] (dAttn[j] - D)         (softmax backward)
//       dQ[d]    = sum_j dS[j] K[kvh, j, d]                   (score backward)
//       dQpre    = R(-theta_pos) dQ                           (RoPE backward)
//   attn_dv_kernel    one block per (newest key jj, KV head):
//       dV[jj, kvh, d] = sum_{h in group} sum_i attn[h, i, L-S+jj] dCtx[i, h, d]
#include "common.cuh"
#include "kernels.cuh"

namespace tlb {

__global__ void attn_rows_kernel(AttnArgs a, RopeFreqs fr) {
    extern __shared__ float4 smem4[];
    __shared__ float red[32];
    float *sS = reinterpret_cast<float *>(smem4);
    float *sd = sS + a.L;
    float *sq = sd + a.hd;
    const int i = blockIdx.x, h = blockIdx.y;
    const int kvh = h / (a.nh / a.nkv);
    const int q_dim = a.nh * a.hd;
    const int jmax = a.causal ? min(a.L, a.pos0 + i + 1) : a.L;
    for (int d = threadIdx.x; d < a.hd; d += blockDim.x) sd[d] = a.dctx[int64_t(i) * q_dim + h * a.hd + d];
    __syncthreads();
    const float *Vh = a.v + int64_t(kvh) * a.sh;
    const float *Kh = a.k + int64_t(kvh) * a.sh;
    for (int j = threadIdx.x; j < jmax; j += blockDim.x) {
        const float *vr = Vh + int64_t(j) * a.sp;
        float acc = 0.f;
        for (int d = 0; d < a.hd; ++d) acc = fmaf(sd[d], vr[d], acc);
        sS[j] = acc;
    }
    const float *P = a.attn + (int64_t(h) * a.S + i) * a.L;
    float part = 0.f;
    for (int j = threadIdx.x; j < jmax; j += blockDim.x) part += P[j] * sS[j];
    const float D = block_sum(part, red);
    for (int j = threadIdx.x; j < jmax; j += blockDim.x) sS[j] = a.scale * P[j] * (sS[j] - D);
    __syncthreads();
    for (int d = threadIdx.x; d < a.hd; d += blockDim.x) {
        float acc = 0.f;
        for (int j = 0; j < jmax; ++j) acc = fmaf(sS[j], Kh[int64_t(j) * a.sp + d], acc);
        sq[d] = acc;
    }
    __syncthreads();
    float *out = a.dq + int64_t(i) * q_dim + h * a.hd;
    if (a.rope) {
        const int half = a.hd >> 1;
        for (int d = threadIdx.x; d < half; d += blockDim.x) {
            float c, s;
            rope_cos_sin(float(a.pos0 + i), fr.hi[d], fr.lo[d], c, s);
            const float y1 = sq[d], y2 = sq[d + half];
            out[d] = y1 * c + y2 * s;
            out[d + half] = -y1 * s + y2 * c;
        }
    } else {
        for (int d = threadIdx.x; d < a.hd; d += blockDim.x) out[d] = sq[d];
    }
}

__global__ void attn_dv_kernel(AttnArgs a) {
    const int jj = blockIdx.x, kvh = blockIdx.y;
    const int group = a.nh / a.nkv;
    const int j = a.pos0 + jj;
    const int q_dim = a.nh * a.hd;
    const int i0 = a.causal ? jj : 0;
    for (int d = threadIdx.x; d < a.hd; d += blockDim.x) {
        float acc = 0.f;
        for (int g = 0; g < group; ++g) {
            const int h = kvh * group + g;
            const float *P = a.attn + int64_t(h) * a.S * a.L + j;
            const float *dc = a.dctx + h * a.hd + d;
            for (int i = i0; i < a.S; ++i) acc = fmaf(P[int64_t(i) * a.L], dc[int64_t(i) * q_dim], acc);
        }
        a.dv[int64_t(jj) * a.nkv * a.hd + kvh * a.hd + d] = acc;
    }
}

int attn_core_launch(const AttnArgs &a, float rope_base, cudaStream_t st) {
    if (a.S == 0) return TLB_OK;
    RopeFreqs fr;
    rope_freqs(fr, a.hd, rope_base);
    const size_t smem = (size_t(a.L) + 2 * size_t(a.hd)) * sizeof(float);
    TLB_REQUIRE(smem <= 200 * 1024, TLB_EUNSUPPORTED, "attn_backward: cache length %d too long", a.L);
    if (smem > 48 * 1024)
        TLB_CUDA(cudaFuncSetAttribute(attn_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      int(smem)));
    attn_rows_kernel<<<dim3(a.S, a.nh), 128, smem, st>>>(a, fr);
    TLB_TRY(check_launch("attn_rows"));
    attn_dv_kernel<<<dim3(a.S, a.nkv), a.hd < 128 ? a.hd : 128, 0, st>>>(a);
    return check_launch("attn_dv");
}

}  // namespace tlb
