// Arguments of the single-token (decode) layer backward kernels (decode.cu).
#pragma once

#include "common.cuh"

namespace tlb {

struct DecodeArgs {
    int H, I, qd, kvd, nh, nkv, hd, L, rank, flags, act, pos, chunk, nchunks;
    float eps, scale, lora_scaling, rope_base;
    const void *w_down, *w_gate, *w_up, *w_o;
    float s_down, s_gate, s_up, s_o;
    const float *g_sub_ffn, *g_ffn, *g_sub_attn;
    const float *x, *gate, *up, *silu_gate, *hidden, *r1, *ctx, *k, *v, *attn, *hq, *hv;
    int64_t sh, sp;
    float *d_hidden;                                   // [H] in: dOut, out: dR1
    float *dF, *dN2, *dR1, *dSub, *dctx;               // workspace vectors
    float *Upart, *Wpart, *Dpart, *dqpre, *dv, *gh;    // workspace attention / LoRA
    tlb_lora lq, lv;
    AdamCoef ka, kb;
    double *sumsq;
    // per-block partial sums (sum dy g x, sum x^2) for the RMSNorm backward of the
    // vector each GEMV produces; n1..n3 = the GEMV grids (blocks of k1, k2, k3)
    float2 *part1, *part2, *part3;
    int n1, n2, n3;
};

constexpr int kDecodeChunk = 64;   // keys per block in the attention pass

bool decode_supported(const tlb_layer_cfg &c, int64_t S, int64_t L);
int decode_rows_per_block();
int decode_layer_launch(const DecodeArgs &a, int wtype, cudaStream_t st);

}  // namespace tlb
