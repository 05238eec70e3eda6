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
    const float *q_raw, *g_q;                          // QK-norm: pre-norm q [qd], gain [hd]
    int64_t sh, sp;
    float *d_hidden;                                   // [H] in: dOut, out: dR1 (single call)
    const float *dout;                                 // [H] the layer's dOut (k1, k3)
    float *dhid_out;                                   // [H] receives dR1 (k4), or NULL
    float *dF, *dN2, *dR1, *dSub, *dctx;               // workspace vectors
    float *Upart, *Wpart, *Dpart, *dqpre, *dv, *gh;    // workspace attention / LoRA
    tlb_lora lq, lv;
    AdamCoef ka, kb;
    double *sumsq;
    const uint32_t *status;   // status block (optional): its step gate set skips AdamW (k7)
    float *Dout;              // [nh] (optional): k6 writes each head's D = sum_j attn dAttn
    // per-block partial sums (sum dy g x, sum x^2) for the RMSNorm backward of the
    // vector each GEMV produces; n1..n3 = the GEMV grids (blocks of k1, k2, k3)
    float2 *part1, *part2, *part3;
    int n1, n2, n3;
    int ns2, ns3;   // column ranges (blocks per row block) of the W_gate | W_up and W_O GEMVs
};

// Weight elements per 16-byte chunk of a row.
template <int WT>
struct EPC {
    static constexpr int v = WT == TLB_W_F32 ? 4 : (WT == TLB_W_BF16 ? 8 : (WT == TLB_W_TERNARY_I8 ? 16 : 64));
};

// Bytes of n weights of a row (n a multiple of 4 for the packed ternary type).
template <int WT>
__host__ __device__ constexpr size_t wbytes(size_t n) {
    return n * 16 / EPC<WT>::v;
}

template <int WT>
__device__ __forceinline__ float chunk_dot(uint4 w, const float *x) {
    if constexpr (WT == TLB_W_F32) {
        return __uint_as_float(w.x) * x[0] + __uint_as_float(w.y) * x[1] + __uint_as_float(w.z) * x[2] +
               __uint_as_float(w.w) * x[3];
    } else if constexpr (WT == TLB_W_BF16) {
        const uint32_t q[4] = {w.x, w.y, w.z, w.w};
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) s += bf16_lo(q[i]) * x[2 * i] + bf16_hi(q[i]) * x[2 * i + 1];
        return s;
    } else {
        const uint32_t q[4] = {w.x, w.y, w.z, w.w};
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float a, b, c, d;
            i8x4_to_f32(q[i], a, b, c, d);
            s0 = fmaf(a, x[4 * i], s0);
            s1 = fmaf(b, x[4 * i + 1], s1);
            s0 = fmaf(c, x[4 * i + 2], s0);
            s1 = fmaf(d, x[4 * i + 3], s1);
        }
        return s0 + s1;
    }
}

// Shared-memory position of float4 unit u of a GEMV vector: lane l reads chunk
// ch = base + l, i.e. units ch*P .. ch*P + P - 1 (P = float4 units per 16-byte weight
// chunk); XOR-ing the unit index within its chunk with bits of ch puts the 8 lanes of
// each 128-byte shared-memory phase on 8 different 16-byte bank groups.
template <int WT>
__device__ __forceinline__ int xunit(int u) {
    constexpr int P = EPC<WT>::v / 4;
    if constexpr (P == 1) {
        return u;
    } else if constexpr (P < 8) {
        const int ch = u / P, k = u % P;
        return ch * P + (k ^ ((ch / (8 / P)) % P));
    } else {
        const int ch = u / P, k = u % P;     // a chunk spans the 8 bank groups twice or more
        return ch * P + (k ^ (ch & 7));
    }
}


constexpr int kDecodeChunk = 32;   // keys per block in the attention pass

bool decode_supported(const tlb_layer_cfg &c, int64_t S, int64_t L);

// Persistent single-kernel version (decode_persistent.cu).  Its workspace needs, besides
// the DecodeArgs regions, a zero-initialised grid-barrier word pair (off_gbar) and
// 3 * kMaxPersistentBlocks float2 partial sums (off_pp).
constexpr int kMaxPersistentBlocks = 1024;
bool persistent_supported(const tlb_layer_cfg &c, int64_t S, int64_t L);
int decode_persistent_launch(const DecodeArgs &d, const tlb_layer_cfg &c, int64_t L, void *ws, size_t off_gbar,
                             size_t off_pp, cudaStream_t st);
int decode_rows_per_block();
int decode_layer_launch(const DecodeArgs &a, int wtype, cudaStream_t st);
// The two halves of the chain: k1 .. k3 (dF, dN2, dR1 and dSub) and k4 .. k7 (attention,
// dQpre, LoRA and AdamW), for callers that overlap one layer's second half with the next
// layer's first half on another stream.
// k1_pdl: launch k1 as a programmatic dependent of the kernel before it on `st` (it
// prefetches its weights into L2, then waits for that kernel).
int decode_ffn_launch(const DecodeArgs &a, int wtype, cudaStream_t st, bool k1_pdl);
// k4, k6 and (with_k7) k7; without it k7 comes later through decode_lora_launch.
int decode_attn_launch(const DecodeArgs &a, cudaStream_t st, bool with_k7 = true);
int decode_lora_launch(const DecodeArgs &a, cudaStream_t st);

}  // namespace tlb
