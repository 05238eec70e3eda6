// Single-token (decode) layer backward: the whole layer in seven bandwidth-bound
// kernels ([FFN] executeFFNBackward chain; [ATT] "Gradient Flow"; [RS] LoRA blocks
// and cpu_adamw).  Every weight byte, cache entry and adapter parameter is read
// from HBM once; the small vectors between the steps stay in L2.
//
//   k1  dF   = s_d W_down dOut                                   GEMV over I rows
//   k2  dG, dU from dF (sub-norm RMSNorm backward + gated activation backward,
//       recomputed per block in shared memory), then
//       dN2  = s_g W_gate dG + s_u W_up dU                        GEMV over H rows
//   k3  dR1  = dOut + RMSNorm_bwd(r1, g_ffn, dN2) (per block, shared memory), then
//       dSub = s_o W_O dR1                                        GEMV over q_dim rows
//   k4  per (KV head, key chunk), one pass over K and V: dCtx of the group's heads
//       (sub-norm backward), dA = dCtx_h . V[j] and the partial sums
//       U_h = sum P dA K[j], W_h = sum P K[j], D_h = sum P dA; the chunk holding the
//       current position also forms dV = sum_group attn[h, pos] dCtx_h and gh_v
//   k6  per head: dQ = scale (U - D W) over all chunks ([ATT] softmax + score
//       backward), RoPE backward -> dQpre, gh_q += s dQpre_h B_q
//   k7  dB = s G h^T and dA = gh x^T for both adapters, AdamW (LoRA+ on B)
//
// k1 also issues L2 bulk prefetches of everything the later kernels read (weights of
// k2/k3, K, V, attention rows, adapter state), so HBM streams the whole step while
// the dependent chain runs; k2..k7 are launched as programmatic dependents.
#include "common.cuh"
#include "kernels.cuh"
#include "decode.cuh"

namespace tlb {

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

template <int WT>
struct EPC {
    static constexpr int v = WT == TLB_W_F32 ? 4 : (WT == TLB_W_BF16 ? 8 : 16);
};

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

// Rows [r0, r0 + R) of NM matrices (same shape [rows, cols]), each dotted with its own
// shared-memory vector, scaled and summed: y[r] = sum_m scale_m W_m[r, :] . x_m.
// One warp; U chunks of 16 bytes per row and matrix in flight per lane.
template <int WT, int NM, int R, int U>
__device__ __forceinline__ void warp_rows(const char *const *W, const float *scale, const float *const *xs,
                                          int r0, int rows, int cols, float *y) {
    constexpr int E = EPC<WT>::v;
    const int lane = threadIdx.x & 31;
    const int nch = cols / E;
    const size_t row_bytes = size_t(cols) * (16 / E);
    float acc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r] = 0.f;
    for (int base = 0; base < nch; base += 32 * U) {
        uint4 w[NM][R][U];
#pragma unroll
        for (int m = 0; m < NM; ++m)
#pragma unroll
            for (int r = 0; r < R; ++r)
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int ch = base + u * 32 + lane;
                    w[m][r][u] = (ch < nch && r0 + r < rows)
                                     ? ld_stream_u4(W[m] + size_t(r0 + r) * row_bytes + size_t(ch) * 16)
                                     : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int ch = base + u * 32 + lane;
            if (ch >= nch) break;
#pragma unroll
            for (int m = 0; m < NM; ++m) {
                float xv[E];
#pragma unroll
                for (int e = 0; e < E; e += 4) {
                    const float4 t = *reinterpret_cast<const float4 *>(xs[m] + ch * E + e);
                    xv[e] = t.x;
                    xv[e + 1] = t.y;
                    xv[e + 2] = t.z;
                    xv[e + 3] = t.w;
                }
#pragma unroll
                for (int r = 0; r < R; ++r) acc[r] = fmaf(scale[m], chunk_dot<WT>(w[m][r][u], xv), acc[r]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const float s = warp_sum(acc[r]);
        if (lane == 0 && r0 + r < rows) y[r0 + r] = s;
    }
}

constexpr int kR = 2, kU = 2;   // rows per warp, chunks in flight per row

// Sum of x^2 and of x * g * dy over n elements (block-wide).
__device__ __forceinline__ float2 rms_sums(const float *x, const float *g, const float *dy, int n, float2 *red) {
    float2 acc = make_float2(0.f, 0.f);
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const float xv = x[i];
        acc.x += xv * xv;
        acc.y += xv * g[i] * dy[i];
    }
    return block_sum2(acc, red);
}

// ------------------------------------------------------------------ k1: dF = s_d W_down dOut

// This block's share of the L2 prefetch list (16-byte aligned pieces of <= 32 KiB).
__device__ void prefetch_share(const DecodeArgs &a, int part, int nparts) {
    const uint64_t b0 = a.pf_total * part / nparts, b1 = a.pf_total * (part + 1) / nparts;
    uint64_t base = 0;
    for (int r = 0; r < a.pf_count; ++r) {
        const uint64_t n = a.pf_bytes[r];
        const uint64_t s = b0 > base ? b0 : base, e = b1 < base + n ? b1 : base + n;
        if (s < e) {
            const uint64_t o0 = (s - base + 15) & ~uint64_t(15), o1 = (e - base) & ~uint64_t(15);
            for (uint64_t o = o0; o < o1; o += 32768) {
                const uint64_t len = o1 - o < 32768 ? o1 - o : 32768;
                l2_prefetch(a.pf_ptr[r] + o, uint32_t(len));
            }
        }
        base += n;
    }
}

template <int WT>
__global__ void __launch_bounds__(kThreads) dec_k1(DecodeArgs a) {
    extern __shared__ float4 sm4[];
    pdl_trigger();
    if (threadIdx.x == 0) prefetch_share(a, blockIdx.x, gridDim.x);
    float *sx = reinterpret_cast<float *>(sm4);
    for (int i = threadIdx.x; i < a.H; i += blockDim.x) sx[i] = a.d_hidden[i];
    if (blockIdx.x == 0 && threadIdx.x < 2 * a.rank) a.gh[threadIdx.x] = 0.f;
    __syncthreads();
    const char *W[1] = {reinterpret_cast<const char *>(a.w_down)};
    const float sc[1] = {a.s_down};
    const float *xs[1] = {sx};
    const int r0 = (blockIdx.x * kWarps + (threadIdx.x >> 5)) * kR;
    if (r0 < a.I) warp_rows<WT, 1, kR, kU>(W, sc, xs, r0, a.I, a.H, a.dF);
}

// ------------------------------------------------------------------ k2: dN2 = W_g dG + W_u dU

template <int WT, int ACT>
__global__ void __launch_bounds__(kThreads) dec_k2(DecodeArgs a) {
    extern __shared__ float4 sm4[];
    __shared__ float2 red[32];
    float *sG = reinterpret_cast<float *>(sm4);
    float *sU = sG + a.I;
    pdl_trigger();
    pdl_wait();
    float rinv = 1.f, c = 0.f;
    const bool sub = a.flags & TLB_SUB_NORM;
    if (sub) {
        const float2 s = rms_sums(a.hidden, a.g_sub_ffn, a.dF, a.I, red);
        const float ms = s.x / float(a.I) + a.eps;
        rinv = rsqrtf(ms);
        c = s.y / float(a.I) / ms;
    }
    const bool cache = (ACT == TLB_ACT_SILU_MUL) && (a.flags & TLB_USE_SILU_CACHE);
    for (int i = threadIdx.x; i < a.I; i += blockDim.x) {
        const float df = a.dF[i];
        const float dh = sub ? rinv * (df * a.g_sub_ffn[i] - a.hidden[i] * c) : df;
        const float g = a.gate[i], u = a.up[i];
        if constexpr (ACT == TLB_ACT_RELU2_MUL) {
            const float r = fmaxf(g, 0.f);
            sG[i] = dh * u * 2.f * r;
            sU[i] = dh * r * r;
        } else {
            const float sig = 1.f / (1.f + expf(-g));
            const float y = g * sig;
            sG[i] = dh * u * (sig * (1.f + g - y));
            sU[i] = dh * (cache ? a.silu_gate[i] : y);
        }
    }
    __syncthreads();
    const char *W[2] = {reinterpret_cast<const char *>(a.w_gate), reinterpret_cast<const char *>(a.w_up)};
    const float sc[2] = {a.s_gate, a.s_up};
    const float *xs[2] = {sG, sU};
    const int r0 = (blockIdx.x * kWarps + (threadIdx.x >> 5)) * kR;
    if (r0 < a.H) warp_rows<WT, 2, kR, kU>(W, sc, xs, r0, a.H, a.I, a.dN2);
}

// ------------------------------------------------------------------ k3: dR1, dSub = s_o W_O dR1

template <int WT>
__global__ void __launch_bounds__(kThreads) dec_k3(DecodeArgs a) {
    extern __shared__ float4 sm4[];
    __shared__ float2 red[32];
    float *sR = reinterpret_cast<float *>(sm4);
    pdl_trigger();
    pdl_wait();
    float rinv = 1.f, c = 0.f;
    const bool pre = a.flags & TLB_PRE_NORM;
    if (pre) {
        const float2 s = rms_sums(a.r1, a.g_ffn, a.dN2, a.H, red);
        const float ms = s.x / float(a.H) + a.eps;
        rinv = rsqrtf(ms);
        c = s.y / float(a.H) / ms;
    }
    const bool resid = a.flags & TLB_RESIDUAL;
    for (int i = threadIdx.x; i < a.H; i += blockDim.x) {
        const float dn = a.dN2[i];
        float v = pre ? rinv * (dn * a.g_ffn[i] - a.r1[i] * c) : dn;
        if (resid) v += a.d_hidden[i];
        sR[i] = v;
        if (blockIdx.x == 0) a.dR1[i] = v;
    }
    __syncthreads();
    const char *W[1] = {reinterpret_cast<const char *>(a.w_o)};
    const float sc[1] = {a.s_o};
    const float *xs[1] = {sR};
    const int r0 = (blockIdx.x * kWarps + (threadIdx.x >> 5)) * kR;
    if (r0 < a.qd) warp_rows<WT, 1, kR, kU>(W, sc, xs, r0, a.qd, a.H, a.dSub);
}

// ------------------------------------------------------------------ k4: attention, one pass over K and V

// Per (KV head, chunk of keys): dCtx of the group's heads (sub-norm backward), then for
// every key j of the chunk and head h of the group
//   dA = dCtx_h . V[j]      U_h += P dA K[j]      W_h += P K[j]      D_h += P dA
// so that dQ_h = scale (U_h - D_h W_h) summed over chunks equals
// scale sum_j P (dA - D_h) K[j] without a barrier on the row sum D_h.
// The chunk holding the current position also forms dV and its LoRA gh_v share.
template <int VPL, int GM>
__global__ void __launch_bounds__(kThreads) dec_k4(DecodeArgs a) {
    constexpr int KPW = kDecodeChunk / kWarps;        // keys per warp
    extern __shared__ float4 sm4[];
    __shared__ float2 red2[32];
    __shared__ float sDp[kWarps][16];
    const int kvh = blockIdx.x, chunk = blockIdx.y;
    const int G = a.nh / a.nkv;
    const int hd = VPL * 32;
    float *sC = reinterpret_cast<float *>(sm4);        // [G][hd] dCtx
    float *sR = sC + G * hd;                           // [kWarps][G][2][hd] reduction
    pdl_trigger();
    pdl_wait();
    float rinv = 1.f, c = 0.f;
    const bool sub = a.flags & TLB_SUB_NORM;
    if (sub) {
        const float2 s = rms_sums(a.ctx, a.g_sub_attn, a.dSub, a.qd, red2);
        const float ms = s.x / float(a.qd) + a.eps;
        rinv = rsqrtf(ms);
        c = s.y / float(a.qd) / ms;
    }
    const int off = kvh * G * hd;
    for (int i = threadIdx.x; i < G * hd; i += blockDim.x) {
        const int q = off + i;
        const float ds = a.dSub[q];
        sC[i] = sub ? rinv * (ds * a.g_sub_attn[q] - a.ctx[q] * c) : ds;
    }
    if (kvh == 0 && chunk == 0)
        for (int i = threadIdx.x; i < a.H; i += blockDim.x) a.d_hidden[i] = a.dR1[i];
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int d0 = lane * VPL;
    float U[GM][VPL], W[GM][VPL];                      // GM >= heads per KV group
#pragma unroll
    for (int g = 0; g < GM; ++g)
#pragma unroll
        for (int v = 0; v < VPL; ++v) U[g][v] = W[g][v] = 0.f;
    float dsum[GM];
#pragma unroll
    for (int g = 0; g < GM; ++g) dsum[g] = 0.f;
    const int jw = chunk * kDecodeChunk + warp * KPW;
#pragma unroll
    for (int k = 0; k < KPW; ++k) {
        const int j = jw + k;
        if (j >= a.L) break;
        float kv[VPL], vv[VPL];
        const float *kr = a.k + int64_t(kvh) * a.sh + int64_t(j) * a.sp + d0;
        const float *vr = a.v + int64_t(kvh) * a.sh + int64_t(j) * a.sp + d0;
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
            kv[v] = kr[v];
            vv[v] = vr[v];
        }
        // P of this key for each head of the group (lanes load in parallel)
        const float pl = lane < G ? a.attn[int64_t(kvh * G + lane) * a.L + j] : 0.f;
#pragma unroll
        for (int g = 0; g < GM; ++g) {
            if (g >= G) break;
            float t = 0.f;
#pragma unroll
            for (int v = 0; v < VPL; ++v) t = fmaf(sC[g * hd + d0 + v], vv[v], t);
            const float dA = warp_sum(t);
            const float P = __shfl_sync(0xffffffffu, pl, g);
            const float pd = P * dA;
            dsum[g] += pd;
#pragma unroll
            for (int v = 0; v < VPL; ++v) {
                U[g][v] = fmaf(pd, kv[v], U[g][v]);
                W[g][v] = fmaf(P, kv[v], W[g][v]);
            }
        }
    }
#pragma unroll
    for (int g = 0; g < GM; ++g) {
        if (g >= G) break;
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
            sR[((warp * G + g) * 2 + 0) * hd + d0 + v] = U[g][v];
            sR[((warp * G + g) * 2 + 1) * hd + d0 + v] = W[g][v];
        }
        if (lane == 0) sDp[warp][g] = dsum[g];
    }
    __syncthreads();
    for (int i = threadIdx.x; i < G * 2 * hd; i += blockDim.x) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) t += sR[w * G * 2 * hd + i];
        const int g = i / (2 * hd), which = (i / hd) & 1, d = i % hd;
        float *dst = which ? a.Wpart : a.Upart;
        dst[(int64_t(chunk) * a.nh + kvh * G + g) * hd + d] = t;
    }
    if (threadIdx.x < G) {
        float t = 0.f;
        for (int w = 0; w < kWarps; ++w) t += sDp[w][threadIdx.x];
        a.Dpart[int64_t(chunk) * a.nh + kvh * G + threadIdx.x] = t;
    }
    // dV of the current token: dV[kvh, d] = sum_g attn[h_g, pos] dCtx_h_g[d]; gh_v share
    if (a.pos / kDecodeChunk == chunk) {
        __shared__ float sv[256];
        __shared__ float rr[16][kWarps];
        for (int d = threadIdx.x; d < hd; d += blockDim.x) {
            float t = 0.f;
            for (int g = 0; g < G; ++g) t = fmaf(a.attn[int64_t(kvh * G + g) * a.L + a.pos], sC[g * hd + d], t);
            sv[d] = t;
            a.dv[kvh * hd + d] = t;
        }
        __syncthreads();
        float acc[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) acc[r] = 0.f;
        for (int d = threadIdx.x; d < hd; d += blockDim.x) {
            const float *br = a.lv.b + int64_t(kvh * hd + d) * a.rank;
#pragma unroll
            for (int r = 0; r < 16; ++r)
                if (r < a.rank) acc[r] = fmaf(sv[d], br[r], acc[r]);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const float t = warp_sum(acc[r]);
            if (lane == 0) rr[r][warp] = t;
        }
        __syncthreads();
        if (threadIdx.x < a.rank) {
            float t = 0.f;
            for (int w = 0; w < kWarps; ++w) t += rr[threadIdx.x][w];
            atomicAdd(a.gh + a.rank + threadIdx.x, a.lora_scaling * t);
        }
    }
}

// ------------------------------------------------------------------ k6: dQpre and gh_q per head

__global__ void __launch_bounds__(kThreads) dec_k6(DecodeArgs a, RopeFreqs fr) {
    __shared__ float sq[256];
    __shared__ float sD;
    __shared__ float red[16][kWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int h = blockIdx.x;
    pdl_trigger();
    pdl_wait();
    if (threadIdx.x < 32) {
        float t = 0.f;
        for (int c = lane; c < a.nchunks; c += 32) t += a.Dpart[int64_t(c) * a.nh + h];
        t = warp_sum(t);
        if (lane == 0) sD = t;
    }
    __syncthreads();
    const float D = sD;
    for (int d = threadIdx.x; d < a.hd; d += blockDim.x) {
        float u = 0.f, w = 0.f;
        for (int c = 0; c < a.nchunks; ++c) {
            const int64_t idx = (int64_t(c) * a.nh + h) * a.hd + d;
            u += a.Upart[idx];
            w += a.Wpart[idx];
        }
        sq[d] = a.scale * (u - D * w);
    }
    __syncthreads();
    const int half = a.hd >> 1;
    for (int d = threadIdx.x; d < half; d += blockDim.x) {
        float y1 = sq[d], y2 = sq[d + half];
        if (a.flags & TLB_ROPE) {
            float cs, sn;
            rope_cos_sin(float(a.pos), fr.hi[d], fr.lo[d], cs, sn);
            const float t1 = y1 * cs + y2 * sn, t2 = -y1 * sn + y2 * cs;
            y1 = t1;
            y2 = t2;
        }
        a.dqpre[h * a.hd + d] = y1;
        a.dqpre[h * a.hd + d + half] = y2;
        sq[d] = y1;
        sq[d + half] = y2;   // each pair is owned by one thread
    }
    __syncthreads();
    // gh_q[r] += s * sum_{d} dQpre[h, d] B_q[h*hd + d, r]   (B before its update)
    float acc[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) acc[r] = 0.f;
    for (int d = threadIdx.x; d < a.hd; d += blockDim.x) {
        const float *br = a.lq.b + int64_t(h * a.hd + d) * a.rank;
#pragma unroll
        for (int r = 0; r < 16; ++r)
            if (r < a.rank) acc[r] = fmaf(sq[d], br[r], acc[r]);
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        const float t = warp_sum(acc[r]);
        if (lane == 0) red[r][warp] = t;
    }
    __syncthreads();
    if (threadIdx.x < a.rank) {
        float t = 0.f;
        for (int w = 0; w < kWarps; ++w) t += red[threadIdx.x][w];
        atomicAdd(a.gh + threadIdx.x, a.lora_scaling * t);
    }
}

// ------------------------------------------------------------------ k7: LoRA gradients + AdamW

__global__ void __launch_bounds__(kThreads) dec_k7(DecodeArgs a) {
    __shared__ float red[32];
    const int64_t nbq = int64_t(a.qd) * a.rank, nbv = int64_t(a.kvd) * a.rank, na = int64_t(a.rank) * a.H;
    const int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    pdl_trigger();
    pdl_wait();
    float g = 0.f;
    int which = -1;   // 0: sumsq of dA, 1: of dB
    if (e < nbq) {
        const int o = int(e / a.rank), r = int(e % a.rank);
        g = a.lora_scaling * a.dqpre[o] * a.hq[r];
        if (a.lq.grad_b) a.lq.grad_b[e] = g;
        float m = a.lq.m_b[e], v = a.lq.v_b[e];
        a.lq.b[e] = adam_elem(a.lq.b[e], g, m, v, a.kb);
        a.lq.m_b[e] = m;
        a.lq.v_b[e] = v;
        which = 1;
    } else if (e < nbq + nbv) {
        const int64_t f = e - nbq;
        const int o = int(f / a.rank), r = int(f % a.rank);
        g = a.lora_scaling * a.dv[o] * a.hv[r];
        if (a.lv.grad_b) a.lv.grad_b[f] = g;
        float m = a.lv.m_b[f], v = a.lv.v_b[f];
        a.lv.b[f] = adam_elem(a.lv.b[f], g, m, v, a.kb);
        a.lv.m_b[f] = m;
        a.lv.v_b[f] = v;
        which = 1;
    } else if (e < nbq + nbv + 2 * na) {
        const int64_t f = e - nbq - nbv;
        const bool isq = f < na;
        const int64_t f2 = isq ? f : f - na;
        const int r = int(f2 / a.H), cidx = int(f2 % a.H);
        const tlb_lora &l = isq ? a.lq : a.lv;
        g = a.gh[(isq ? 0 : a.rank) + r] * a.x[cidx];
        if (l.grad_a) l.grad_a[f2] = g;
        float m = l.m_a[f2], v = l.v_a[f2];
        l.a[f2] = adam_elem(l.a[f2], g, m, v, a.ka);
        l.m_a[f2] = m;
        l.v_a[f2] = v;
        which = 0;
    }
    if (a.sumsq) {
        // blocks never straddle the dB / dA boundary when both counts are multiples of the
        // block size; otherwise the two sums are reduced separately
        const float sa = block_sum(which == 0 ? g * g : 0.f, red);
        const float sb = block_sum(which == 1 ? g * g : 0.f, red);
        if (threadIdx.x == 0) {
            if (sa != 0.f) atomicAdd(a.sumsq, double(sa));
            if (sb != 0.f) atomicAdd(a.sumsq + 1, double(sb));
        }
    }
}

template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, size_t smem, cudaStream_t st, bool pdl, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
    }
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <int VPL>
cudaError_t launch_k4_g(int G, dim3 g4, size_t sm4, cudaStream_t st, const DecodeArgs &a) {
    if (G <= 1) return launch(dec_k4<VPL, 1>, g4, sm4, st, true, a);
    if (G <= 2) return launch(dec_k4<VPL, 2>, g4, sm4, st, true, a);
    if (G <= 4) return launch(dec_k4<VPL, 4>, g4, sm4, st, true, a);
    if (G <= 8) return launch(dec_k4<VPL, 8>, g4, sm4, st, true, a);
    if constexpr (VPL <= 4) return launch(dec_k4<VPL, 16>, g4, sm4, st, true, a);
    return cudaErrorInvalidValue;
}

cudaError_t launch_k4(int G, int hd, dim3 g4, size_t sm4, cudaStream_t st, const DecodeArgs &a) {
    switch (hd) {
        case 32: return launch_k4_g<1>(G, g4, sm4, st, a);
        case 64: return launch_k4_g<2>(G, g4, sm4, st, a);
        case 128: return launch_k4_g<4>(G, g4, sm4, st, a);
        default: return launch_k4_g<8>(G, g4, sm4, st, a);
    }
}

template <int WT>
int launch_all(const DecodeArgs &a, cudaStream_t st) {
    const int rows_per_block = kWarps * kR;
    TLB_CUDA(launch(dec_k1<WT>, dim3(unsigned(ceil_div(a.I, rows_per_block))), size_t(a.H) * 4, st, false, a));
    TLB_TRY(check_launch("decode k1"));
    const size_t sm2 = size_t(2) * a.I * 4;
    const dim3 g2(unsigned(ceil_div(a.H, rows_per_block)));
    if (a.act == TLB_ACT_RELU2_MUL) TLB_CUDA(launch(dec_k2<WT, TLB_ACT_RELU2_MUL>, g2, sm2, st, true, a));
    else TLB_CUDA(launch(dec_k2<WT, TLB_ACT_SILU_MUL>, g2, sm2, st, true, a));
    TLB_TRY(check_launch("decode k2"));
    TLB_CUDA(launch(dec_k3<WT>, dim3(unsigned(ceil_div(a.qd, rows_per_block))), size_t(a.H) * 4, st, true, a));
    TLB_TRY(check_launch("decode k3"));
    const int G = a.nh / a.nkv;
    const dim3 g4(a.nkv, a.nchunks);
    const size_t sm4 = (size_t(G) * a.hd + size_t(kWarps) * G * 2 * a.hd) * 4;
    TLB_CUDA(launch_k4(G, a.hd, g4, sm4, st, a));
    TLB_TRY(check_launch("decode k4"));
    RopeFreqs fr;
    rope_freqs(fr, a.hd, a.rope_base);
    TLB_CUDA(launch(dec_k6, dim3(a.nh), 0, st, true, a, fr));
    TLB_TRY(check_launch("decode k6"));
    const int64_t n7 = int64_t(a.qd + a.kvd) * a.rank + 2 * int64_t(a.rank) * a.H;
    TLB_CUDA(launch(dec_k7, dim3(unsigned(ceil_div(n7, kThreads))), 0, st, true, a));
    return check_launch("decode k7");
}

}  // namespace

bool decode_supported(const tlb_layer_cfg &c, int64_t S, int64_t L) {
    const int G = c.n_heads / c.n_kv_heads;
    const int E = c.wtype == TLB_W_F32 ? 4 : (c.wtype == TLB_W_BF16 ? 8 : 16);
    const int hd = c.head_dim;
    const int gmax = hd > 128 ? 8 : 16;   // heads per KV group held in registers by k4
    const size_t sm4 = (size_t(G) * hd + size_t(kWarps) * G * 2 * hd) * 4;
    return S == 1 && G <= gmax && c.rank <= 16 && (hd == 32 || hd == 64 || hd == 128 || hd == 256) &&
           c.dim % E == 0 && c.ffn_dim % E == 0 && size_t(2) * c.ffn_dim * 4 <= 200 * 1024 &&
           sm4 <= 200 * 1024 && L >= 1;
}

int decode_layer_launch(const DecodeArgs &a, int wtype, cudaStream_t st) {
    switch (wtype) {
        case TLB_W_F32: return launch_all<TLB_W_F32>(a, st);
        case TLB_W_BF16: return launch_all<TLB_W_BF16>(a, st);
        default: return launch_all<TLB_W_TERNARY_I8>(a, st);
    }
}

}  // namespace tlb
