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
//   k4  per (KV head, key chunk): dCtx of the group's heads (sub-norm backward),
//       dAttn[h, j] = dCtx_h . V[j], partial sums of attn * dAttn
//   k5  per (KV head, key chunk): D_h, dS = scale attn (dAttn - D_h),
//       partial dQ_h = sum_j dS[h, j] K[j]
//   k6  per head: dQ = sum of partials, RoPE backward -> dQpre, gh_q += s dQpre_h B_q;
//       per KV head: dV = sum_group attn[h, pos] dCtx_h, gh_v += s dV B_v
//   k7  dB = s G h^T and dA = gh x^T for both adapters, AdamW (LoRA+ on B)
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

template <int WT>
__global__ void __launch_bounds__(kThreads) dec_k1(DecodeArgs a) {
    extern __shared__ float4 sm4[];
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

// ------------------------------------------------------------------ k4: dCtx, dAttn, partial D

__global__ void __launch_bounds__(kThreads) dec_k4(DecodeArgs a) {
    extern __shared__ float4 sm4[];
    __shared__ float2 red[32];
    __shared__ float sD[kWarps][16];
    const int kvh = blockIdx.x, chunk = blockIdx.y;
    const int G = a.nh / a.nkv;
    float *sC = reinterpret_cast<float *>(sm4);          // [G * hd]
    float rinv = 1.f, c = 0.f;
    const bool sub = a.flags & TLB_SUB_NORM;
    if (sub) {
        const float2 s = rms_sums(a.ctx, a.g_sub_attn, a.dSub, a.qd, red);
        const float ms = s.x / float(a.qd) + a.eps;
        rinv = rsqrtf(ms);
        c = s.y / float(a.qd) / ms;
    }
    const int off = kvh * G * a.hd;
    for (int i = threadIdx.x; i < G * a.hd; i += blockDim.x) {
        const int q = off + i;
        const float ds = a.dSub[q];
        const float v = sub ? rinv * (ds * a.g_sub_attn[q] - a.ctx[q] * c) : ds;
        sC[i] = v;
        if (chunk == 0) a.dctx[q] = v;
    }
    if (kvh == 0 && chunk == 0)
        for (int i = threadIdx.x; i < a.H; i += blockDim.x) a.d_hidden[i] = a.dR1[i];
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float dpart[16];
#pragma unroll
    for (int g = 0; g < 16; ++g) dpart[g] = 0.f;
    const int j0 = chunk * a.chunk;
    const int j1 = min(a.L, j0 + a.chunk);
    for (int j = j0 + warp; j < j1; j += kWarps) {
        const float *vr = a.v + int64_t(kvh) * a.sh + int64_t(j) * a.sp;
        float dots[16];
#pragma unroll
        for (int g = 0; g < 16; ++g) dots[g] = 0.f;
        for (int d = lane; d < a.hd; d += 32) {
            const float vv = vr[d];
#pragma unroll
            for (int g = 0; g < 16; ++g)
                if (g < G) dots[g] = fmaf(sC[g * a.hd + d], vv, dots[g]);
        }
#pragma unroll
        for (int g = 0; g < 16; ++g) {
            if (g < G) {
                const float t = warp_sum(dots[g]);
                const int h = kvh * G + g;
                if (lane == 0) {
                    a.dattn[int64_t(h) * a.L + j] = t;
                    dpart[g] += a.attn[int64_t(h) * a.L + j] * t;
                }
            }
        }
    }
    if (lane == 0)
#pragma unroll
        for (int g = 0; g < 16; ++g) sD[warp][g] = dpart[g];
    __syncthreads();
    if (threadIdx.x < G) {
        float s = 0.f;
        for (int w = 0; w < kWarps; ++w) s += sD[w][threadIdx.x];
        a.Dpart[int64_t(chunk) * a.nh + kvh * G + threadIdx.x] = s;
    }
}

// ------------------------------------------------------------------ k5: dS, partial dQ

__global__ void __launch_bounds__(kThreads) dec_k5(DecodeArgs a) {
    extern __shared__ float4 sm4[];
    const int kvh = blockIdx.x, chunk = blockIdx.y;
    const int G = a.nh / a.nkv;
    const int j0 = chunk * a.chunk;
    const int n = min(a.L, j0 + a.chunk) - j0;
    float *sS = reinterpret_cast<float *>(sm4);         // [G][chunk]
    __shared__ float sDh[16];
    if (threadIdx.x < G) {
        float s = 0.f;
        for (int c = 0; c < a.nchunks; ++c) s += a.Dpart[int64_t(c) * a.nh + kvh * G + threadIdx.x];
        sDh[threadIdx.x] = s;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < G * n; i += blockDim.x) {
        const int g = i / n, jj = i % n;
        const int64_t idx = int64_t(kvh * G + g) * a.L + j0 + jj;
        sS[g * a.chunk + jj] = a.scale * a.attn[idx] * (a.dattn[idx] - sDh[g]);
    }
    __syncthreads();
    for (int o = threadIdx.x; o < G * a.hd; o += blockDim.x) {
        const int g = o / a.hd, d = o % a.hd;
        const float *kc = a.k + int64_t(kvh) * a.sh + int64_t(j0) * a.sp + d;
        float acc = 0.f;
        for (int jj = 0; jj < n; ++jj) acc = fmaf(sS[g * a.chunk + jj], kc[int64_t(jj) * a.sp], acc);
        a.dqpart[(int64_t(chunk) * a.nh + kvh * G + g) * a.hd + d] = acc;
    }
}

// ------------------------------------------------------------------ k6: dQpre, dV, LoRA gh

__global__ void __launch_bounds__(kThreads) dec_k6(DecodeArgs a, RopeFreqs fr) {
    __shared__ float sv[256];
    __shared__ float red[16][kWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int b = blockIdx.x;
    float *G;          // gradient row slice this block produces
    const float *B;    // adapter B rows matching the slice
    float *gh;
    int o0;
    if (b < a.nh) {                      // head b: dQ, RoPE backward
        const int h = b;
        for (int d = threadIdx.x; d < a.hd; d += blockDim.x) {
            float s = 0.f;
            for (int c = 0; c < a.nchunks; ++c) s += a.dqpart[(int64_t(c) * a.nh + h) * a.hd + d];
            sv[d] = s;
        }
        __syncthreads();
        const int half = a.hd >> 1;
        for (int d = threadIdx.x; d < half; d += blockDim.x) {
            float y1 = sv[d], y2 = sv[d + half];
            if (a.flags & TLB_ROPE) {
                float cs, sn;
                rope_cos_sin(float(a.pos), fr.hi[d], fr.lo[d], cs, sn);
                const float t1 = y1 * cs + y2 * sn, t2 = -y1 * sn + y2 * cs;
                y1 = t1;
                y2 = t2;
            }
            a.dqpre[h * a.hd + d] = y1;
            a.dqpre[h * a.hd + d + half] = y2;
        }
        __syncthreads();
        G = a.dqpre;
        B = a.lq.b;
        gh = a.gh;
        o0 = h * a.hd;
    } else {                             // KV head: dV of the current token
        const int kvh = b - a.nh;
        const int grp = a.nh / a.nkv;
        for (int d = threadIdx.x; d < a.hd; d += blockDim.x) {
            float s = 0.f;
            for (int g = 0; g < grp; ++g) {
                const int h = kvh * grp + g;
                s = fmaf(a.attn[int64_t(h) * a.L + a.pos], a.dctx[h * a.hd + d], s);
            }
            a.dv[kvh * a.hd + d] = s;
        }
        __syncthreads();
        G = a.dv;
        B = a.lv.b;
        gh = a.gh + a.rank;
        o0 = kvh * a.hd;
    }
    // gh[r] += s * sum_{o in slice} G[o] B[o, r]  (B before its update)
    float acc[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) acc[r] = 0.f;
    for (int o = threadIdx.x; o < a.hd; o += blockDim.x) {
        const float gv = G[o0 + o];
        const float *br = B + int64_t(o0 + o) * a.rank;
#pragma unroll
        for (int r = 0; r < 16; ++r)
            if (r < a.rank) acc[r] = fmaf(gv, br[r], acc[r]);
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        const float t = warp_sum(acc[r]);
        if (lane == 0) red[r][warp] = t;
    }
    __syncthreads();
    if (threadIdx.x < a.rank) {
        float s = 0.f;
        for (int w = 0; w < kWarps; ++w) s += red[threadIdx.x][w];
        atomicAdd(gh + threadIdx.x, a.lora_scaling * s);
    }
}

// ------------------------------------------------------------------ k7: LoRA gradients + AdamW

__global__ void __launch_bounds__(kThreads) dec_k7(DecodeArgs a) {
    __shared__ float red[32];
    const int64_t nbq = int64_t(a.qd) * a.rank, nbv = int64_t(a.kvd) * a.rank, na = int64_t(a.rank) * a.H;
    const int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
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

template <int WT>
int launch_all(const DecodeArgs &a, cudaStream_t st) {
    const size_t sm1 = size_t(a.H) * 4, sm2 = size_t(2) * a.I * 4, sm3 = size_t(a.H) * 4;
    const int rows_per_block = kWarps * kR;
    auto big = [](const void *f, size_t s) -> cudaError_t {
        return s > 48 * 1024 ? cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, int(s))
                             : cudaSuccess;
    };
    TLB_CUDA(big((const void *)dec_k1<WT>, sm1));
    dec_k1<WT><<<unsigned(ceil_div(a.I, rows_per_block)), kThreads, sm1, st>>>(a);
    TLB_TRY(check_launch("decode k1"));
    if (a.act == TLB_ACT_RELU2_MUL) {
        TLB_CUDA(big((const void *)dec_k2<WT, TLB_ACT_RELU2_MUL>, sm2));
        dec_k2<WT, TLB_ACT_RELU2_MUL><<<unsigned(ceil_div(a.H, rows_per_block)), kThreads, sm2, st>>>(a);
    } else {
        TLB_CUDA(big((const void *)dec_k2<WT, TLB_ACT_SILU_MUL>, sm2));
        dec_k2<WT, TLB_ACT_SILU_MUL><<<unsigned(ceil_div(a.H, rows_per_block)), kThreads, sm2, st>>>(a);
    }
    TLB_TRY(check_launch("decode k2"));
    TLB_CUDA(big((const void *)dec_k3<WT>, sm3));
    dec_k3<WT><<<unsigned(ceil_div(a.qd, rows_per_block)), kThreads, sm3, st>>>(a);
    TLB_TRY(check_launch("decode k3"));
    const int G = a.nh / a.nkv;
    dec_k4<<<dim3(a.nkv, a.nchunks), kThreads, size_t(G) * a.hd * 4, st>>>(a);
    TLB_TRY(check_launch("decode k4"));
    dec_k5<<<dim3(a.nkv, a.nchunks), kThreads, size_t(G) * a.chunk * 4, st>>>(a);
    TLB_TRY(check_launch("decode k5"));
    RopeFreqs fr;
    rope_freqs(fr, a.hd, a.rope_base);
    dec_k6<<<a.nh + a.nkv, kThreads, 0, st>>>(a, fr);
    TLB_TRY(check_launch("decode k6"));
    const int64_t n7 = int64_t(a.qd + a.kvd) * a.rank + 2 * int64_t(a.rank) * a.H;
    dec_k7<<<unsigned(ceil_div(n7, kThreads)), kThreads, 0, st>>>(a);
    return check_launch("decode k7");
}

}  // namespace

bool decode_supported(const tlb_layer_cfg &c, int64_t S, int64_t L) {
    const int G = c.n_heads / c.n_kv_heads;
    const int E = c.wtype == TLB_W_F32 ? 4 : (c.wtype == TLB_W_BF16 ? 8 : 16);
    return S == 1 && G <= 16 && c.rank <= 16 && c.head_dim <= 256 && c.dim % E == 0 && c.ffn_dim % E == 0 &&
           size_t(2) * c.ffn_dim * 4 <= 200 * 1024 && L >= 1;
}

int decode_layer_launch(const DecodeArgs &a, int wtype, cudaStream_t st) {
    switch (wtype) {
        case TLB_W_F32: return launch_all<TLB_W_F32>(a, st);
        case TLB_W_BF16: return launch_all<TLB_W_BF16>(a, st);
        default: return launch_all<TLB_W_TERNARY_I8>(a, st);
    }
}

}  // namespace tlb
