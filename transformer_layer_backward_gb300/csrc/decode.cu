// Single-token (decode) layer backward: the whole layer in seven bandwidth-bound
// kernels ([FFN] executeFFNBackward chain; [ATT] "Gradient Flow"; [RS] LoRA blocks
// and cpu_adamw).  Every weight byte, cache entry and adapter parameter is read
// from HBM once; the small vectors between the steps stay in L2.
//
//   k1  dF   = s_d W_down dOut                                   GEMV over I rows
//   k2  dG, dU from dF (sub-norm RMSNorm backward + gated activation backward), then
//       dN2  = s_g W_gate dG + s_u W_up dU                        GEMV over H rows
//       (int8, bf16 and fp32 weights: column-stationary, each thread's dG, dU values in
//       registers and the rows streamed past them; packed 2-bit weights: dG, dU
//       recomputed per block into a shared-memory vector)
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
// The vector a GEMV multiplies sits in shared memory in a swizzled order, so the
// 16-byte reads of the 32 lanes (each lane owning one 16-byte chunk of a weight row)
// fall in distinct banks.  The two sums an RMSNorm backward needs over a vector a
// GEMV produces are accumulated per block by that GEMV and summed by the consumer.
#include <algorithm>
#include <mutex>
#include <unordered_set>

#include "common.cuh"
#include "kernels.cuh"
#include "decode.cuh"

namespace tlb {

namespace {

constexpr int kWarps = 8;                // GEMV / LoRA kernels
constexpr int kThreads = kWarps * 32;
constexpr int kAWarps = 8;               // attention kernel (holds per-head accumulators)
constexpr int kAThreads = kAWarps * 32;
constexpr int kQWarps = 32;              // k6: thread groups over the chunk partials of one head
constexpr int kQThreads = kQWarps * 32;

// Rows [r0, r0 + R) of NM matrices (same shape [rows, cols]), each dotted with its own
// shared-memory vector (swizzled by xunit), scaled and summed:
//   y[r] = sum_m scale_m W_m[r, :] . x_m.
// One warp; U chunks of 16 bytes per row and matrix in flight per lane.  Returns the
// row values to every lane in out[R] (0 for rows past the end).
template <int WT, int NM, int R, int U, bool ATOMIC = false>
__device__ __forceinline__ void warp_rows(const char *const *W, const float *scale, const float *const *xs,
                                          int r0, int rows, int cols, float *y, float *out,
                                          size_t row_bytes = 0) {
    constexpr int E = EPC<WT>::v;
    constexpr int P = E / 4;
    const int lane = threadIdx.x & 31;
    const int nch = cols / E;
    if (row_bytes == 0) row_bytes = wbytes<WT>(size_t(cols));
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
            if constexpr (WT == TLB_W_TERNARY_2B) {
                // 64 packed weights per chunk: byte k of the chunk against float4 unit k;
                // sum w x = sum q x - sum x with the codes q = w + 1
#pragma unroll
                for (int m = 0; m < NM; ++m) {
                    float part[R], xsum = 0.f;
#pragma unroll
                    for (int r = 0; r < R; ++r) part[r] = 0.f;
#pragma unroll
                    for (int k = 0; k < P; ++k) {
                        const float4 t = reinterpret_cast<const float4 *>(xs[m])[xunit<WT>(ch * P + k)];
                        xsum += (t.x + t.y) + (t.z + t.w);
#pragma unroll
                        for (int r = 0; r < R; ++r) {
                            const uint4 &q = w[m][r][u];
                            const uint32_t word = k < 4 ? q.x : (k < 8 ? q.y : (k < 12 ? q.z : q.w));
                            part[r] += t2_qdot4(word >> (8 * (k & 3)), t);
                        }
                    }
#pragma unroll
                    for (int r = 0; r < R; ++r) acc[r] = fmaf(scale[m], part[r] - xsum, acc[r]);
                }
                continue;
            }
#pragma unroll
            for (int m = 0; m < NM; ++m) {
                float xv[E];
#pragma unroll
                for (int k = 0; k < P; ++k) {
                    const float4 t = reinterpret_cast<const float4 *>(xs[m])[xunit<WT>(ch * P + k)];
                    xv[4 * k] = t.x;
                    xv[4 * k + 1] = t.y;
                    xv[4 * k + 2] = t.z;
                    xv[4 * k + 3] = t.w;
                }
#pragma unroll
                for (int r = 0; r < R; ++r) acc[r] = fmaf(scale[m], chunk_dot<WT>(w[m][r][u], xv), acc[r]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const float s = warp_sum(acc[r]);
        out[r] = (r0 + r < rows) ? s : 0.f;
        if (lane == 0 && r0 + r < rows) {
            if constexpr (ATOMIC) atomicAdd(y + r0 + r, s);
            else y[r0 + r] = s;
        }
    }
}

// Copy n floats (n % 4 == 0) from global into shared memory in the GEMV order.
template <int WT>
__device__ __forceinline__ void stage_vector(float *sx, const float *x, int n) {
    const float4 *x4 = reinterpret_cast<const float4 *>(x);
    float4 *s4 = reinterpret_cast<float4 *>(sx);
    for (int u = threadIdx.x; u < (n >> 2); u += blockDim.x) s4[xunit<WT>(u)] = x4[u];
}

// Per-block partial sums (sum y g z, sum z^2) over this block's GEMV rows, written to
// part[blockIdx.x]; the consumer of y adds them up (RMSNorm backward of y with input z).
template <int R>
__device__ __forceinline__ void block_partials(const float *vals, int r0, int rows, const float *g,
                                               const float *z, float2 *part, float2 *red) {
    float2 acc = make_float2(0.f, 0.f);
    if ((threadIdx.x & 31) == 0) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (r0 + r < rows) {
                const float zz = z[r0 + r];
                acc.x += vals[r] * g[r0 + r] * zz;
                acc.y += zz * zz;
            }
        }
    }
    acc = block_sum2(acc, red);
    if (threadIdx.x == 0) part[blockIdx.x] = acc;
}

// Sum of the first n partials (every thread gets the result).
__device__ __forceinline__ float2 sum_partials(const float2 *part, int n, float2 *red) {
    float2 acc = make_float2(0.f, 0.f);
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const float2 p = part[i];
        acc.x += p.x;
        acc.y += p.y;
    }
    return block_sum2(acc, red);
}

// rinv and c of RMSNorm backward from (sum dy g x, sum x^2): dx = rinv (dy g - x c).
__device__ __forceinline__ void rms_coef2(float2 s, int n, float eps, float &rinv, float &c) {
    const float ms = s.y / float(n) + eps;
    rinv = rsqrtf(ms);
    c = s.x / float(n) / ms;
}

constexpr int kR = 2, kU = 2;   // rows per warp, chunks in flight per row and matrix

// L2 prefetch of [p, p + bytes) when both are 16-byte multiples (else nothing).  The
// kernels after k1 start early (programmatic dependent launch), prefetch the weights and
// caches they will read -- which depend on nothing the chain computes -- and only then
// wait for the previous kernel's results.
__device__ __forceinline__ void prefetch_l2(const void *p, size_t bytes) {
    if (bytes > 0 && bytes < (size_t(1) << 31) && ((reinterpret_cast<uintptr_t>(p) | bytes) & 15) == 0)
        l2_prefetch(p, uint32_t(bytes));
}

// ------------------------------------------------------------------ k1: dF = s_d W_down dOut

template <int WT>
__global__ void __launch_bounds__(kThreads) dec_k1(DecodeArgs a) {
    extern __shared__ float4 sm4[];
    __shared__ float2 red[32];
    float *sx = reinterpret_cast<float *>(sm4);
    {
        // this block's W_down rows, which depend on nothing before it, go to L2 first
        const int rows = kWarps * kR, r0 = blockIdx.x * rows;
        if (threadIdx.x == 0 && r0 < a.I)
            prefetch_l2(static_cast<const char *>(a.w_down) + wbytes<WT>(size_t(r0) * a.H),
                        wbytes<WT>(size_t(min(rows, a.I - r0)) * a.H));
    }
    pdl_trigger();
    pdl_wait();
    stage_vector<WT>(sx, a.dout, a.H);
    if (blockIdx.x == 0 && threadIdx.x < 2 * a.rank) a.gh[threadIdx.x] = 0.f;
    // dN2 and dSub are sums of per-block column-range products in k2 and k3
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < a.H + a.qd; i += gridDim.x * blockDim.x)
        (i < a.H ? a.dN2[i] : a.dSub[i - a.H]) = 0.f;
    __syncthreads();
    const char *W[1] = {reinterpret_cast<const char *>(a.w_down)};
    const float sc[1] = {a.s_down};
    const float *xs[1] = {sx};
    const int r0 = (blockIdx.x * kWarps + (threadIdx.x >> 5)) * kR;
    float vals[kR] = {};
    if (r0 < a.I) warp_rows<WT, 1, kR, kU>(W, sc, xs, r0, a.I, a.H, a.dF, vals);
    if (a.flags & TLB_SUB_NORM) block_partials<kR>(vals, r0, a.I, a.g_sub_ffn, a.hidden, a.part1, red);
}

// ------------------------------------------------------------------ k2: dN2 = W_g dG + W_u dU

template <int WT, int ACT>
__global__ void __launch_bounds__(kThreads) dec_k2(DecodeArgs a) {
    extern __shared__ float4 sm4[];
    __shared__ float2 red[32];
    // this block's column range [c0, c0 + nc) of dG, dU and of the W_gate / W_up rows
    const int nc = a.I / a.ns2, c0 = blockIdx.y * nc;
    float *sG = reinterpret_cast<float *>(sm4);
    float *sU = sG + nc;
    {
        const int lane = threadIdx.x & 31, r = (blockIdx.x * kWarps + (threadIdx.x >> 5)) * kR + (lane % kR);
        if (lane < 2 * kR && r < a.H)
            prefetch_l2(reinterpret_cast<const char *>(lane < kR ? a.w_gate : a.w_up) +
                            wbytes<WT>(size_t(r) * a.I + c0), wbytes<WT>(size_t(nc)));
    }
    pdl_trigger();
    pdl_wait();
    float rinv = 1.f, c = 0.f;
    const bool sub = a.flags & TLB_SUB_NORM;
    if (sub) rms_coef2(sum_partials(a.part1, a.n1, red), a.I, a.eps, rinv, c);
    const bool cache = (ACT == TLB_ACT_SILU_MUL) && (a.flags & TLB_USE_SILU_CACHE);
    {
        // dh (sub-norm backward) and the gated-activation backward, float4 at a time,
        // two float4 of each of the six inputs in flight per thread
        constexpr int B = 2;
        const int n4 = nc >> 2;
        const float4 *dF4 = reinterpret_cast<const float4 *>(a.dF + c0);
        const float4 *hid4 = reinterpret_cast<const float4 *>(a.hidden + c0);
        const float4 *gam4 = reinterpret_cast<const float4 *>(a.g_sub_ffn + c0);
        const float4 *gat4 = reinterpret_cast<const float4 *>(a.gate + c0);
        const float4 *up4 = reinterpret_cast<const float4 *>(a.up + c0);
        const float4 *sg4 = reinterpret_cast<const float4 *>(a.silu_gate + c0);
        for (int base = threadIdx.x; base < n4; base += blockDim.x * B) {
            float4 df[B], hd[B], gm[B], ga[B], uu[B], sl[B];
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const int i = base + b * blockDim.x;
                const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
                const bool ok = i < n4;
                df[b] = ok ? dF4[i] : z;
                hd[b] = ok && sub ? hid4[i] : z;
                gm[b] = ok && sub ? gam4[i] : z;
                ga[b] = ok ? gat4[i] : z;
                uu[b] = ok ? up4[i] : z;
                sl[b] = ok && cache ? sg4[i] : z;
            }
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const int i = base + b * blockDim.x;
                if (i >= n4) break;
                const float dfv[4] = {df[b].x, df[b].y, df[b].z, df[b].w};
                const float hdv[4] = {hd[b].x, hd[b].y, hd[b].z, hd[b].w};
                const float gmv[4] = {gm[b].x, gm[b].y, gm[b].z, gm[b].w};
                const float gav[4] = {ga[b].x, ga[b].y, ga[b].z, ga[b].w};
                const float uuv[4] = {uu[b].x, uu[b].y, uu[b].z, uu[b].w};
                const float slv[4] = {sl[b].x, sl[b].y, sl[b].z, sl[b].w};
                float og[4], ou[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float dh = sub ? rinv * (dfv[e] * gmv[e] - hdv[e] * c) : dfv[e];
                    const float g = gav[e], u = uuv[e];
                    if constexpr (ACT == TLB_ACT_RELU2_MUL) {
                        const float r = fmaxf(g, 0.f);
                        og[e] = dh * u * 2.f * r;
                        ou[e] = dh * r * r;
                    } else {
                        const float sig = 1.f / (1.f + expf(-g));
                        const float y = g * sig;
                        og[e] = dh * u * (sig * (1.f + g - y));
                        ou[e] = dh * (cache ? slv[e] : y);
                    }
                }
                reinterpret_cast<float4 *>(sG)[xunit<WT>(i)] = make_float4(og[0], og[1], og[2], og[3]);
                reinterpret_cast<float4 *>(sU)[xunit<WT>(i)] = make_float4(ou[0], ou[1], ou[2], ou[3]);
            }
        }
    }
    __syncthreads();
    const char *W[2] = {reinterpret_cast<const char *>(a.w_gate) + wbytes<WT>(size_t(c0)),
                        reinterpret_cast<const char *>(a.w_up) + wbytes<WT>(size_t(c0))};
    const float sc[2] = {a.s_gate, a.s_up};
    const float *xs[2] = {sG, sU};
    const int r0 = (blockIdx.x * kWarps + (threadIdx.x >> 5)) * kR;
    float vals[kR] = {};
    if (r0 < a.H) warp_rows<WT, 2, kR, kU, true>(W, sc, xs, r0, a.H, nc, a.dN2, vals, wbytes<WT>(size_t(a.I)));
}

// Column-stationary form of k2 (int8, bf16 and fp32 weights): each thread owns one
// 16-byte chunk of columns of both W_gate and W_up (E = 16 / 8 / 4 columns), forms its own
// dG and dU for those columns in registers (no shared-memory vector), and streams the
// block's rows kRowBatch at a time, double-buffered: a batch's two 16-byte loads per row
// are issued before the previous batch is dotted, and the first batch goes out before the
// wait on k1.  Each row's sum over the block's columns is reduced across the warp by
// halving exchanges, then across the warps in shared memory, and added into dN2 (the
// column blocks of a row meet there).
constexpr int kRowBatch = 4;

template <int WT, int ACT>
__global__ void __launch_bounds__(256, 2) dec_k2c(DecodeArgs a) {
    constexpr int E = EPC<WT>::v;
    extern __shared__ float red2[];            // [warps][rows of the block]
    __shared__ float2 red[32];
    const int nch = a.I / E;                   // 16-byte chunks per row
    const int ch = int(blockIdx.y) * blockDim.x + threadIdx.x;
    const bool col_ok = ch < nch;
    const int rows = a.H, r0 = int(int64_t(blockIdx.x) * rows / gridDim.x);
    const int r1 = int(int64_t(blockIdx.x + 1) * rows / gridDim.x), nr = r1 - r0;
    const size_t rb = wbytes<WT>(size_t(a.I));
    const char *wg = static_cast<const char *>(a.w_gate), *wu = static_cast<const char *>(a.w_up);
    {   // this block's rows of both matrices, over its column range, into L2 before the wait
        const int c0 = int(blockIdx.y) * blockDim.x, c1 = min(nch, c0 + int(blockDim.x));
        for (int k = threadIdx.x; k < 2 * nr; k += blockDim.x) {
            const char *base = (k & 1 ? wu : wg) + size_t(r0 + (k >> 1)) * rb + size_t(c0) * 16;
            prefetch_l2(base, size_t(c1 - c0) * 16);
        }
    }
    const char *pg = wg + size_t(ch) * 16, *pu = wu + size_t(ch) * 16;
    uint4 qg[2][kRowBatch], qu[2][kRowBatch];
    auto load = [&](int buf, int rr) {
#pragma unroll
        for (int k = 0; k < kRowBatch; ++k) {
            const bool ok = col_ok && rr + k < nr;
            const size_t off = size_t(r0 + rr + k) * rb;
            qg[buf][k] = ok ? ld_stream_u4(pg + off) : make_uint4(0, 0, 0, 0);
            qu[buf][k] = ok ? ld_stream_u4(pu + off) : make_uint4(0, 0, 0, 0);
        }
    };
    load(0, 0);                                // the weights depend on nothing before this kernel
    pdl_trigger();
    pdl_wait();
    float rinv = 1.f, c = 0.f;
    const bool sub = a.flags & TLB_SUB_NORM;
    if (sub) rms_coef2(sum_partials(a.part1, a.n1, red), a.I, a.eps, rinv, c);
    const bool cache = (ACT == TLB_ACT_SILU_MUL) && (a.flags & TLB_USE_SILU_CACHE);
    // dh (sub-norm backward) and the gated-activation backward of this thread's E columns
    float xg[E], xu[E];
    {
        constexpr int F = E / 4;
        const int j0 = col_ok ? ch * E : 0;
        float4 df[F], hd[F], gm[F], ga[F], uu[F], sl[F];
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int f = 0; f < F; ++f) {
            const int j = j0 + 4 * f;
            df[f] = col_ok ? *reinterpret_cast<const float4 *>(a.dF + j) : z;
            hd[f] = col_ok && sub ? *reinterpret_cast<const float4 *>(a.hidden + j) : z;
            gm[f] = col_ok && sub ? *reinterpret_cast<const float4 *>(a.g_sub_ffn + j) : z;
            ga[f] = col_ok ? *reinterpret_cast<const float4 *>(a.gate + j) : z;
            uu[f] = col_ok ? *reinterpret_cast<const float4 *>(a.up + j) : z;
            sl[f] = col_ok && cache ? *reinterpret_cast<const float4 *>(a.silu_gate + j) : z;
        }
#pragma unroll
        for (int f = 0; f < F; ++f) {
            const float dfv[4] = {df[f].x, df[f].y, df[f].z, df[f].w};
            const float hdv[4] = {hd[f].x, hd[f].y, hd[f].z, hd[f].w};
            const float gmv[4] = {gm[f].x, gm[f].y, gm[f].z, gm[f].w};
            const float gav[4] = {ga[f].x, ga[f].y, ga[f].z, ga[f].w};
            const float uuv[4] = {uu[f].x, uu[f].y, uu[f].z, uu[f].w};
            const float slv[4] = {sl[f].x, sl[f].y, sl[f].z, sl[f].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float dh = sub ? rinv * (dfv[e] * gmv[e] - hdv[e] * c) : dfv[e];
                const float g = gav[e], u = uuv[e];
                float og, ou;
                if constexpr (ACT == TLB_ACT_RELU2_MUL) {
                    const float r = fmaxf(g, 0.f);
                    og = dh * u * 2.f * r;
                    ou = dh * r * r;
                } else {
                    const float sig = 1.f / (1.f + expf(-g));
                    const float y = g * sig;
                    og = dh * u * (sig * (1.f + g - y));
                    ou = dh * (cache ? slv[e] : y);
                }
                xg[4 * f + e] = col_ok ? og : 0.f;
                xu[4 * f + e] = col_ok ? ou : 0.f;
            }
        }
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1;
    const int krow = 2 * b4 + b3;              // the batch row whose warp sum this lane ends with
    static_assert(kRowBatch == 4, "two halving levels");
    auto process = [&](int buf, int rr) {
        float v[kRowBatch];
#pragma unroll
        for (int k = 0; k < kRowBatch; ++k)
            v[k] = fmaf(a.s_gate, chunk_dot<WT>(qg[buf][k], xg), a.s_up * chunk_dot<WT>(qu[buf][k], xu));
        // sum over the warp's lanes: each level keeps half of the rows and adds the partner's
        float v2[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const float send = b4 ? v[i] : v[2 + i];
            v2[i] = (b4 ? v[2 + i] : v[i]) + __shfl_xor_sync(0xffffffffu, send, 16);
        }
        float v1 = (b3 ? v2[1] : v2[0]) + __shfl_xor_sync(0xffffffffu, b3 ? v2[0] : v2[1], 8);
        v1 += __shfl_xor_sync(0xffffffffu, v1, 4);
        v1 += __shfl_xor_sync(0xffffffffu, v1, 2);
        v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
        if ((lane & 7) == 0 && rr + krow < nr) red2[warp * nr + rr + krow] = v1;
    };
    // two batches per pass, so that the buffer of each load and dot is a constant
    for (int rr = 0; rr < nr; rr += 2 * kRowBatch) {
        if (rr + kRowBatch < nr) load(1, rr + kRowBatch);          // next batch in flight
        process(0, rr);
        if (rr + 2 * kRowBatch < nr) load(0, rr + 2 * kRowBatch);
        if (rr + kRowBatch < nr) process(1, rr + kRowBatch);
    }
    __syncthreads();
    for (int r = threadIdx.x; r < nr; r += blockDim.x) {
        float s = 0.f;
        for (int w = 0; w < nwarps; ++w) s += red2[w * nr + r];
        atomicAdd(a.dN2 + r0 + r, s);
    }
}

// ------------------------------------------------------------------ k3: dR1, dSub = s_o W_O dR1

template <int WT>
__global__ void __launch_bounds__(kThreads) dec_k3(DecodeArgs a) {
    extern __shared__ float4 sm4[];
    __shared__ float2 red[32];
    // this block's column range [c0, c0 + nc) of dR1 and of the W_O rows
    const int nc = a.H / a.ns3, c0 = blockIdx.y * nc, n4 = nc >> 2;
    // [sR (swizzled dR1) | sDo | sGam | sR1] over the range (nc floats each), then sGR over H
    float *sR = reinterpret_cast<float *>(sm4);
    float4 *sDo = sm4 + n4, *sGam = sm4 + 2 * n4, *sR1 = sm4 + 3 * n4, *sGR = sm4 + 4 * n4;
    pdl_trigger();
    const bool pre = a.flags & TLB_PRE_NORM, resid = a.flags & TLB_RESIDUAL;
    // Before the wait: gamma_ffn * r1 over all H and sum r1^2 (the pre-norm sums need all
    // of dim), and dOut, gamma_ffn, r1 over the range.
    float rr = 0.f;
    const int h4 = a.H >> 2;
    if (pre) {
        const float4 *g4 = reinterpret_cast<const float4 *>(a.g_ffn), *r4 = reinterpret_cast<const float4 *>(a.r1);
        for (int i = threadIdx.x; i < h4; i += blockDim.x) {
            const float4 g = g4[i], x = r4[i];
            sGR[i] = make_float4(g.x * x.x, g.y * x.y, g.z * x.z, g.w * x.w);
            rr += dot4(x, x);
        }
    }
    for (int i = threadIdx.x; i < n4; i += blockDim.x) {
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        sDo[i] = resid ? reinterpret_cast<const float4 *>(a.dout + c0)[i] : z;
        sGam[i] = pre ? reinterpret_cast<const float4 *>(a.g_ffn + c0)[i] : z;
        sR1[i] = pre ? reinterpret_cast<const float4 *>(a.r1 + c0)[i] : z;
    }
    {   // this block's W_O rows into L2, after the staging loads above (so they do not queue
        // behind this prefetch while the previous kernel still streams its weights)
        const int lane = threadIdx.x & 31, r = (blockIdx.x * kWarps + (threadIdx.x >> 5)) * kR + lane;
        if (lane < kR && r < a.qd)
            prefetch_l2(reinterpret_cast<const char *>(a.w_o) + wbytes<WT>(size_t(r) * a.H + c0), wbytes<WT>(size_t(nc)));
    }
    pdl_wait();
    // After the wait: dN2 (one round of loads), the pre-norm coefficients, dR1 over the range.
    float rinv = 1.f, c = 0.f;
    const float4 *dn4 = reinterpret_cast<const float4 *>(a.dN2);
    if (pre) {
        constexpr int B = 4;
        float4 dn[B];
#pragma unroll
        for (int b = 0; b < B; ++b) {
            const int i = threadIdx.x + b * blockDim.x;
            dn[b] = i < h4 ? __ldcg(dn4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float dot = 0.f;
        for (int base = threadIdx.x; base < h4; base += blockDim.x * B) {
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const int i = base + b * blockDim.x;
                if (i >= h4) break;
                const float4 d = base == int(threadIdx.x) ? dn[b] : __ldcg(dn4 + i);
                dot += dot4(d, sGR[i]);
                sGR[i] = d;
            }
        }
        rms_coef2(block_sum2(make_float2(dot, rr), red), a.H, a.eps, rinv, c);   // synchronises
    }
    for (int i = threadIdx.x; i < n4; i += blockDim.x) {
        const float4 dn = pre ? sGR[(c0 >> 2) + i] : __ldcg(dn4 + (c0 >> 2) + i);
        const float4 gm = sGam[i], r = sR1[i], dO = sDo[i];
        float4 v;
        v.x = (pre ? rinv * (dn.x * gm.x - r.x * c) : dn.x) + dO.x;
        v.y = (pre ? rinv * (dn.y * gm.y - r.y * c) : dn.y) + dO.y;
        v.z = (pre ? rinv * (dn.z * gm.z - r.z * c) : dn.z) + dO.z;
        v.w = (pre ? rinv * (dn.w * gm.w - r.w * c) : dn.w) + dO.w;
        reinterpret_cast<float4 *>(sR)[xunit<WT>(i)] = v;
        if (blockIdx.x == 0) reinterpret_cast<float4 *>(a.dR1 + c0)[i] = v;
    }
    __syncthreads();
    const char *W[1] = {reinterpret_cast<const char *>(a.w_o) + wbytes<WT>(size_t(c0))};
    const float sc[1] = {a.s_o};
    const float *xs[1] = {sR};
    const int r0 = (blockIdx.x * kWarps + (threadIdx.x >> 5)) * kR;
    float vals[kR] = {};
    if (r0 < a.qd) warp_rows<WT, 1, kR, kU, true>(W, sc, xs, r0, a.qd, nc, a.dSub, vals, wbytes<WT>(size_t(a.H)));
}

// ------------------------------------------------------------------ k4: attention, one pass over K and V

// Per (KV head, chunk of keys): dCtx of the group's heads (sub-norm backward), then for
// every key j of the chunk and head h of the group
//   dA = dCtx_h . V[j]      U_h += P dA K[j]      W_h += P K[j]      D_h += P dA
// so that dQ_h = scale (U_h - D_h W_h) summed over chunks equals
// scale sum_j P (dA - D_h) K[j] without a barrier on the row sum D_h.
// The chunk holding the current position also forms dV and its LoRA gh_v share.
template <int VPL, int GM>
__global__ void __launch_bounds__(kAThreads) dec_k4(DecodeArgs a) {
    constexpr int KPW = kDecodeChunk / kAWarps;        // keys per warp
    extern __shared__ float4 sm4[];
    __shared__ float2 red2[32];
    __shared__ float sDp[kAWarps][16];
    const int kvh = blockIdx.x, chunk = blockIdx.y;
    const bool dv_block = chunk == a.nchunks;          // the extra block of each KV head: dV, gh_v
    const int G = a.nh / a.nkv;
    const int hd = VPL * 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int d0 = lane * VPL;
    float *sC = reinterpret_cast<float *>(sm4);        // [G][hd] dCtx
    float *sR = sC + G * hd;                           // [kAWarps][G][2][hd] reduction (dV block: B_v rows)
    float *sGC = sR + kAWarps * G * 2 * hd;            // [qd] gamma * ctx, then dSub
    const bool sub = a.flags & TLB_SUB_NORM;
    {
        const int j0 = chunk * kDecodeChunk, nj = dv_block ? 0 : min(kDecodeChunk, a.L - j0);
        if (threadIdx.x < 2 * kDecodeChunk) {        // one K or V row per thread
            const int j = threadIdx.x % kDecodeChunk;
            const float *base = threadIdx.x < kDecodeChunk ? a.k : a.v;
            if (j < nj) prefetch_l2(base + int64_t(kvh) * a.sh + int64_t(j0 + j) * a.sp, size_t(hd) * 4);
        } else if (threadIdx.x < 2 * kDecodeChunk + G && nj > 0) {
            const int g = threadIdx.x - 2 * kDecodeChunk;
            prefetch_l2(a.attn + int64_t(kvh * G + g) * a.L + j0, size_t(nj) * 4);
        }
    }
    pdl_trigger();
    // Before the wait: this warp's K and V rows and P values, gamma * ctx over all q_dim
    // entries and sum ctx^2 (the sub-norm sums need all of them), and for the dV block
    // the KV head's rows of B_v.
    const int jw = chunk * kDecodeChunk + warp * KPW;
    float kv[KPW][VPL], vv[KPW][VPL], pl[KPW];
#pragma unroll
    for (int k = 0; k < KPW; ++k) {
        const int j = jw + k;
        const bool ok = !dv_block && j < a.L;
        const float *kr = a.k + int64_t(kvh) * a.sh + int64_t(ok ? j : 0) * a.sp + d0;
        const float *vr = a.v + int64_t(kvh) * a.sh + int64_t(ok ? j : 0) * a.sp + d0;
#pragma unroll
        for (int v = 0; v < VPL; ++v) {
            kv[k][v] = ok ? kr[v] : 0.f;
            vv[k][v] = ok ? vr[v] : 0.f;
        }
        // P of this key for each head of the group (lanes load in parallel)
        pl[k] = ok && lane < G ? a.attn[int64_t(kvh * G + lane) * a.L + j] : 0.f;
    }
    float cc = 0.f;
    if (sub) {
        const float4 *g4 = reinterpret_cast<const float4 *>(a.g_sub_attn);
        const float4 *c4 = reinterpret_cast<const float4 *>(a.ctx);
        for (int i = threadIdx.x; i < (a.qd >> 2); i += blockDim.x) {
            const float4 g = g4[i], x = c4[i];
            reinterpret_cast<float4 *>(sGC)[i] = make_float4(g.x * x.x, g.y * x.y, g.z * x.z, g.w * x.w);
            cc += dot4(x, x);
        }
    }
    if (dv_block)
        for (int i = threadIdx.x; i < hd * a.rank; i += blockDim.x) sR[i] = a.lv.b[int64_t(kvh) * hd * a.rank + i];
    pdl_wait();
    // After the wait: dSub (one round of loads), the sub-norm coefficients, dCtx.
    float rinv = 1.f, c = 0.f;
    if (sub) {
        constexpr int B = 4;
        const float4 *ds4 = reinterpret_cast<const float4 *>(a.dSub);
        const int n4 = a.qd >> 2;
        float4 dsv[B];
#pragma unroll
        for (int b = 0; b < B; ++b) {
            const int i = threadIdx.x + b * blockDim.x;
            dsv[b] = i < n4 ? __ldcg(ds4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float dot = 0.f;
        for (int base = threadIdx.x; base < n4; base += blockDim.x * B) {
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const int i = base + b * blockDim.x;
                if (i >= n4) break;
                const float4 d = base == int(threadIdx.x) ? dsv[b] : __ldcg(ds4 + i);
                dot += dot4(d, reinterpret_cast<const float4 *>(sGC)[i]);
                reinterpret_cast<float4 *>(sGC)[i] = d;      // each thread rereads only its own entries
            }
        }
        rms_coef2(block_sum2(make_float2(dot, cc), red2), a.qd, a.eps, rinv, c);
    }
    const int off = kvh * G * hd;
    for (int i = threadIdx.x; i < G * hd; i += blockDim.x) {
        const int q = off + i;
        sC[i] = sub ? rinv * (sGC[q] * a.g_sub_attn[q] - a.ctx[q] * c) : __ldcg(a.dSub + q);
    }
    if (kvh == 0 && chunk == 0 && a.dhid_out != nullptr)
        for (int i = threadIdx.x; i < a.H; i += blockDim.x) a.dhid_out[i] = __ldcg(a.dR1 + i);
    __syncthreads();
    if (dv_block) {
        // dV of the current token: dV[kvh, d] = sum_g attn[h_g, pos] dCtx_h_g[d]; gh_v share
        __shared__ float sv[256];
        __shared__ float rr[16][kAWarps];
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
#pragma unroll
            for (int r = 0; r < 16; ++r)
                if (r < a.rank) acc[r] = fmaf(sv[d], sR[d * a.rank + r], acc[r]);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const float t = warp_sum(acc[r]);
            if (lane == 0) rr[r][warp] = t;
        }
        __syncthreads();
        if (threadIdx.x < a.rank) {
            float t = 0.f;
            for (int w = 0; w < kAWarps; ++w) t += rr[threadIdx.x][w];
            atomicAdd(a.gh + a.rank + threadIdx.x, a.lora_scaling * t);
        }
        return;
    }
    float U[GM][VPL], W[GM][VPL];                      // GM >= heads per KV group
#pragma unroll
    for (int g = 0; g < GM; ++g)
#pragma unroll
        for (int v = 0; v < VPL; ++v) U[g][v] = W[g][v] = 0.f;
    float dsum[GM];
#pragma unroll
    for (int g = 0; g < GM; ++g) dsum[g] = 0.f;
#pragma unroll
    for (int k = 0; k < KPW; ++k) {
        if (jw + k >= a.L) break;
#pragma unroll
        for (int g = 0; g < GM; ++g) {
            if (g >= G) break;
            float t = 0.f;
#pragma unroll
            for (int v = 0; v < VPL; ++v) t = fmaf(sC[g * hd + d0 + v], vv[k][v], t);
            const float dA = warp_sum(t);
            const float P = __shfl_sync(0xffffffffu, pl[k], g);
            const float pd = P * dA;
            dsum[g] += pd;
#pragma unroll
            for (int v = 0; v < VPL; ++v) {
                U[g][v] = fmaf(pd, kv[k][v], U[g][v]);
                W[g][v] = fmaf(P, kv[k][v], W[g][v]);
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
        for (int w = 0; w < kAWarps; ++w) t += sR[w * G * 2 * hd + i];
        const int g = i / (2 * hd), which = (i / hd) & 1, d = i % hd;
        float *dst = which ? a.Wpart : a.Upart;
        dst[(int64_t(chunk) * a.nh + kvh * G + g) * hd + d] = t;
    }
    if (threadIdx.x < G) {
        float t = 0.f;
        for (int w = 0; w < kAWarps; ++w) t += sDp[w][threadIdx.x];
        a.Dpart[int64_t(chunk) * a.nh + kvh * G + threadIdx.x] = t;
    }
}

// ------------------------------------------------------------------ k6: dQpre and gh_q per head

__global__ void __launch_bounds__(kQThreads) dec_k6(DecodeArgs a, RopeFreqs fr) {
    __shared__ float sq[256];
    __shared__ float sD;
    __shared__ float red[16][kQWarps];
    __shared__ float sB[256 * 16];
    __shared__ float sCos[128], sSin[128];
    __shared__ float sQx[256], sGq[256], sNorm[2];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int h = blockIdx.x;
    const bool qkn = (a.flags & TLB_QK_NORM) != 0;
    pdl_trigger();
    // Before the wait: this head's rows of B_q (only this layer's k7, later, writes them)
    // and the rotation angles of the current position.
    for (int i = threadIdx.x; i < a.hd * a.rank; i += blockDim.x) sB[i] = a.lq.b[int64_t(h) * a.hd * a.rank + i];
    if (a.flags & TLB_ROPE)
        for (int d = threadIdx.x; d < (a.hd >> 1); d += blockDim.x)
            rope_cos_sin(float(a.pos), fr.hi[d], fr.lo[d], sCos[d], sSin[d]);
    if (qkn)                    // this head's pre-norm q and the norm's gain
        for (int d = threadIdx.x; d < a.hd; d += blockDim.x) {
            sQx[d] = a.q_raw[int64_t(h) * a.hd + d];
            sGq[d] = a.g_q[d];
        }
    pdl_wait();
    // blockDim / hd thread groups each sum a slice of the chunks (four chunks in flight per
    // thread), then combine
    __shared__ float su[kQThreads], sw[kQThreads];
    const int groups = blockDim.x / a.hd;
    const int grp = threadIdx.x / a.hd, d = threadIdx.x % a.hd;
    if (threadIdx.x < 32) {
        float t = 0.f;
        for (int c = lane; c < a.nchunks; c += 32) t += a.Dpart[int64_t(c) * a.nh + h];
        t = warp_sum(t);
        if (lane == 0) sD = t;
    }
    if (grp < groups) {
        float u[4] = {0.f, 0.f, 0.f, 0.f}, w[4] = {0.f, 0.f, 0.f, 0.f};
        int c = grp;
        for (; c + 3 * groups < a.nchunks; c += 4 * groups) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int64_t idx = (int64_t(c + k * groups) * a.nh + h) * a.hd + d;
                u[k] += a.Upart[idx];
                w[k] += a.Wpart[idx];
            }
        }
        for (; c < a.nchunks; c += groups) {
            const int64_t idx = (int64_t(c) * a.nh + h) * a.hd + d;
            u[0] += a.Upart[idx];
            w[0] += a.Wpart[idx];
        }
        su[threadIdx.x] = (u[0] + u[1]) + (u[2] + u[3]);
        sw[threadIdx.x] = (w[0] + w[1]) + (w[2] + w[3]);
    }
    __syncthreads();
    const float D = sD;
    if (a.Dout != nullptr && threadIdx.x == 0) a.Dout[h] = D;
    for (int dd = threadIdx.x; dd < a.hd; dd += blockDim.x) {
        float u = 0.f, w = 0.f;
        for (int g = 0; g < groups; ++g) {
            u += su[g * a.hd + dd];
            w += sw[g * a.hd + dd];
        }
        sq[dd] = a.scale * (u - D * w);
    }
    __syncthreads();
    const int half = a.hd >> 1;
    for (int d = threadIdx.x; d < half; d += blockDim.x) {
        float y1 = sq[d], y2 = sq[d + half];
        if (a.flags & TLB_ROPE) {
            const float cs = sCos[d], sn = sSin[d];
            const float t1 = y1 * cs + y2 * sn, t2 = -y1 * sn + y2 * cs;
            y1 = t1;
            y2 = t2;
        }
        sq[d] = y1;
        sq[d + half] = y2;   // each pair is owned by one thread
    }
    __syncthreads();
    if (qkn) {
        // QK-norm backward over the head (rms = sqrt(mean(x^2) + eps) of the pre-norm q x):
        // dx = (g dy - x sum(g dy x) / (hd rms^2)) / rms
        if (warp == 0) {
            float xx = 0.f, gx = 0.f;
            for (int d = lane; d < a.hd; d += 32) {
                xx += sQx[d] * sQx[d];
                gx += sGq[d] * sq[d] * sQx[d];
            }
            xx = warp_sum(xx);
            gx = warp_sum(gx);
            if (lane == 0) {
                sNorm[0] = xx;
                sNorm[1] = gx;
            }
        }
        __syncthreads();
        const float rms = sqrtf(sNorm[0] / float(a.hd) + a.eps), c = sNorm[1] / (float(a.hd) * rms * rms);
        for (int d = threadIdx.x; d < a.hd; d += blockDim.x) sq[d] = (sGq[d] * sq[d] - sQx[d] * c) / rms;
        __syncthreads();
    }
    for (int d = threadIdx.x; d < a.hd; d += blockDim.x) a.dqpre[h * a.hd + d] = sq[d];
    // gh_q[r] += s * sum_{d} dQpre[h, d] B_q[h*hd + d, r]   (B before its update)
    float acc[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) acc[r] = 0.f;
    for (int d = threadIdx.x; d < a.hd; d += blockDim.x) {
#pragma unroll
        for (int r = 0; r < 16; ++r)
            if (r < a.rank) acc[r] = fmaf(sq[d], sB[d * a.rank + r], acc[r]);
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        const float t = warp_sum(acc[r]);
        if (lane == 0) red[r][warp] = t;
    }
    __syncthreads();
    if (threadIdx.x < a.rank) {
        float t = 0.f;
        for (int w = 0; w < kQWarps; ++w) t += red[threadIdx.x][w];
        atomicAdd(a.gh + threadIdx.x, a.lora_scaling * t);
    }
}

// ------------------------------------------------------------------ k7: LoRA gradients + AdamW

// One thread per adapter element.  Before the wait: the element's parameter, moments and
// the cached factor it multiplies (h or x); after it: the chain's factor (dQpre, dV or
// gh), the gradient and the AdamW step.
__global__ void __launch_bounds__(kThreads) dec_k7(DecodeArgs a) {
    __shared__ float red[32];
    pdl_trigger();
    const int64_t nbq = int64_t(a.qd) * a.rank, nbv = int64_t(a.kvd) * a.rank, na = int64_t(a.rank) * a.H;
    const int64_t n = nbq + nbv + 2 * na;
    const int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    // which: 0 B_q, 1 B_v, 2 A_q, 3 A_v; f: index within it; o, r: its factors' indices
    int which = -1;
    int64_t f = 0;
    int o = 0, r = 0;
    if (e < nbq) {
        which = 0;
        f = e;
    } else if (e < nbq + nbv) {
        which = 1;
        f = e - nbq;
    } else if (e < n) {
        f = e - nbq - nbv;
        which = f < na ? 2 : 3;
        if (which == 3) f -= na;
    }
    const tlb_lora &l = (which == 0 || which == 2) ? a.lq : a.lv;
    float p = 0.f, m = 0.f, v = 0.f, fac = 0.f;
    if (which >= 0) {
        if (which <= 1) {
            o = int(f / a.rank);
            r = int(f % a.rank);
            p = l.b[f];
            m = l.m_b[f];
            v = l.v_b[f];
            fac = (which == 0 ? a.hq : a.hv)[r];
        } else {
            r = int(f / a.H);
            o = int(f % a.H);
            p = l.a[f];
            m = l.m_a[f];
            v = l.v_a[f];
            fac = a.x[o];
        }
    }
    pdl_wait();
    float sa = 0.f, sb = 0.f;   // dA^2, dB^2
    const bool step = a.status == nullptr || __ldcg(a.status + kStatusGate) == 0u;
    if (which >= 0) {
        float g;
        if (which == 0) g = a.lora_scaling * __ldcg(a.dqpre + o) * fac;
        else if (which == 1) g = a.lora_scaling * __ldcg(a.dv + o) * fac;
        else g = __ldcg(a.gh + (which == 2 ? 0 : a.rank) + r) * fac;
        if (which <= 1) {
            if (l.grad_b) l.grad_b[f] = g;
            if (step) {
                l.b[f] = adam_elem(p, g, m, v, a.kb);
                l.m_b[f] = m;
                l.v_b[f] = v;
            }
            sb = g * g;
        } else {
            if (l.grad_a) l.grad_a[f] = g;
            if (step) {
                l.a[f] = adam_elem(p, g, m, v, a.ka);
                l.m_a[f] = m;
                l.v_a[f] = v;
            }
            sa = g * g;
        }
    }
    if (a.sumsq) {
        const float ta = block_sum(sa, red);
        const float tb = block_sum(sb, red);
        if (threadIdx.x == 0) {
            if (ta != 0.f) atomicAdd(a.sumsq, double(ta));
            if (tb != 0.f) atomicAdd(a.sumsq + 1, double(tb));
        }
    }
}

template <typename... KArgs, typename... Args>
cudaError_t launch_b(void (*kernel)(KArgs...), dim3 grid, int block, size_t smem, cudaStream_t st, bool pdl,
                     Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;   // k2..k7 start early and wait on the kernel before them
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
    }
    // The largest shared-memory carveout: with the default split an SM hosts only two k2
    // blocks (28 KB each), and the rest of the grid waits for a second wave.  The weight
    // streams bypass L1, so the smaller L1 costs nothing.
    static std::mutex mu;
    static std::unordered_set<const void *> carved;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (carved.insert(reinterpret_cast<const void *>(kernel)).second) {
            cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                                 int(cudaSharedmemCarveoutMaxShared));
            if (e != cudaSuccess) return e;
        }
    }
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, size_t smem, cudaStream_t st, bool pdl, Args... args) {
    return launch_b(kernel, grid, kThreads, smem, st, pdl, args...);
}

template <int VPL>
cudaError_t launch_k4_g(int G, dim3 g4, size_t sm4, cudaStream_t st, const DecodeArgs &a) {
    if (G <= 1) return launch_b(dec_k4<VPL, 1>, g4, kAThreads, sm4, st, true, a);
    if (G <= 2) return launch_b(dec_k4<VPL, 2>, g4, kAThreads, sm4, st, true, a);
    if (G <= 4) return launch_b(dec_k4<VPL, 4>, g4, kAThreads, sm4, st, true, a);
    if (G <= 8) return launch_b(dec_k4<VPL, 8>, g4, kAThreads, sm4, st, true, a);
    if constexpr (VPL <= 4) return launch_b(dec_k4<VPL, 16>, g4, kAThreads, sm4, st, true, a);
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
int launch_ffn(const DecodeArgs &a, cudaStream_t st, bool k1_pdl) {
    TLB_CUDA(launch(dec_k1<WT>, dim3(unsigned(a.n1)), size_t(a.H) * 4, st, k1_pdl, a));
    TLB_TRY(check_launch("decode k1"));
    if constexpr (WT != TLB_W_TERNARY_2B) {
        // column-stationary k2: column blocks of at most 256 chunks (a whole number of warps),
        // about two blocks per SM in all
        const int nch = a.I / EPC<WT>::v, ncb = (nch + 255) / 256;
        const int bs = ((nch + ncb - 1) / ncb + 31) / 32 * 32;
        const int nrb = std::max(1, std::min(a.H, 2 * num_sms() / ncb));
        const size_t smc = size_t(bs / 32) * ceil_div(a.H, nrb) * 4;
        const dim3 gc{unsigned(nrb), unsigned(ncb)};
        if (a.act == TLB_ACT_RELU2_MUL) TLB_CUDA(launch_b(dec_k2c<WT, TLB_ACT_RELU2_MUL>, gc, bs, smc, st, true, a));
        else TLB_CUDA(launch_b(dec_k2c<WT, TLB_ACT_SILU_MUL>, gc, bs, smc, st, true, a));
    } else {
        const size_t sm2 = size_t(2) * (a.I / a.ns2) * 4;
        const dim3 g2(unsigned(a.n2), unsigned(a.ns2));
        if (a.act == TLB_ACT_RELU2_MUL) TLB_CUDA(launch(dec_k2<WT, TLB_ACT_RELU2_MUL>, g2, sm2, st, true, a));
        else TLB_CUDA(launch(dec_k2<WT, TLB_ACT_SILU_MUL>, g2, sm2, st, true, a));
    }
    TLB_TRY(check_launch("decode k2"));
    TLB_CUDA(launch(dec_k3<WT>, dim3(unsigned(a.n3), unsigned(a.ns3)), (size_t(4) * (a.H / a.ns3) + a.H) * 4, st,
                    true, a));
    TLB_TRY(check_launch("decode k3"));
    return TLB_OK;
}

int launch_k7(const DecodeArgs &a, cudaStream_t st) {
    const int64_t n7 = int64_t(a.qd + a.kvd) * a.rank + 2 * int64_t(a.rank) * a.H;
    TLB_CUDA(launch(dec_k7, dim3(unsigned(ceil_div(n7, kThreads))), 0, st, true, a));
    return check_launch("decode k7");
}

int launch_attn(const DecodeArgs &a, cudaStream_t st, bool with_k7) {
    const int G = a.nh / a.nkv;
    const dim3 g4(a.nkv, a.nchunks + 1);     // the last block of each KV head forms dV and gh_v
    const size_t sm4 = (size_t(G) * a.hd + size_t(kAWarps) * G * 2 * a.hd + size_t(a.qd)) * 4;
    TLB_CUDA(launch_k4(G, a.hd, g4, sm4, st, a));
    TLB_TRY(check_launch("decode k4"));
    RopeFreqs fr;
    rope_freqs(fr, a.hd, a.rope_base);
    TLB_CUDA(launch_b(dec_k6, dim3(a.nh), kQThreads, 0, st, true, a, fr));
    TLB_TRY(check_launch("decode k6"));
    return with_k7 ? launch_k7(a, st) : TLB_OK;
}

}  // namespace

int decode_rows_per_block() { return kWarps * kR; }

bool decode_supported(const tlb_layer_cfg &c, int64_t S, int64_t L) {
    const int G = c.n_heads / c.n_kv_heads;
    const int E = c.wtype == TLB_W_F32 ? 4 : (c.wtype == TLB_W_BF16 ? 8 : (c.wtype == TLB_W_TERNARY_I8 ? 16 : 64));
    const int hd = c.head_dim;
    const int gmax = hd > 128 ? 8 : 16;   // heads per KV group held in registers by k4
    const size_t sm4 = (size_t(G) * hd + size_t(kAWarps) * G * 2 * hd + size_t(c.n_heads) * hd) * 4;
    return S == 1 && G <= gmax && c.rank <= 16 && (hd == 32 || hd == 64 || hd == 128 || hd == 256) &&
           c.dim % E == 0 && c.ffn_dim % E == 0 && size_t(2) * c.ffn_dim * 4 <= 200 * 1024 &&
           sm4 <= 200 * 1024 && size_t(5) * c.dim * 4 <= 200 * 1024 && L >= 1;
}

int decode_ffn_launch(const DecodeArgs &a, int wtype, cudaStream_t st, bool k1_pdl) {
    switch (wtype) {
        case TLB_W_F32: return launch_ffn<TLB_W_F32>(a, st, k1_pdl);
        case TLB_W_BF16: return launch_ffn<TLB_W_BF16>(a, st, k1_pdl);
        case TLB_W_TERNARY_2B: return launch_ffn<TLB_W_TERNARY_2B>(a, st, k1_pdl);
        default: return launch_ffn<TLB_W_TERNARY_I8>(a, st, k1_pdl);
    }
}

int decode_attn_launch(const DecodeArgs &a, cudaStream_t st, bool with_k7) { return launch_attn(a, st, with_k7); }

int decode_lora_launch(const DecodeArgs &a, cudaStream_t st) { return launch_k7(a, st); }

int decode_layer_launch(const DecodeArgs &a, int wtype, cudaStream_t st) {
    // k1 too starts as a programmatic dependent of whatever kernel precedes the call: before
    // its wait it only prefetches its W_down rows into L2
    TLB_TRY(decode_ffn_launch(a, wtype, st, true));
    return decode_attn_launch(a, st);
}

}  // namespace tlb
