// Bandwidth-bound standalone steps: softmax backward, gated-activation backward,
// RMSNorm backward, RoPE backward and AdamW.  Each element is read once from HBM
// with 128-bit loads where the layout allows; row reductions stay in registers
// (warp shuffles, then shared memory across the warps of a row).
#include <cmath>

#include "common.cuh"
#include "kernels.cuh"

namespace tlb {

// ------------------------------------------------------------------ row reductions

// Sum over the TPR consecutive threads owning one row (TPR a power of two <= 1024).
// Every thread of the block must call it; `red` has blockDim/32 slots.
template <int TPR>
__device__ __forceinline__ float row_reduce(float v, float *red) {
    if constexpr (TPR <= 32) {
#pragma unroll
        for (int o = TPR / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        return v;
    } else {
        constexpr int W = TPR / 32;
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        v = warp_sum(v);
        if (lane == 0) red[warp] = v;
        __syncthreads();
        const int first = (warp / W) * W;
        float t = 0.f;
#pragma unroll
        for (int i = 0; i < W; ++i) t += red[first + i];
        __syncthreads();
        return t;
    }
}

template <int TPR>
__device__ __forceinline__ float2 row_reduce2(float2 v, float2 *red) {
    if constexpr (TPR <= 32) {
#pragma unroll
        for (int o = TPR / 2; o > 0; o >>= 1) {
            v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
            v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
        }
        return v;
    } else {
        constexpr int W = TPR / 32;
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        v = warp_sum2(v);
        if (lane == 0) red[warp] = v;
        __syncthreads();
        const int first = (warp / W) * W;
        float2 t = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < W; ++i) {
            t.x += red[first + i].x;
            t.y += red[first + i].y;
        }
        __syncthreads();
        return t;
    }
}

// ------------------------------------------------------------------ softmax backward

// Row r of rows x (len4*4): VPT float4 per thread, TPR threads per row, the row
// held in registers between the dot product and the output.
template <int VPT, int TPR>
__global__ void __launch_bounds__(TPR > 256 ? TPR : 256)
softmax_bwd_vec_kernel(const float4 *__restrict__ attn, const float4 *__restrict__ dattn,
                       float4 *__restrict__ ds, int64_t rows, int len4) {
    __shared__ float red[32];
    const int rpb = blockDim.x / TPR;
    const int sub = threadIdx.x / TPR, t = threadIdx.x % TPR;
    const int64_t row = int64_t(blockIdx.x) * rpb + sub;
    const bool active = row < rows;
    const int64_t base = row * len4;
    float4 a[VPT], g[VPT];
    float dot = 0.f;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int idx = v * TPR + t;
        if (active && idx < len4) {
            a[v] = ld_stream(attn + base + idx);
            g[v] = ld_stream(dattn + base + idx);
        } else {
            a[v] = make_float4(0.f, 0.f, 0.f, 0.f);
            g[v] = a[v];
        }
        dot += dot4(a[v], g[v]);
    }
    dot = row_reduce<TPR>(dot, red);
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int idx = v * TPR + t;
        if (active && idx < len4) {
            float4 o;
            o.x = a[v].x * (g[v].x - dot);
            o.y = a[v].y * (g[v].y - dot);
            o.z = a[v].z * (g[v].z - dot);
            o.w = a[v].w * (g[v].w - dot);
            __stcs(ds + base + idx, o);
        }
    }
}

// Rows longer than the register-resident variants hold: one block per row, two
// passes; the second pass re-reads the row from L2 (rows in flight stay far below
// the L2 size), so HBM still sees each element once.
__global__ void __launch_bounds__(1024)
softmax_bwd_2pass_vec_kernel(const float4 *__restrict__ attn, const float4 *__restrict__ dattn,
                             float4 *__restrict__ ds, int64_t len4) {
    __shared__ float red[32];
    const int64_t base = int64_t(blockIdx.x) * len4;
    float dot = 0.f;
    for (int64_t j = threadIdx.x; j < len4; j += blockDim.x) dot += dot4(attn[base + j], dattn[base + j]);
    dot = block_sum(dot, red);
    for (int64_t j = threadIdx.x; j < len4; j += blockDim.x) {
        const float4 a = attn[base + j], g = dattn[base + j];
        __stcs(ds + base + j, make_float4(a.x * (g.x - dot), a.y * (g.y - dot), a.z * (g.z - dot),
                                          a.w * (g.w - dot)));
    }
}

// Any length and alignment: one block per row, two passes over the row.
__global__ void softmax_bwd_generic_kernel(const float *__restrict__ attn,
                                           const float *__restrict__ dattn,
                                           float *__restrict__ ds, int64_t len) {
    __shared__ float red[32];
    const int64_t base = int64_t(blockIdx.x) * len;
    float dot = 0.f;
    for (int64_t j = threadIdx.x; j < len; j += blockDim.x) dot += attn[base + j] * dattn[base + j];
    dot = block_sum(dot, red);
    for (int64_t j = threadIdx.x; j < len; j += blockDim.x)
        ds[base + j] = attn[base + j] * (dattn[base + j] - dot);
}

template <int VPT, int TPR>
static void launch_softmax_vec(const float *a, const float *g, float *o, int64_t rows, int len4,
                               cudaStream_t st) {
    const int block = TPR > 256 ? TPR : 256;
    const int rpb = block / TPR;
    softmax_bwd_vec_kernel<VPT, TPR><<<(unsigned)ceil_div(rows, rpb), block, 0, st>>>(
        reinterpret_cast<const float4 *>(a), reinterpret_cast<const float4 *>(g),
        reinterpret_cast<float4 *>(o), rows, len4);
}

int softmax_backward_launch(const float *attn, const float *dattn, float *ds, int64_t rows,
                            int64_t len, cudaStream_t st) {
    if (rows == 0 || len == 0) return TLB_OK;
    TLB_REQUIRE(rows < (int64_t(1) << 31), TLB_EUNSUPPORTED, "softmax_backward: rows >= 2^31");
    const bool vec = (len % 4 == 0) && aligned16(attn) && aligned16(dattn) && aligned16(ds);
    const int64_t len4 = len / 4;
    if (vec && len4 <= 4096) {
        const int l4 = int(len4);
        if (l4 <= 32) launch_softmax_vec<1, 32>(attn, dattn, ds, rows, l4, st);
        else if (l4 <= 64) launch_softmax_vec<2, 32>(attn, dattn, ds, rows, l4, st);
        else if (l4 <= 128) launch_softmax_vec<4, 32>(attn, dattn, ds, rows, l4, st);
        else if (l4 <= 256) launch_softmax_vec<4, 64>(attn, dattn, ds, rows, l4, st);
        else if (l4 <= 512) launch_softmax_vec<4, 128>(attn, dattn, ds, rows, l4, st);
        else if (l4 <= 1024) launch_softmax_vec<4, 256>(attn, dattn, ds, rows, l4, st);
        else if (l4 <= 2048) launch_softmax_vec<4, 512>(attn, dattn, ds, rows, l4, st);
        else launch_softmax_vec<4, 1024>(attn, dattn, ds, rows, l4, st);
    } else if (vec) {
        softmax_bwd_2pass_vec_kernel<<<(unsigned)rows, 1024, 0, st>>>(
            reinterpret_cast<const float4 *>(attn), reinterpret_cast<const float4 *>(dattn),
            reinterpret_cast<float4 *>(ds), len4);
    } else {
        softmax_bwd_generic_kernel<<<(unsigned)rows, 256, 0, st>>>(attn, dattn, ds, len);
    }
    return check_launch("softmax_backward");
}

// ------------------------------------------------------------------ RMSNorm backward

template <int VPT, int TPR>
__global__ void __launch_bounds__(TPR > 256 ? TPR : 256)
rmsnorm_bwd_vec_kernel(const float4 *__restrict__ x, const float4 *__restrict__ gamma,
                       const float4 *dy, float4 *dx, int64_t rows, int n4, float inv_n,
                       float eps, int accumulate) {
    __shared__ float2 red[32];
    const int rpb = blockDim.x / TPR;
    const int sub = threadIdx.x / TPR, t = threadIdx.x % TPR;
    const int64_t row = int64_t(blockIdx.x) * rpb + sub;
    const bool active = row < rows;
    const int64_t base = row * n4;
    float4 xv[VPT], gy[VPT];
    float2 acc = make_float2(0.f, 0.f);   // (sum x^2, sum dy*gamma*x)
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int idx = v * TPR + t;
        if (active && idx < n4) {
            xv[v] = ld_stream(x + base + idx);
            const float4 d = dy[base + idx];
            const float4 g = __ldg(gamma + idx);
            gy[v] = make_float4(d.x * g.x, d.y * g.y, d.z * g.z, d.w * g.w);
        } else {
            xv[v] = make_float4(0.f, 0.f, 0.f, 0.f);
            gy[v] = xv[v];
        }
        acc.x += dot4(xv[v], xv[v]);
        acc.y += dot4(gy[v], xv[v]);
    }
    acc = row_reduce2<TPR>(acc, red);
    const float ms = acc.x * inv_n + eps;           // rms^2
    const float rinv = rsqrtf(ms);
    const float c = acc.y * inv_n / ms;             // dot / (n rms^2)
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int idx = v * TPR + t;
        if (active && idx < n4) {
            float4 o;
            o.x = rinv * (gy[v].x - xv[v].x * c);
            o.y = rinv * (gy[v].y - xv[v].y * c);
            o.z = rinv * (gy[v].z - xv[v].z * c);
            o.w = rinv * (gy[v].w - xv[v].w * c);
            if (accumulate) {
                const float4 p = dx[base + idx];
                o.x += p.x;
                o.y += p.y;
                o.z += p.z;
                o.w += p.w;
            }
            dx[base + idx] = o;
        }
    }
}

__global__ void rmsnorm_bwd_generic_kernel(const float *__restrict__ x, const float *__restrict__ gamma,
                                           const float *dy, float *dx, int64_t n, float eps,
                                           int accumulate) {
    __shared__ float2 red[32];
    const int64_t base = int64_t(blockIdx.x) * n;
    float2 acc = make_float2(0.f, 0.f);
    for (int64_t j = threadIdx.x; j < n; j += blockDim.x) {
        const float xv = x[base + j], gy = dy[base + j] * gamma[j];
        acc.x += xv * xv;
        acc.y += gy * xv;
    }
    acc = block_sum2(acc, red);
    const float ms = acc.x / float(n) + eps;
    const float rinv = rsqrtf(ms);
    const float c = acc.y / float(n) / ms;
    // dx may alias dy: each element is read and then written by the same thread.
    for (int64_t j = threadIdx.x; j < n; j += blockDim.x) {
        const float xv = x[base + j], gy = dy[base + j] * gamma[j];
        float o = rinv * (gy - xv * c);
        if (accumulate) o += dx[base + j];
        dx[base + j] = o;
    }
}

template <int VPT, int TPR>
static void launch_rms_vec(const float *x, const float *g, const float *dy, float *dx, int64_t rows,
                           int n4, float eps, int acc, cudaStream_t st) {
    const int block = TPR > 256 ? TPR : 256;
    const int rpb = block / TPR;
    rmsnorm_bwd_vec_kernel<VPT, TPR><<<(unsigned)ceil_div(rows, rpb), block, 0, st>>>(
        reinterpret_cast<const float4 *>(x), reinterpret_cast<const float4 *>(g),
        reinterpret_cast<const float4 *>(dy), reinterpret_cast<float4 *>(dx), rows, n4,
        1.0f / float(n4 * 4), eps, acc);
}

int rmsnorm_backward_launch(const float *x, const float *gamma, const float *dy, float *dx,
                            int64_t rows, int64_t n, float eps, int accumulate, cudaStream_t st) {
    if (rows == 0 || n == 0) return TLB_OK;
    TLB_REQUIRE(rows < (int64_t(1) << 31), TLB_EUNSUPPORTED, "rmsnorm_backward: rows >= 2^31");
    const bool vec = (n % 4 == 0) && aligned16(x) && aligned16(gamma) && aligned16(dy) && aligned16(dx);
    const int64_t n4 = n / 4;
    if (vec && n4 <= 4096) {
        const int m = int(n4);
        if (m <= 32) launch_rms_vec<1, 32>(x, gamma, dy, dx, rows, m, eps, accumulate, st);
        else if (m <= 64) launch_rms_vec<2, 32>(x, gamma, dy, dx, rows, m, eps, accumulate, st);
        else if (m <= 128) launch_rms_vec<4, 32>(x, gamma, dy, dx, rows, m, eps, accumulate, st);
        else if (m <= 256) launch_rms_vec<4, 64>(x, gamma, dy, dx, rows, m, eps, accumulate, st);
        else if (m <= 512) launch_rms_vec<4, 128>(x, gamma, dy, dx, rows, m, eps, accumulate, st);
        else if (m <= 1024) launch_rms_vec<4, 256>(x, gamma, dy, dx, rows, m, eps, accumulate, st);
        else if (m <= 2048) launch_rms_vec<4, 512>(x, gamma, dy, dx, rows, m, eps, accumulate, st);
        else launch_rms_vec<4, 1024>(x, gamma, dy, dx, rows, m, eps, accumulate, st);
    } else {
        rmsnorm_bwd_generic_kernel<<<(unsigned)rows, 256, 0, st>>>(x, gamma, dy, dx, n, eps, accumulate);
    }
    return check_launch("rmsnorm_backward");
}

// ------------------------------------------------------------------ gated activation backward


template <int ACT, bool CACHE>
__global__ void act_bwd_kernel(const float4 *__restrict__ gate, const float4 *__restrict__ up,
                               const float4 *__restrict__ sg, const float4 *__restrict__ dh,
                               float4 *__restrict__ dgate, float4 *__restrict__ dup, int64_t n4) {
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
         i += int64_t(gridDim.x) * blockDim.x) {
        const float4 g = ld_stream(gate + i), u = ld_stream(up + i), d = ld_stream(dh + i);
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        if constexpr (CACHE) s = ld_stream(sg + i);
        float4 og, ou;
        act_bwd_elem<ACT, CACHE>(g.x, u.x, s.x, d.x, og.x, ou.x);
        act_bwd_elem<ACT, CACHE>(g.y, u.y, s.y, d.y, og.y, ou.y);
        act_bwd_elem<ACT, CACHE>(g.z, u.z, s.z, d.z, og.z, ou.z);
        act_bwd_elem<ACT, CACHE>(g.w, u.w, s.w, d.w, og.w, ou.w);
        __stcs(dgate + i, og);
        __stcs(dup + i, ou);
    }
}

template <int ACT, bool CACHE>
__global__ void act_bwd_scalar_kernel(const float *__restrict__ gate, const float *__restrict__ up,
                                      const float *__restrict__ sg, const float *__restrict__ dh,
                                      float *__restrict__ dgate, float *__restrict__ dup, int64_t n) {
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += int64_t(gridDim.x) * blockDim.x) {
        float og, ou;
        act_bwd_elem<ACT, CACHE>(gate[i], up[i], CACHE ? sg[i] : 0.f, dh[i], og, ou);
        dgate[i] = og;
        dup[i] = ou;
    }
}

template <int ACT, bool CACHE>
static void launch_act(const float *g, const float *u, const float *s, const float *dh, float *dg,
                       float *du, int64_t n, bool vec, cudaStream_t st) {
    if (vec) {
        act_bwd_kernel<ACT, CACHE><<<stream_grid(n / 4, 256), 256, 0, st>>>(
            reinterpret_cast<const float4 *>(g), reinterpret_cast<const float4 *>(u),
            reinterpret_cast<const float4 *>(s), reinterpret_cast<const float4 *>(dh),
            reinterpret_cast<float4 *>(dg), reinterpret_cast<float4 *>(du), n / 4);
    } else {
        act_bwd_scalar_kernel<ACT, CACHE><<<stream_grid(n, 256), 256, 0, st>>>(g, u, s, dh, dg, du, n);
    }
}

int act_backward_launch(int act, const float *gate, const float *up, const float *silu_gate,
                        const float *dh, float *dgate, float *dup, int64_t n, cudaStream_t st) {
    if (n == 0) return TLB_OK;
    const bool cache = silu_gate != nullptr && act == TLB_ACT_SILU_MUL;
    const bool vec = (n % 4 == 0) && aligned16(gate) && aligned16(up) && aligned16(dh) &&
                     aligned16(dgate) && aligned16(dup) && (!cache || aligned16(silu_gate));
    if (act == TLB_ACT_RELU2_MUL)
        launch_act<TLB_ACT_RELU2_MUL, false>(gate, up, nullptr, dh, dgate, dup, n, vec, st);
    else if (cache)
        launch_act<TLB_ACT_SILU_MUL, true>(gate, up, silu_gate, dh, dgate, dup, n, vec, st);
    else
        launch_act<TLB_ACT_SILU_MUL, false>(gate, up, nullptr, dh, dgate, dup, n, vec, st);
    return check_launch("act_backward");
}

template <int ACT, bool CACHE>
__global__ void act_bwd_bf16_kernel(const float4 *__restrict__ gate, const float4 *__restrict__ up,
                                    const float4 *__restrict__ sg, const float4 *__restrict__ dh,
                                    uint2 *__restrict__ dgate, uint2 *__restrict__ dup, int64_t n4) {
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
         i += int64_t(gridDim.x) * blockDim.x) {
        const float4 g = ld_stream(gate + i), u = ld_stream(up + i), d = ld_stream(dh + i);
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        if constexpr (CACHE) s = ld_stream(sg + i);
        float4 og, ou;
        act_bwd_elem<ACT, CACHE>(g.x, u.x, s.x, d.x, og.x, ou.x);
        act_bwd_elem<ACT, CACHE>(g.y, u.y, s.y, d.y, og.y, ou.y);
        act_bwd_elem<ACT, CACHE>(g.z, u.z, s.z, d.z, og.z, ou.z);
        act_bwd_elem<ACT, CACHE>(g.w, u.w, s.w, d.w, og.w, ou.w);
        dgate[i] = pack_bf16x4(og.x, og.y, og.z, og.w);
        dup[i] = pack_bf16x4(ou.x, ou.y, ou.z, ou.w);
    }
}

int act_backward_bf16_launch(int act, const float *gate, const float *up, const float *silu_gate, const float *dh,
                             void *dgate, void *dup, int64_t n, cudaStream_t st) {
    if (n == 0) return TLB_OK;
    const bool cache = silu_gate != nullptr && act == TLB_ACT_SILU_MUL;
    TLB_REQUIRE(n % 4 == 0 && aligned16(gate) && aligned16(up) && aligned16(dh) && aligned16(dgate) &&
                    aligned16(dup) && (!cache || aligned16(silu_gate)),
                TLB_EUNSUPPORTED, "act_backward (bf16 out): n %% 4 or alignment");
    const unsigned grid = stream_grid(n / 4, 256);
    const float4 *g4 = reinterpret_cast<const float4 *>(gate), *u4 = reinterpret_cast<const float4 *>(up);
    const float4 *s4 = reinterpret_cast<const float4 *>(silu_gate), *d4 = reinterpret_cast<const float4 *>(dh);
    uint2 *og = reinterpret_cast<uint2 *>(dgate), *ou = reinterpret_cast<uint2 *>(dup);
    if (act == TLB_ACT_RELU2_MUL)
        act_bwd_bf16_kernel<TLB_ACT_RELU2_MUL, false><<<grid, 256, 0, st>>>(g4, u4, nullptr, d4, og, ou, n / 4);
    else if (cache)
        act_bwd_bf16_kernel<TLB_ACT_SILU_MUL, true><<<grid, 256, 0, st>>>(g4, u4, s4, d4, og, ou, n / 4);
    else
        act_bwd_bf16_kernel<TLB_ACT_SILU_MUL, false><<<grid, 256, 0, st>>>(g4, u4, nullptr, d4, og, ou, n / 4);
    return check_launch("act_backward_bf16");
}

// ------------------------------------------------------------------ RoPE backward

// One thread per (row, head, d) with d < head_dim/2: rotates the pair (d, d + half).
// dx may alias dy (each pair is read, then written, by one thread).
__global__ void rope_bwd_kernel(const float *dy, float *dx, int64_t rows, int n_heads, int head_dim,
                                int64_t pos0, RopeFreqs fr) {
    const int half = head_dim >> 1;
    const int64_t total = rows * n_heads * half;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int d = int(i % half);
        const int64_t rh = i / half;              // row * n_heads + head
        const int64_t row = rh / n_heads;
        const int64_t off = rh * head_dim + d;
        float c, s;
        rope_cos_sin(float(pos0 + row), fr.hi[d], fr.lo[d], c, s);
        const float y1 = dy[off], y2 = dy[off + half];
        dx[off] = y1 * c + y2 * s;
        dx[off + half] = -y1 * s + y2 * c;
    }
}

// The angle depends on the position and the frequency index only, so one thread per
// (row, group of hpt heads, four frequencies) computes its four cos/sin pairs once and
// rotates those pairs in each head of its group, with 128-bit loads and stores (HU
// heads in flight).  hpt is all the heads unless rows are too few to fill the GPU.
// Needs head_dim/2 a multiple of 4 and 16-byte aligned buffers; dx may alias dy.
template <int HU>
__global__ void __launch_bounds__(256)
rope_bwd_vec_kernel(const float4 *dy, float4 *dx, int64_t rows, int n_heads, int hpt, int half4,
                    int64_t pos0, RopeFreqs fr) {
    const int groups = (n_heads + hpt - 1) / hpt;
    const int64_t total = rows * groups * half4;
    const int64_t hd4 = 2 * int64_t(half4);
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t rg = i / half4;
        const int q = int(i - rg * half4);
        const int64_t row = rg / groups;
        const int h0 = int(rg - row * groups) * hpt;
        const int h1 = min(h0 + hpt, n_heads);
        const float pos = float(pos0 + row);
        float c[4], s[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) rope_cos_sin(pos, fr.hi[4 * q + k], fr.lo[4 * q + k], c[k], s[k]);
        const int64_t base = row * n_heads * hd4 + q;
        for (int h = h0; h < h1; h += HU) {
            float4 a[HU], b[HU];
#pragma unroll
            for (int u = 0; u < HU; ++u) {
                if (h + u < h1) {
                    a[u] = __ldcs(dy + base + (h + u) * hd4);
                    b[u] = __ldcs(dy + base + (h + u) * hd4 + half4);
                }
            }
#pragma unroll
            for (int u = 0; u < HU; ++u) {
                if (h + u < h1) {
                    float4 o1, o2;
                    o1.x = a[u].x * c[0] + b[u].x * s[0];
                    o2.x = -a[u].x * s[0] + b[u].x * c[0];
                    o1.y = a[u].y * c[1] + b[u].y * s[1];
                    o2.y = -a[u].y * s[1] + b[u].y * c[1];
                    o1.z = a[u].z * c[2] + b[u].z * s[2];
                    o2.z = -a[u].z * s[2] + b[u].z * c[2];
                    o1.w = a[u].w * c[3] + b[u].w * s[3];
                    o2.w = -a[u].w * s[3] + b[u].w * c[3];
                    __stcs(dx + base + (h + u) * hd4, o1);
                    __stcs(dx + base + (h + u) * hd4 + half4, o2);
                }
            }
        }
    }
}

int rope_backward_launch(const float *dy, float *dx, int64_t rows, int n_heads, int head_dim,
                         int64_t pos0, float base, cudaStream_t st) {
    if (rows == 0 || n_heads == 0) return TLB_OK;
    RopeFreqs fr;
    rope_freqs(fr, head_dim, base);
    const int half = head_dim / 2;
    if (half % 4 == 0 && aligned16(dy) && aligned16(dx)) {
        // heads per thread: all of them once the (row, frequency) items alone fill
        // about 1024 threads per SM, fewer (down to one) below that
        const int64_t items = rows * (half / 4), fill = int64_t(num_sms()) * 1024;
        const int64_t want = items * n_heads / fill;
        const int hpt = int(want < 1 ? 1 : (want > n_heads ? n_heads : want));
        const int64_t total = items * ((n_heads + hpt - 1) / hpt);
        rope_bwd_vec_kernel<4><<<stream_grid(total, 256), 256, 0, st>>>(
            reinterpret_cast<const float4 *>(dy), reinterpret_cast<float4 *>(dx), rows, n_heads, hpt,
            half / 4, pos0, fr);
    } else {
        const int64_t total = rows * n_heads * half;
        rope_bwd_kernel<<<stream_grid(total, 256), 256, 0, st>>>(dy, dx, rows, n_heads, head_dim, pos0, fr);
    }
    return check_launch("rope_backward");
}

// ------------------------------------------------------------------ AdamW

__global__ void adamw_kernel(float4 *p, const float4 *__restrict__ g, float4 *m, float4 *v, int64_t n4,
                             AdamCoef k, double *sumsq) {
    __shared__ float red[32];
    float ss = 0.f;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
         i += int64_t(gridDim.x) * blockDim.x) {
        float4 pp = p[i], mm = m[i], vv = v[i];
        const float4 gg = ld_stream(g + i);
        pp.x = adam_elem(pp.x, gg.x, mm.x, vv.x, k);
        pp.y = adam_elem(pp.y, gg.y, mm.y, vv.y, k);
        pp.z = adam_elem(pp.z, gg.z, mm.z, vv.z, k);
        pp.w = adam_elem(pp.w, gg.w, mm.w, vv.w, k);
        ss += dot4(gg, gg);
        p[i] = pp;
        m[i] = mm;
        v[i] = vv;
    }
    if (sumsq != nullptr) {
        ss = block_sum(ss, red);
        if (threadIdx.x == 0) atomicAdd(sumsq, double(ss));
    }
}

__global__ void adamw_scalar_kernel(float *p, const float *__restrict__ g, float *m, float *v, int64_t n,
                                    AdamCoef k, double *sumsq) {
    __shared__ float red[32];
    float ss = 0.f;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += int64_t(gridDim.x) * blockDim.x) {
        float mm = m[i], vv = v[i];
        const float gg = g[i];
        p[i] = adam_elem(p[i], gg, mm, vv, k);
        m[i] = mm;
        v[i] = vv;
        ss += gg * gg;
    }
    if (sumsq != nullptr) {
        ss = block_sum(ss, red);
        if (threadIdx.x == 0) atomicAdd(sumsq, double(ss));
    }
}

int adamw_launch(float *p, const float *g, float *m, float *v, int64_t n, const tlb_adamw_cfg &cfg,
                 float lr_mult, double *sumsq, cudaStream_t st) {
    if (n == 0) return TLB_OK;
    const AdamCoef k = adam_coef(cfg, lr_mult);
    if (n % 4 == 0 && aligned16(p) && aligned16(g) && aligned16(m) && aligned16(v)) {
        adamw_kernel<<<stream_grid(n / 4, 256), 256, 0, st>>>(
            reinterpret_cast<float4 *>(p), reinterpret_cast<const float4 *>(g),
            reinterpret_cast<float4 *>(m), reinterpret_cast<float4 *>(v), n / 4, k, sumsq);
    } else {
        adamw_scalar_kernel<<<stream_grid(n, 256), 256, 0, st>>>(p, g, m, v, n, k, sumsq);
    }
    return check_launch("adamw");
}


// ------------------------------------------------------------------ finiteness check

// Any non-finite element of x[0, n) records kDevNonFinite (first device error wins) and
// the site in the workspace status block.
__global__ void finite_check_kernel(const float *__restrict__ x, int64_t n, uint32_t *status, uint32_t site,
                                    int vec) {
    bool bad = false;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (vec) {
        const float4 *x4 = reinterpret_cast<const float4 *>(x);
        for (; i < n / 4; i += stride) {
            const float4 v = ld_stream(x4 + i);
            bad |= !(isfinite(v.x) && isfinite(v.y) && isfinite(v.z) && isfinite(v.w));
        }
        i = n / 4 * 4 + int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    }
    for (; i < n; i += stride) bad |= !isfinite(x[i]);
    if (__syncthreads_or(bad) && threadIdx.x == 0 &&
        atomicCAS(status + kStatusCode, 0u, uint32_t(kDevNonFinite)) == 0u)
        atomicExch(status + kStatusWhere, site);
}

__global__ void finite_gate_kernel(const uint32_t *status, uint32_t *gate_block) {
    gate_block[kStatusGate] = __ldcg(status + kStatusCode) == uint32_t(kDevNonFinite) ? 1u : 0u;
}

int finite_gate_launch(const uint32_t *status, uint32_t *gate_block, cudaStream_t st) {
    finite_gate_kernel<<<1, 1, 0, st>>>(status, gate_block);
    return check_launch("finite_gate");
}

int finite_check_launch(const float *x, int64_t n, uint32_t *status, uint32_t site, cudaStream_t st) {
    if (n == 0) return TLB_OK;
    const int vec = aligned16(x) ? 1 : 0;
    finite_check_kernel<<<stream_grid(vec ? n / 4 + 1 : n, 256), 256, 0, st>>>(x, n, status, site, vec);
    return check_launch("finite_check");
}

}  // namespace tlb
