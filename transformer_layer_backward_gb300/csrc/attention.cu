// Attention backward over cached K/V with GQA, from dCtx down to dQpre and dV
// ([ATT] "Gradient Flow", apply / softmax / score / RoPE backward; [RS]
// backward_through_layers, attention block).
//
// Sequence kernels (S > 1, head_dim 32/64/128): attn_dq_tiled and attn_dv_tiled below.
// General kernels (any S, L, strides; decode rows and other head sizes):
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

constexpr int kT = 64;          // tile edge
constexpr int kTP = kT + 4;     // padded row of a transposed tile (float4-aligned, 4-way store conflicts)

__global__ void attn_rows_kernel(AttnArgs a, RopeFreqs fr) {
    extern __shared__ float4 smem4[];
    __shared__ float red[32];
    float *sS = reinterpret_cast<float *>(smem4);
    float *sd = sS + a.L;
    float *sq = sd + a.hd;
    float *sqr = sq + a.hd;                      // recompute: the query row, then P[0 .. L)
    float *sP = sqr + a.hd;
    const int i = blockIdx.x, h = blockIdx.y;
    const int kvh = h / (a.nh / a.nkv);
    const int q_dim = a.nh * a.hd;
    const int jmax = a.causal ? min(a.L, a.pos0 + i + 1) : a.L;
    const bool rc = a.lse != nullptr;
    for (int d = threadIdx.x; d < a.hd; d += blockDim.x) {
        sd[d] = a.dctx[int64_t(i) * q_dim + h * a.hd + d];
        if (rc) sqr[d] = a.q[int64_t(i) * q_dim + h * a.hd + d];
    }
    __syncthreads();
    const float *Vh = a.v + int64_t(kvh) * a.sh;
    const float *Kh = a.k + int64_t(kvh) * a.sh;
    const float lse = rc ? a.lse[int64_t(h) * a.S + i] : 0.f;
    for (int j = threadIdx.x; j < jmax; j += blockDim.x) {
        const float *vr = Vh + int64_t(j) * a.sp;
        float acc = 0.f;
        for (int d = 0; d < a.hd; ++d) acc = fmaf(sd[d], vr[d], acc);
        sS[j] = acc;
        if (rc) {
            const float *kr = Kh + int64_t(j) * a.sp;
            float s = 0.f;
            for (int d = 0; d < a.hd; ++d) s = fmaf(sqr[d], kr[d], s);
            sP[j] = expf(a.scale * s - lse);
        }
    }
    __syncthreads();
    const float *P = rc ? sP : a.attn + (int64_t(h) * a.S + i) * a.L;
    float part = 0.f;
    for (int j = threadIdx.x; j < jmax; j += blockDim.x) part += P[j] * sS[j];
    const float D = block_sum(part, red);
    if (a.D != nullptr && threadIdx.x == 0) a.D[int64_t(h) * a.S + i] = D;
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

// Recomputed attention: one block per (newest key jj, KV head), the P values of up to
// blockDim (head, query) pairs at a time formed one pair per thread (scale q . k - lse),
// then every thread adds their share of the pairs' dCtx rows into its head_dim columns.
__global__ void attn_dv_rc_kernel(AttnArgs a) {
    extern __shared__ float4 smem4[];
    float *sK = reinterpret_cast<float *>(smem4);      // [hd] K row of the key
    float *sPp = sK + a.hd;                            // [blockDim] P of the current pairs
    const int jj = blockIdx.x, kvh = blockIdx.y, G = a.nh / a.nkv;
    const int j = a.pos0 + jj, q_dim = a.nh * a.hd;
    const int i0 = a.causal ? jj : 0;
    const int nq = a.S - i0, npairs = G * nq;
    const float *Kj = a.k + int64_t(kvh) * a.sh + int64_t(j) * a.sp;
    for (int d = threadIdx.x; d < a.hd; d += blockDim.x) sK[d] = Kj[d];
    constexpr int kMaxCols = 2;                        // head_dim <= 256, blockDim 128
    float acc[kMaxCols] = {0.f, 0.f};
    __syncthreads();
    for (int p0 = 0; p0 < npairs; p0 += blockDim.x) {
        const int pp = p0 + threadIdx.x;
        float P = 0.f;
        if (pp < npairs) {
            const int h = kvh * G + pp / nq, i = i0 + pp % nq;
            const float *qr = a.q + int64_t(i) * q_dim + h * a.hd;
            float t = 0.f;
            for (int d = 0; d < a.hd; ++d) t = fmaf(qr[d], sK[d], t);
            P = expf(a.scale * t - a.lse[int64_t(h) * a.S + i]);
        }
        sPp[threadIdx.x] = P;
        __syncthreads();
        const int n = min(int(blockDim.x), npairs - p0);
        for (int t = 0; t < n; ++t) {
            const int pt = p0 + t;
            const int h = kvh * G + pt / nq, i = i0 + pt % nq;
            const float *dc = a.dctx + int64_t(i) * q_dim + h * a.hd;
#pragma unroll
            for (int k = 0; k < kMaxCols; ++k) {
                const int d = threadIdx.x + k * blockDim.x;
                if (d < a.hd) acc[k] = fmaf(sPp[t], dc[d], acc[k]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int k = 0; k < kMaxCols; ++k) {
        const int d = threadIdx.x + k * blockDim.x;
        if (d < a.hd) a.dv[int64_t(jj) * a.nkv * a.hd + kvh * a.hd + d] = acc[k];
    }
}

// Recomputed attention in the tiled kernels: the 4 x 4 micro-tile of P at query rows
// 4 ty + r and keys 4 tx + c from transposed q and K tiles in shared memory.
template <int HD>
__device__ __forceinline__ void p_tile(const float *sQt, const float *sKt, const float (&lse)[4], float scale,
                                       int q0, int j0, const AttnArgs &a, int tx, int ty, float (&pv)[4][4]) {
    float s[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) s[r][c] = 0.f;
#pragma unroll 4
    for (int d = 0; d < HD; ++d) {
        const float4 qv = *reinterpret_cast<const float4 *>(sQt + d * kTP + 4 * ty);
        const float4 kv = *reinterpret_cast<const float4 *>(sKt + d * kTP + 4 * tx);
        const float qr[4] = {qv.x, qv.y, qv.z, qv.w}, kc[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) s[r][c] = fmaf(qr[r], kc[c], s[r][c]);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int i = q0 + 4 * ty + r;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int j = j0 + 4 * tx + c;          // cache position
            const bool vis = i < a.S && j < a.L && (!a.causal || j <= a.pos0 + i);
            pv[r][c] = vis ? expf(scale * s[r][c] - lse[r]) : 0.f;
        }
    }
}

// [HD][kTP] transposed tile of rows r0 .. r0 + kT of src (row stride ld, head offset
// already applied), zero past nrow.
template <int HD>
__device__ __forceinline__ void load_t(float *dst, const float *src, int64_t ld, int r0, int nrow, int tid) {
    for (int e = tid; e < kT * HD; e += 256) {
        const int i = e / HD, d = e % HD;
        dst[d * kTP + i] = (r0 + i < nrow) ? src[int64_t(r0 + i) * ld + d] : 0.f;
    }
}

// ------------------------------------------------------------------ tiled kernels

// Tiled fp32 attention backward (64 x 64 tiles, 256 threads, 4 x 4 register tiles).
//   attn_dq_tiled: block = (64 query rows, head h).  Pass 1 runs dAttn = dCtx V^T tile by
//     tile and accumulates the row sums D = sum_j P dAttn; pass 2 recomputes dAttn, forms
//     dS = scale P (dAttn - D) and accumulates dQ += dS K; RoPE backward in the epilogue.
//   attn_dv_tiled: block = (64 of the S newest keys, KV head): dV = sum_group P^T dCtx.
// With TLB_CAUSAL, key tiles past the last visible key of a query tile are skipped and the
// masked entries inside a diagonal tile are read as zero, as in the per-row kernels.

template <int HD, bool RC>
__global__ void __launch_bounds__(256) attn_dq_tiled(AttnArgs a, RopeFreqs fr) {
    extern __shared__ float4 sm4[];
    float *sCt = reinterpret_cast<float *>(sm4);        // [HD][kTP]   dCtx tile, transposed
    float *sVt = sCt + HD * kTP;                        // [HD][kTP]   V tile, transposed
    float *sK = sVt + HD * kTP;                         // [kT][HD+4]  K tile
    float *sSt = sK + kT * (HD + 4);                    // [kT][kTP]   dS tile, transposed
    float *sQt = sSt + kT * kTP;                        // RC: [HD][kTP] q tile, transposed
    float *sKt = sQt + HD * kTP;                        // RC: [HD][kTP] K tile, transposed
    __shared__ float sD[kT];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int h = blockIdx.y, kvh = h / (a.nh / a.nkv);
    const int q0 = blockIdx.x * kT;
    const int q_dim = a.nh * HD;
    const int jend = a.causal ? min(a.L, a.pos0 + q0 + kT) : a.L;
    const int nkt = (jend + kT - 1) / kT;
    const float *Vh = a.v + int64_t(kvh) * a.sh, *Kh = a.k + int64_t(kvh) * a.sh;
    const float *Ph = a.attn + int64_t(h) * a.S * a.L;
    // dCtx tile, transposed
    for (int e = tid; e < kT * HD; e += 256) {
        const int i = e / HD, d = e % HD;
        sCt[d * kTP + i] = (q0 + i < a.S) ? a.dctx[int64_t(q0 + i) * q_dim + h * HD + d] : 0.f;
    }
    float lse[4] = {0.f, 0.f, 0.f, 0.f};
    if constexpr (RC) {
        load_t<HD>(sQt, a.q + h * HD, q_dim, q0, a.S, tid);
#pragma unroll
        for (int r = 0; r < 4; ++r)
            lse[r] = q0 + 4 * ty + r < a.S ? a.lse[int64_t(h) * a.S + q0 + 4 * ty + r] : 0.f;
    }
    auto load_vt = [&](int j0) {
        if constexpr (RC) load_t<HD>(sKt, Kh, a.sp, j0, a.L, tid);
        for (int e = tid; e < kT * HD; e += 256) {
            const int j = e / HD, d = e % HD;
            sVt[d * kTP + j] = (j0 + j < a.L) ? Vh[int64_t(j0 + j) * a.sp + d] : 0.f;
        }
    };
    // dAttn micro-tile rows 4ty.., cols 4tx.. of the current key tile
    auto dattn_tile = [&](float (&acc)[4][4]) {
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
#pragma unroll 4
        for (int d = 0; d < HD; ++d) {
            const float4 cv = *reinterpret_cast<const float4 *>(sCt + d * kTP + 4 * ty);
            const float4 vv = *reinterpret_cast<const float4 *>(sVt + d * kTP + 4 * tx);
            const float cr[4] = {cv.x, cv.y, cv.z, cv.w}, vc[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(cr[r], vc[c], acc[r][c]);
        }
    };
    auto load_p = [&](int j0, float (&pv)[4][4]) {
        if constexpr (RC) {
            p_tile<HD>(sQt, sKt, lse, a.scale, q0, j0, a, tx, ty, pv);
            return;
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = q0 + 4 * ty + r;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int j = j0 + 4 * tx + c;
                const bool vis = i < a.S && j < a.L && (!a.causal || j <= a.pos0 + i);
                pv[r][c] = vis ? Ph[int64_t(i) * a.L + j] : 0.f;
            }
        }
    };
    // ---------------- pass 1: D
    float dp[4] = {0.f, 0.f, 0.f, 0.f};
    for (int kt = 0; kt < nkt; ++kt) {
        __syncthreads();
        load_vt(kt * kT);
        __syncthreads();
        float acc[4][4], pv[4][4];
        dattn_tile(acc);
        load_p(kt * kT, pv);
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c) dp[r] = fmaf(pv[r][c], acc[r][c], dp[r]);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        float v = dp[r];
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);   // the 16 tx of this ty
        if (tx == 0) {
            sD[4 * ty + r] = v;
            if (a.D != nullptr && q0 + 4 * ty + r < a.S) a.D[int64_t(h) * a.S + q0 + 4 * ty + r] = v;
        }
    }
    // ---------------- pass 2: dS and dQ
    constexpr int CPT = HD / 16;                 // dQ columns per thread
    float dq[4][CPT];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < CPT; ++c) dq[r][c] = 0.f;
    for (int kt = 0; kt < nkt; ++kt) {
        const int j0 = kt * kT;
        __syncthreads();
        load_vt(j0);
        for (int e = tid; e < kT * HD; e += 256) {
            const int j = e / HD, d = e % HD;
            sK[j * (HD + 4) + d] = (j0 + j < a.L) ? Kh[int64_t(j0 + j) * a.sp + d] : 0.f;
        }
        __syncthreads();
        float acc[4][4], pv[4][4];
        dattn_tile(acc);
        load_p(j0, pv);
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 4; ++c)
                sSt[(4 * tx + c) * kTP + 4 * ty + r] = a.scale * pv[r][c] * (acc[r][c] - sD[4 * ty + r]);
        __syncthreads();
#pragma unroll 4
        for (int j = 0; j < kT; ++j) {
            const float4 sv = *reinterpret_cast<const float4 *>(sSt + j * kTP + 4 * ty);
            const float sr[4] = {sv.x, sv.y, sv.z, sv.w};
            float kv[CPT];
#pragma unroll
            for (int c = 0; c < CPT; c += 2) {
                const float2 t = *reinterpret_cast<const float2 *>(sK + j * (HD + 4) + tx * CPT + c);
                kv[c] = t.x;
                kv[c + 1] = t.y;
            }
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < CPT; ++c) dq[r][c] = fmaf(sr[r], kv[c], dq[r][c]);
        }
    }
    // ---------------- epilogue: RoPE backward through shared memory (pairs d, d + HD/2)
    __syncthreads();
    float *sQ = sK;                                   // [kT][HD+4]
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < CPT; ++c) sQ[(4 * ty + r) * (HD + 4) + tx * CPT + c] = dq[r][c];
    __syncthreads();
    constexpr int half = HD / 2;
    for (int e = tid; e < kT * half; e += 256) {
        const int i = e / half, d = e % half;
        if (q0 + i >= a.S) continue;
        float y1 = sQ[i * (HD + 4) + d], y2 = sQ[i * (HD + 4) + d + half];
        if (a.rope) {
            float cs, sn;
            rope_cos_sin(float(a.pos0 + q0 + i), fr.hi[d], fr.lo[d], cs, sn);
            const float t1 = y1 * cs + y2 * sn, t2 = -y1 * sn + y2 * cs;
            y1 = t1;
            y2 = t2;
        }
        float *out = a.dq + int64_t(q0 + i) * q_dim + h * HD;
        out[d] = y1;
        out[d + half] = y2;
    }
}

template <int HD, bool RC>
__global__ void __launch_bounds__(256) attn_dv_tiled(AttnArgs a) {
    extern __shared__ float4 sm4[];
    float *sP = reinterpret_cast<float *>(sm4);         // [kT][kTP]   P tile [query][key]
    float *sC = sP + kT * kTP;                          // [kT][HD+4]  dCtx tile
    float *sQt = sC + kT * (HD + 4);                    // RC: [HD][kTP] q tile, transposed
    float *sKt = sQt + HD * kTP;                        // RC: [HD][kTP] K tile, transposed
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int kvh = blockIdx.y, G = a.nh / a.nkv;
    const int k0 = blockIdx.x * kT;                     // among the S newest keys
    const int q_dim = a.nh * HD;
    constexpr int CPT = HD / 16;
    float dv[4][CPT];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < CPT; ++c) dv[r][c] = 0.f;
    // query i sees key pos0 + jj iff i >= jj: query tiles from the one holding row k0
    const int qt0 = a.causal ? k0 / kT : 0;
    const int nqt = (a.S + kT - 1) / kT;
    if constexpr (RC) load_t<HD>(sKt, a.k + int64_t(kvh) * a.sh, a.sp, a.pos0 + k0, a.pos0 + a.S, tid);
    for (int g = 0; g < G; ++g) {
        const int h = kvh * G + g;
        const float *Ph = a.attn + int64_t(h) * a.S * a.L + a.pos0;
        for (int qt = qt0; qt < nqt; ++qt) {
            const int q0 = qt * kT;
            __syncthreads();
            if constexpr (RC) {
                load_t<HD>(sQt, a.q + h * HD, q_dim, q0, a.S, tid);
                __syncthreads();
                float lse[4], pv[4][4];
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    lse[r] = q0 + 4 * ty + r < a.S ? a.lse[int64_t(h) * a.S + q0 + 4 * ty + r] : 0.f;
                p_tile<HD>(sQt, sKt, lse, a.scale, q0, a.pos0 + k0, a, tx, ty, pv);
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int c = 0; c < 4; ++c)    // keys past the S newest read as 0
                        sP[(4 * ty + r) * kTP + 4 * tx + c] = k0 + 4 * tx + c < a.S ? pv[r][c] : 0.f;
            } else {
                for (int e = tid; e < kT * kT; e += 256) {
                    const int i = e / kT, j = e % kT;
                    const bool vis = q0 + i < a.S && k0 + j < a.S && (!a.causal || q0 + i >= k0 + j);
                    sP[i * kTP + j] = vis ? Ph[int64_t(q0 + i) * a.L + k0 + j] : 0.f;
                }
            }
            for (int e = tid; e < kT * HD; e += 256) {
                const int i = e / HD, d = e % HD;
                sC[i * (HD + 4) + d] = (q0 + i < a.S) ? a.dctx[int64_t(q0 + i) * q_dim + h * HD + d] : 0.f;
            }
            __syncthreads();
#pragma unroll 4
            for (int i = 0; i < kT; ++i) {
                const float4 pv = *reinterpret_cast<const float4 *>(sP + i * kTP + 4 * ty);
                const float pr[4] = {pv.x, pv.y, pv.z, pv.w};
                float cv[CPT];
#pragma unroll
                for (int c = 0; c < CPT; c += 2) {
                    const float2 t = *reinterpret_cast<const float2 *>(sC + i * (HD + 4) + tx * CPT + c);
                    cv[c] = t.x;
                    cv[c + 1] = t.y;
                }
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int c = 0; c < CPT; ++c) dv[r][c] = fmaf(pr[r], cv[c], dv[r][c]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int jj = k0 + 4 * ty + r;
        if (jj >= a.S) continue;
#pragma unroll
        for (int c = 0; c < CPT; ++c) a.dv[int64_t(jj) * a.nkv * HD + kvh * HD + tx * CPT + c] = dv[r][c];
    }
}

template <int HD, bool RC>
int launch_tiled_rc(const AttnArgs &a, const RopeFreqs &fr, cudaStream_t st) {
    const size_t rc = RC ? size_t(2) * HD * kTP : 0;     // transposed q and K tiles
    const size_t smq = (size_t(2) * HD * kTP + size_t(kT) * (HD + 4) + size_t(kT) * kTP + rc) * 4;
    const size_t smv = (size_t(kT) * kTP + size_t(kT) * (HD + 4) + rc) * 4;
    if (smq > 48 * 1024)
        TLB_CUDA(cudaFuncSetAttribute(attn_dq_tiled<HD, RC>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smq)));
    if (smv > 48 * 1024)
        TLB_CUDA(cudaFuncSetAttribute(attn_dv_tiled<HD, RC>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smv)));
    attn_dq_tiled<HD, RC><<<dim3(unsigned(ceil_div(a.S, kT)), unsigned(a.nh)), 256, smq, st>>>(a, fr);
    TLB_TRY(check_launch("attn_dq_tiled"));
    attn_dv_tiled<HD, RC><<<dim3(unsigned(ceil_div(a.S, kT)), unsigned(a.nkv)), 256, smv, st>>>(a);
    return check_launch("attn_dv_tiled");
}

template <int HD>
int launch_tiled(const AttnArgs &a, const RopeFreqs &fr, cudaStream_t st) {
    return a.lse != nullptr ? launch_tiled_rc<HD, true>(a, fr, st) : launch_tiled_rc<HD, false>(a, fr, st);
}

int attn_core_launch(const AttnArgs &a, float rope_base, cudaStream_t st) {
    if (a.S == 0) return TLB_OK;
    RopeFreqs fr;
    rope_freqs(fr, a.hd, rope_base);
    if (a.S > 1) {
        if (a.hd == 128) return launch_tiled<128>(a, fr, st);
        if (a.hd == 64) return launch_tiled<64>(a, fr, st);
        if (a.hd == 32) return launch_tiled<32>(a, fr, st);
    }
    const size_t smem = (size_t(a.L) + 2 * size_t(a.hd) + (a.lse != nullptr ? size_t(a.L) + a.hd : 0)) * sizeof(float);
    TLB_REQUIRE(smem <= 200 * 1024, TLB_EUNSUPPORTED, "attn_backward: cache length %d too long", a.L);
    if (smem > 48 * 1024)
        TLB_CUDA(cudaFuncSetAttribute(attn_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      int(smem)));
    attn_rows_kernel<<<dim3(a.S, a.nh), 128, smem, st>>>(a, fr);
    TLB_TRY(check_launch("attn_rows"));
    if (a.lse != nullptr) {
        attn_dv_rc_kernel<<<dim3(a.S, a.nkv), 128, (size_t(a.hd) + 128) * 4, st>>>(a);
        return check_launch("attn_dv_rc");
    }
    attn_dv_kernel<<<dim3(a.S, a.nkv), a.hd < 128 ? a.hd : 128, 0, st>>>(a);
    return check_launch("attn_dv");
}


// ------------------------------------------------------------------ key gradient (exact d_in)

// Any shape: one block per (new key jj, KV head).  The dS values of up to blockDim (head,
// query) pairs at a time are formed one pair per thread (a dot over head_dim), then every
// thread adds their share into the head_dim columns it owns.
__global__ void attn_dk_rows_kernel(AttnArgs a, const float *__restrict__ q, const float *__restrict__ Dv,
                                    float *dk) {
    extern __shared__ float4 smem4[];
    float *sV = reinterpret_cast<float *>(smem4);      // [hd] V row of the key
    float *sDs = sV + a.hd;                            // [blockDim] dS of the current pairs
    const int jj = blockIdx.x, kvh = blockIdx.y, G = a.nh / a.nkv;
    const int j = a.pos0 + jj, q_dim = a.nh * a.hd;
    const int i0 = a.causal ? jj : 0;                   // query i sees key pos0 + jj iff i >= jj
    const int nq = a.S - i0, npairs = G * nq;
    const float *Vj = a.v + int64_t(kvh) * a.sh + int64_t(j) * a.sp;
    const float *Kj = a.k + int64_t(kvh) * a.sh + int64_t(j) * a.sp;
    float *sK = sDs + blockDim.x;                      // recompute: [hd] K row of the key
    const bool rc = a.lse != nullptr;
    for (int d = threadIdx.x; d < a.hd; d += blockDim.x) {
        sV[d] = Vj[d];
        if (rc) sK[d] = Kj[d];
    }
    constexpr int kMaxCols = 2;                         // head_dim <= 256, blockDim >= 128
    float acc[kMaxCols] = {0.f, 0.f};
    __syncthreads();
    for (int p0 = 0; p0 < npairs; p0 += blockDim.x) {
        const int pp = p0 + threadIdx.x;
        float ds = 0.f;
        if (pp < npairs) {
            const int h = kvh * G + pp / nq, i = i0 + pp % nq;
            float P;
            if (rc) {
                const float *qr = q + int64_t(i) * q_dim + h * a.hd;
                float t = 0.f;
                for (int d = 0; d < a.hd; ++d) t = fmaf(qr[d], sK[d], t);
                P = expf(a.scale * t - a.lse[int64_t(h) * a.S + i]);
            } else {
                P = a.attn[(int64_t(h) * a.S + i) * a.L + j];
            }
            const float *dc = a.dctx + int64_t(i) * q_dim + h * a.hd;
            float t = 0.f;
            for (int d = 0; d < a.hd; ++d) t = fmaf(dc[d], sV[d], t);
            ds = P * (t - Dv[int64_t(h) * a.S + i]);
        }
        sDs[threadIdx.x] = ds;
        __syncthreads();
        const int n = min(int(blockDim.x), npairs - p0);
        for (int t = 0; t < n; ++t) {
            const int pt = p0 + t;
            const int h = kvh * G + pt / nq, i = i0 + pt % nq;
            const float *qr = q + int64_t(i) * q_dim + h * a.hd;
            const float s = sDs[t];
#pragma unroll
            for (int k = 0; k < kMaxCols; ++k) {
                const int d = threadIdx.x + k * blockDim.x;
                if (d < a.hd) acc[k] = fmaf(s, qr[d], acc[k]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int k = 0; k < kMaxCols; ++k) {
        const int d = threadIdx.x + k * blockDim.x;
        if (d < a.hd) dk[int64_t(jj) * a.nkv * a.hd + kvh * a.hd + d] = a.scale * acc[k];
    }
}

// S > 1, head_dim 32 / 64 / 128: block = (64 new keys, KV head), 256 threads.  For every
// head of the group and query tile: T = dCtx V^T on the tile (4 x 4 per thread, from
// transposed tiles so that each step is two 16-byte shared loads), dS = P (T - D) in
// shared memory, then dK += dS^T q (4 keys x HD/16 columns per thread).
template <int HD, bool RC>
__global__ void __launch_bounds__(256) attn_dk_tiled(AttnArgs a, const float *__restrict__ q,
                                                     const float *__restrict__ Dv, float *dk) {
    extern __shared__ float4 sm4[];
    float *sVt = reinterpret_cast<float *>(sm4);        // [HD][kTP]   V rows of the key tile, transposed
    float *sCt = sVt + HD * kTP;                        // [HD][kTP]   dCtx tile, transposed
    float *sQ = sCt + HD * kTP;                         // [kT][HD+4]  q tile [query][d]
    float *sS = sQ + kT * (HD + 4);                     // [kT][kTP]   dS tile [query][key]
    float *sQt = sS + kT * kTP;                         // RC: [HD][kTP] q tile, transposed
    float *sKt = sQt + HD * kTP;                        // RC: [HD][kTP] K rows of the key tile, transposed
    __shared__ float sDq[kT];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int kvh = blockIdx.y, G = a.nh / a.nkv, g = blockIdx.z;   // one head of the group per block
    const int k0 = blockIdx.x * kT;                     // among the S newest keys
    const int q_dim = a.nh * HD;
    constexpr int CPT = HD / 16;
    for (int e = tid; e < kT * HD; e += 256) {
        const int j = e / HD, d = e % HD;
        sVt[d * kTP + j] =
            (k0 + j < a.S) ? a.v[int64_t(kvh) * a.sh + int64_t(a.pos0 + k0 + j) * a.sp + d] : 0.f;
    }
    float acc[4][CPT];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < CPT; ++c) acc[r][c] = 0.f;
    const int qt0 = a.causal ? k0 / kT : 0;
    const int nqt = (a.S + kT - 1) / kT;
    if constexpr (RC) load_t<HD>(sKt, a.k + int64_t(kvh) * a.sh, a.sp, a.pos0 + k0, a.pos0 + a.S, tid);
    {
        const int h = kvh * G + g;
        const float *Ph = a.attn + int64_t(h) * a.S * a.L + a.pos0;
        for (int qt = qt0; qt < nqt; ++qt) {
            const int q0 = qt * kT;
            __syncthreads();
            for (int e = tid; e < kT * HD; e += 256) {
                const int i = e / HD, d = e % HD;
                const bool in = q0 + i < a.S;
                sCt[d * kTP + i] = in ? a.dctx[int64_t(q0 + i) * q_dim + h * HD + d] : 0.f;
                sQ[i * (HD + 4) + d] = in ? q[int64_t(q0 + i) * q_dim + h * HD + d] : 0.f;
            }
            if (tid < kT) sDq[tid] = q0 + tid < a.S ? Dv[int64_t(h) * a.S + q0 + tid] : 0.f;
            if constexpr (RC) load_t<HD>(sQt, q + h * HD, q_dim, q0, a.S, tid);
            __syncthreads();
            float pv[4][4];
            if constexpr (RC) {
                float lse[4];
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    lse[r] = q0 + 4 * ty + r < a.S ? a.lse[int64_t(h) * a.S + q0 + 4 * ty + r] : 0.f;
                p_tile<HD>(sQt, sKt, lse, a.scale, q0, a.pos0 + k0, a, tx, ty, pv);
            }
            // T[i][j] for query rows 4 ty + r and keys 4 tx + c
            float t[4][4];
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) t[r][c] = 0.f;
#pragma unroll 8
            for (int d = 0; d < HD; ++d) {
                const float4 cq = *reinterpret_cast<const float4 *>(sCt + d * kTP + 4 * ty);
                const float4 vk = *reinterpret_cast<const float4 *>(sVt + d * kTP + 4 * tx);
                const float cr[4] = {cq.x, cq.y, cq.z, cq.w}, vc[4] = {vk.x, vk.y, vk.z, vk.w};
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int c = 0; c < 4; ++c) t[r][c] = fmaf(cr[r], vc[c], t[r][c]);
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int i = q0 + 4 * ty + r;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int jk = k0 + 4 * tx + c;
                    const bool vis = i < a.S && jk < a.S && (!a.causal || i >= jk);
                    float P;
                    if constexpr (RC) P = jk < a.S ? pv[r][c] : 0.f;
                    else P = vis ? Ph[int64_t(i) * a.L + jk] : 0.f;
                    sS[(4 * ty + r) * kTP + 4 * tx + c] = P * (t[r][c] - sDq[4 * ty + r]);
                }
            }
            __syncthreads();
#pragma unroll 4
            for (int i = 0; i < kT; ++i) {
                const float4 sv = *reinterpret_cast<const float4 *>(sS + i * kTP + 4 * ty);
                const float sr[4] = {sv.x, sv.y, sv.z, sv.w};
                float qv[CPT];
#pragma unroll
                for (int c = 0; c < CPT; c += 2) {
                    const float2 u = *reinterpret_cast<const float2 *>(sQ + i * (HD + 4) + tx * CPT + c);
                    qv[c] = u.x;
                    qv[c + 1] = u.y;
                }
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int c = 0; c < CPT; ++c) acc[r][c] = fmaf(sr[r], qv[c], acc[r][c]);
            }
        }
    }
    // this head's share: dk holds [G][S, kv_dim] partials, added in head order afterwards
    float *out = dk + int64_t(g) * a.S * a.nkv * HD;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int jj = k0 + 4 * ty + r;
        if (jj >= a.S) continue;
#pragma unroll
        for (int c = 0; c < CPT; ++c) out[int64_t(jj) * a.nkv * HD + kvh * HD + tx * CPT + c] = a.scale * acc[r][c];
    }
}

// dk[e] = sum over the group's heads g (in order) of part[g][e]
__global__ void attn_dk_sum_kernel(const float *__restrict__ part, float *dk, int64_t n, int G) {
    for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < n; e += int64_t(gridDim.x) * blockDim.x) {
        float s = part[e];
        for (int g = 1; g < G; ++g) s += part[int64_t(g) * n + e];
        dk[e] = s;
    }
}

template <int HD, bool RC>
int launch_dk_tiled_rc(const AttnArgs &a, const float *q, const float *D, float *dst, cudaStream_t st) {
    const int G = a.nh / a.nkv;
    const size_t sm = (size_t(RC ? 4 : 2) * HD * kTP + size_t(kT) * (HD + 4) + size_t(kT) * kTP) * 4;
    if (sm > 48 * 1024)
        TLB_CUDA(cudaFuncSetAttribute(attn_dk_tiled<HD, RC>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sm)));
    attn_dk_tiled<HD, RC><<<dim3(unsigned(ceil_div(a.S, kT)), unsigned(a.nkv), unsigned(G)), 256, sm, st>>>(a, q, D,
                                                                                                          dst);
    return check_launch("attn_dk_tiled");
}

template <int HD>
int launch_dk_tiled(const AttnArgs &a, const float *q, const float *D, float *dk, float *part, cudaStream_t st) {
    const int G = a.nh / a.nkv;
    float *dst = G > 1 ? part : dk;
    if (a.lse != nullptr) TLB_TRY((launch_dk_tiled_rc<HD, true>(a, q, D, dst, st)));
    else TLB_TRY((launch_dk_tiled_rc<HD, false>(a, q, D, dst, st)));
    if (G == 1) return TLB_OK;
    const int64_t n = int64_t(a.S) * a.nkv * HD;
    attn_dk_sum_kernel<<<stream_grid(n, 256), 256, 0, st>>>(part, dk, n, G);
    return check_launch("attn_dk_sum");
}

size_t attn_dk_bytes(int64_t S, int nh, int nkv, int hd) {
    return nh > nkv ? size_t(nh) * S * hd * 4 : 0;     // per-head partials of the tiled kernel
}

int attn_dk_launch(const AttnArgs &a, const float *q, const float *D, float *dk, float *part, cudaStream_t st) {
    if (a.S == 0) return TLB_OK;
    if (a.S > 1) {
        if (a.hd == 128) return launch_dk_tiled<128>(a, q, D, dk, part, st);
        if (a.hd == 64) return launch_dk_tiled<64>(a, q, D, dk, part, st);
        if (a.hd == 32) return launch_dk_tiled<32>(a, q, D, dk, part, st);
    }
    const int threads = 128;
    attn_dk_rows_kernel<<<dim3(unsigned(a.S), unsigned(a.nkv)), threads, (size_t(2 * a.hd) + threads) * 4, st>>>(
        a, q, D, dk);
    return check_launch("attn_dk_rows");
}

}  // namespace tlb
