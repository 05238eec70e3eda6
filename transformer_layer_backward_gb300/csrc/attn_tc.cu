// Tensor-core attention backward for sequences ([ATT] "Gradient Flow": apply, softmax,
// score and RoPE backward; [RS] backward_through_layers, attention block), with tf32
// operands and fp32 accumulation in tensor memory.  GQA: kvh = h / (nh / nkv).
//
//   attn_tc_prep  tf32-rounded copies laid out for TMA (32 x 32 tile transposes):
//                   dCT [nh][hd][S4]   Kt [nkv][hd][L4]   Vr [nkv][L][hd]
//                 and the RoPE (cos, sin) table of the S new positions.  dCT is skipped
//                 when the O-projection product has written it from its epilogue; the
//                 dQ kernel then loads its dCtx rows from dCT too.
//   attn_tc_dq    CTA = (head h, 128 queries), 10 warps: TMA producer, MMA issuer, and
//                 8 epilogue warps in two groups that take alternate key tiles (one query
//                 row = one TMEM lane per thread).  dCtx_h sits in tensor memory as the A
//                 operand of T; E replaces T in its tensor-memory buffer (two buffers) and
//                 is the A operand of U; the staged P tile is the A operand of W.  Per tile
//                 of 64 keys j (V_j, K_j^T and the P tile arrive by TMA in two rings, two
//                 tiles deep: V is released when T_j is formed, K^T and P after U and W):
//                   T  = dCtx_h V_j^T                        tcgen05.mma, T in TMEM
//                   E  = P (.) T,  D += rowsum(E)            epilogue, fp32
//                   U += E K_j,    W += P K_j                tcgen05.mma (E tf32 in TMEM, P in smem)
//                 then dQ = scale (U - D W), which equals scale sum_j P (T - D) K_j with D
//                 the literal row sum of P (.) dAttn, and RoPE backward on the way out.
//   attn_tc_dv    CTA = (head h, 128 of the S newest keys), two CTAs per SM: over 32-query
//                 items, dV_h += P_h^T dCtx_h.  P tiles come by TMA and the writer warps
//                 put them transposed (tf32) into tensor memory as the A operand;
//                 dCtx^T tiles (B) by TMA; three items in flight.  With
//                 several heads per KV head the per-head sums go to a workspace and
//                 attn_tc_dv_sum adds them in head order.
// All MMAs: M = 128, K = 8 per instruction, both operands K-major with 128-byte swizzle.
// Causal: key tiles past a query tile's last visible key are skipped; masked entries of
// P inside a diagonal tile read as zero.  Every mbarrier wait is bounded.
#include <cuda.h>

#include <cstring>

#include "async.cuh"
#include "common.cuh"
#include "kernels.cuh"
#include "tc.cuh"

namespace tlb {

namespace {

constexpr int kQM = 128;        // queries per dQ CTA
constexpr int kQK = 64;         // keys per dQ tile (two 32-key swizzle atoms)
constexpr int kQSlots = 2;      // dQ tiles in flight (V, K^T, P staged up to two tiles ahead)
constexpr int kVK = 128;        // keys per dV CTA
constexpr int kVQ = 32;         // queries per dV item
constexpr int kVSlots = 3;      // dV items staged ahead (P tile and dCtx^T tile rings)
constexpr int kAttnThreads = 320;    // producer warp, MMA warp, 8 epilogue warps
constexpr int kEpiWarps = 8;          // two per TMEM lane quarter, each half of the columns

struct AttnTcParams {
    CUtensorMap v;              // Vr   {hd, L, nkv}, box {32, 32, 1}
    CUtensorMap kt;             // Kt   {L, hd, nkv}, box {32, hd, 1}
    CUtensorMap dct;            // dCT  {S, hd, nh},  box {32, hd, 1}
    CUtensorMap pq;             // attn {L, S, nh},   box {32, 128, 1}   (dQ: 128 queries x 32 keys)
    CUtensorMap pv;             // attn {L, S, nh},   box {32, 32, 1}    (dV: 32 queries x 32 keys)
    const float *dctx;          // dCtx [S, nh * hd], or null: the dQ kernel reads dcT instead
    const float *dcT;           // the tf32 dCtx^T [nh * hd][ld_ct] in the scratch
    int ld_ct;
    float *dq;                  // [S, nh * hd]
    float *dv;                  // [S, nkv * hd], or per-head partial sums [nh / nkv][S, nkv * hd]
    int S, L, nh, nkv, pos0, causal, rope;
    float scale;
    uint32_t *status;
    float *D;                   // [nh, S] row sums D (optional)
    const float2 *rt;           // [S][hd / 2] (cos, sin) of the RoPE angles of positions pos0 + i
};

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void st_shared_v4(uint8_t *p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(p)), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// 2^x by the special-function unit (relative error near 2^-22; results below the normal
// range flush to zero).  The recomputed attention weights go through it as
// exp(scale s - lse) = 2^(scale log2(e) s - lse log2(e)), then to tf32 (2^-11).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
constexpr float kLog2e = 1.4426950408889634f;

// Byte offset of 16-byte chunk `ch` (0..7) of row r in a K-major 128-byte-swizzled box.
__device__ __forceinline__ uint32_t sw128_off(int r, int ch) { return uint32_t(r) * 128u + (uint32_t(ch ^ (r & 7)) << 4); }

// ------------------------------------------------------------------ prep

// 64 x 64 tiles of three sources, every value rounded to tf32:
//   dCtx [S, nh*hd] -> dCT [nh*hd][S4] (transposed);  K -> Kt [nkv*hd][L4] (transposed);
//   V -> Vr [nkv][L][hd].
// Each thread loads four float4 of its tile (16-byte loads of rows of 64 floats); a
// transposed tile goes out through shared memory, one warp writing 32 consecutive floats
// of an output row per store, and V is written straight from the registers.  vec_kv:
// K and V rows allow 16-byte loads (else those two load one float at a time).
constexpr int kPrepT = 64;
__global__ void __launch_bounds__(256) attn_tc_prep_kernel(AttnArgs a, float *dCT, float *Kt, float *Vr,
                                                           int S4, int L4, int nt_dc, int nt_kv, int vec_kv,
                                                           const __grid_constant__ RopeFreqs fr, float2 *rt,
                                                           float *Kr) {
    __shared__ float tile[kPrepT][kPrepT + 1];
    const int qd = a.nh * a.hd, kvd = a.nkv * a.hd;
    const int nkvj = Kr != nullptr ? 3 : 2;        // K^T, V rows, and the K rows when recomputing
    int t = blockIdx.x;
    if (t >= nt_dc + nkvj * nt_kv) {
        // the RoPE table: (cos, sin) of (pos0 + i) f_d for the S new positions, the angles
        // every head's dQ epilogue rotates by
        const int hh = a.hd / 2;
        const int64_t e0 = int64_t(t - nt_dc - nkvj * nt_kv) * 1024, n = int64_t(a.S) * hh;
        for (int k = 0; k < 4; ++k) {
            const int64_t e = e0 + threadIdx.x + 256 * k;
            if (e >= n) break;
            const int i = int(e / hh), d = int(e % hh);
            float c, sn;
            rope_cos_sin(float(a.pos0 + i), fr.hi[d], fr.lo[d], c, sn);
            rt[e] = make_float2(c, sn);
        }
        return;
    }
    int job, rows, cols;
    if (t < nt_dc) {
        job = 0;
        rows = a.S;
        cols = qd;
    } else {
        t -= nt_dc;
        job = t / nt_kv + 1;                       // 1: K^T, 2: V rows, 3: K rows
        t %= nt_kv;
        rows = a.L;
        cols = kvd;
    }
    const int nct = cols / kPrepT;
    const int r0 = (t / nct) * kPrepT, c0 = (t % nct) * kPrepT;
    const int tid = threadIdx.x;
    float4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int e = tid + 256 * k, rr = e >> 4, c = c0 + 4 * (e & 15), r = r0 + rr;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < rows) {
            if (job == 0) {
                x = *reinterpret_cast<const float4 *>(a.dctx + int64_t(r) * qd + c);
            } else {
                const int kvh = c / a.hd, d = c % a.hd;
                const float *src = (job == 2 ? a.v : a.k) + int64_t(kvh) * a.sh + int64_t(r) * a.sp + d;
                if (vec_kv) x = *reinterpret_cast<const float4 *>(src);
                else x = make_float4(src[0], src[1], src[2], src[3]);
            }
        }
        v[k] = make_float4(__uint_as_float(to_tf32(x.x)), __uint_as_float(to_tf32(x.y)),
                           __uint_as_float(to_tf32(x.z)), __uint_as_float(to_tf32(x.w)));
    }
    if (job >= 2) {
        float *rows_out = job == 2 ? Vr : Kr;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int e = tid + 256 * k, rr = e >> 4, c = c0 + 4 * (e & 15), r = r0 + rr;
            if (r < rows) {
                const int hh = c / a.hd, d = c % a.hd;
                *reinterpret_cast<float4 *>(rows_out + (int64_t(hh) * a.L + r) * a.hd + d) = v[k];
            }
        }
        return;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int e = tid + 256 * k, rr = e >> 4, cc = 4 * (e & 15);
        tile[rr][cc] = v[k].x;
        tile[rr][cc + 1] = v[k].y;
        tile[rr][cc + 2] = v[k].z;
        tile[rr][cc + 3] = v[k].w;
    }
    __syncthreads();
    // transposed: output row c0 + cc (head, d), columns r0 + 0 .. 63; lane = column
    float *dst = job == 0 ? dCT : Kt;
    const int ld = job == 0 ? S4 : L4;
    const int lane = tid & 31, w = tid >> 5;
#pragma unroll 4
    for (int k = 0; k < (kPrepT * kPrepT) / 256; ++k) {
        const int cc = w + 8 * (k >> 1), rr = lane + 32 * (k & 1), r = r0 + rr;
        if (r < rows) dst[int64_t(c0 + cc) * ld + r] = tile[rr][cc];
    }
}

// ------------------------------------------------------------------ dQ

template <int HD>
struct DqLayout {
    static constexpr int NB = HD / 32;                   // 128-byte boxes along head_dim
    static constexpr int NA = kQK / 32;                  // 32-key swizzle atoms of a tile
    // shared memory: two rings of kQSlots slots each, V_j (freed once T_j is formed) and
    // {K_j^T, P tile} (freed once U and W have taken tile j).  K^T and P are NA atoms of
    // 32 keys each (rows of 128 bytes), side by side.
    static constexpr int V_BYTES = kQK * HD * 4, KT_BYTES = HD * kQK * 4, P_BYTES = kQM * kQK * 4;
    static constexpr int KT_ATOM = HD * 128, P_ATOM = kQM * 128;
    static constexpr int KSLOT = KT_BYTES + P_BYTES;
    static constexpr int K0 = kQSlots * V_BYTES;
    static constexpr int TOTAL = K0 + kQSlots * KSLOT;
    __host__ __device__ static constexpr int V(int s) { return s * V_BYTES; }
    __host__ __device__ static constexpr int KT(int s) { return K0 + s * KSLOT; }
    __host__ __device__ static constexpr int P(int s) { return K0 + s * KSLOT + KT_BYTES; }
    // tensor memory columns: dCtx (A of T), the T double buffer, U, W.  E_j replaces T_j
    // in its buffer and is the A operand of U; T_j+2 goes there once U_j has completed.
    static constexpr uint32_t TDC = 0, TT = HD, TU = HD + 2 * kQK, TW = TU + HD;
    static constexpr uint32_t COLS = (TW + HD) <= 256 ? 256 : 512;
};

template <int HD>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_tc_dq_kernel(const __grid_constant__ AttnTcParams p) {
    using Ly = DqLayout<HD>;
    constexpr int NB = Ly::NB;
    static_assert(Ly::TW + HD <= 512 && kQK % 32 == 0, "tensor memory");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    // vfull/vfree: V ring; kfull/kfree: K^T + P ring; dcready: dCtx in TMEM; tfull: T_j in
    // its buffer; afull: E_j written over it (and the masked P tile in shared memory);
    // afree: U_j has read E_j, so T_j+2 may take the buffer.  Per buffer, double-buffered.
    __shared__ uint64_t vfull[kQSlots], vfree[kQSlots], kfull[kQSlots], kfree[kQSlots], dcready, tfull[2], afull[2],
        afree[2], ufull;
    __shared__ uint32_t tmem_base;
    __shared__ int s_abort, s_v_issued, s_v_used, s_k_issued, s_k_used;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // blocks start in x-fastest order: x = head, y = query tile from the last (longest) one,
    // so every head's longest tiles start first
    const int h = blockIdx.x, kvh = h / (p.nh / p.nkv);
    const int q0 = int(gridDim.y - 1 - blockIdx.y) * kQM;
    const int kend = p.causal ? min(p.L, p.pos0 + q0 + kQM) : p.L;
    const int nt = (kend + kQK - 1) / kQK;

    if (threadIdx.x == 0) {
        s_abort = 0;
        s_v_issued = s_v_used = s_k_issued = s_k_used = 0;
        for (int s = 0; s < kQSlots; ++s) {
            mbar_init(&vfull[s], 1);
            mbar_init(&vfree[s], 1);
            mbar_init(&kfull[s], 1);
            mbar_init(&kfree[s], 1);
        }
        mbar_init(&dcready, kEpiWarps);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&afull[b], kEpiWarps / 2);    // the four warps of the group that forms E_j
            mbar_init(&afree[b], 1);
        }
        mbar_init(&ufull, 1);
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base, Ly::COLS);
        tmem_relinquish();
    }
    fence_mbar_init();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (kQSlots tiles ahead)
        if (lane == 0) {
            for (int j = 0; j < nt; ++j) {
                const int s = j % kQSlots, k0 = j * kQK;
                // V slot: tile j - kQSlots has formed its T; K^T + P slot: its U and W are done
                if (j >= kQSlots && !mbar_wait(&vfree[s], (j / kQSlots - 1) & 1, p.status, 20u)) {
                    s_abort = 1;
                    break;
                }
                mbar_arrive_expect_tx(&vfull[s], Ly::V_BYTES);
                for (int b = 0; b < NB; ++b)
                    tma_load_3d(sm + Ly::V(s) + b * (kQK * 128), &p.v, b * 32, k0, kvh, &vfull[s]);
                s_v_issued = j + 1;
                if (j >= kQSlots && !mbar_wait(&kfree[s], (j / kQSlots - 1) & 1, p.status, 21u)) {
                    s_abort = 1;
                    break;
                }
                mbar_arrive_expect_tx(&kfull[s], Ly::KSLOT);
                for (int a = 0; a < Ly::NA; ++a) {
                    tma_load_3d(sm + Ly::KT(s) + a * Ly::KT_ATOM, &p.kt, k0 + 32 * a, 0, kvh, &kfull[s]);
                    tma_load_3d(sm + Ly::P(s) + a * Ly::P_ATOM, &p.pq, k0 + 32 * a, q0, h, &kfull[s]);
                }
                s_k_issued = j + 1;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t id1 = idesc_tf32(kQM, kQK), id2 = idesc_tf32(kQM, HD);
            auto mma_t = [&](int j) -> bool {            // T[j % 2] = dCtx V_j^T, dCtx from TMEM
                const int s = j % kQSlots;
                if (!mbar_wait(&vfull[s], (j / kQSlots) & 1, p.status, 22u)) return false;
                s_v_used = j + 1;
                tc_fence_after();
                const uint8_t *b = sm + Ly::V(s);
#pragma unroll
                for (int kb = 0; kb < NB; ++kb)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_tf32_ts(tmem + Ly::TT + uint32_t((j & 1) * kQK), tmem + Ly::TDC + uint32_t(kb * 32 + k * 8),
                                    sw128_desc(b + kb * (kQK * 128)) + 2 * k, id1, (kb | k) ? 1u : 0u);
                mma_commit(&vfree[s]);
                mma_commit(&tfull[j & 1]);
                return true;
            };
            bool ok = mbar_wait(&dcready, 0, p.status, 23u);
            tc_fence_after();
            ok = ok && mma_t(0) && (nt < 2 || mma_t(1));
            for (int j = 0; ok && j < nt; ++j) {
                const int s = j % kQSlots;
                if (!mbar_wait(&afull[j & 1], (j >> 1) & 1, p.status, 24u) ||
                    !mbar_wait(&kfull[s], (j / kQSlots) & 1, p.status, 25u)) {
                    ok = false;
                    break;
                }
                s_k_used = j + 1;
                tc_fence_after();
                const uint32_t te = tmem + Ly::TT + uint32_t((j & 1) * kQK);    // E_j, where T_j was
                // U_j first and its commit, then W_j: the wait for U_j below (before T_j+2 may
                // take E_j's buffer) overlaps W_j in the tensor pipe instead of draining it
#pragma unroll
                for (int a = 0; a < Ly::NA; ++a) {
                    const uint64_t kd = sw128_desc(sm + Ly::KT(s) + a * Ly::KT_ATOM);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_tf32_ts(tmem + Ly::TU, te + uint32_t(32 * a + 8 * k), kd + 2 * k, id2,
                                    (j > 0 || a > 0 || k > 0) ? 1u : 0u);
                }
                mma_commit(&afree[j & 1]);
#pragma unroll
                for (int a = 0; a < Ly::NA; ++a) {
                    const uint64_t kd = sw128_desc(sm + Ly::KT(s) + a * Ly::KT_ATOM);
                    const uint64_t pd = sw128_desc(sm + Ly::P(s) + a * Ly::P_ATOM);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_tf32(tmem + Ly::TW, pd + 2 * k, kd + 2 * k, id2, (j > 0 || a > 0 || k > 0) ? 1u : 0u);
                }
                mma_commit(&kfree[s]);
                // T_j+2 overwrites E_j: issue it once U_j has read E_j
                if (j + 2 < nt) {
                    if (!mbar_wait(&afree[j & 1], (j >> 1) & 1, p.status, 28u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (!(ok = mma_t(j + 2))) break;
                }
            }
            if (!ok) s_abort = 1;
            mma_commit(&ufull);                     // fires once every MMA issued above is complete
            mbar_wait(&ufull, 0, nullptr, 0u);
        }
    } else {
        // ------------------------------------------------ epilogue: two groups of four warps (one
        // per TMEM lane quarter), one query row per thread
        const int quarter = warp & 3, hf = (warp - 2) >> 2;
        const int r = quarter * 32 + lane, i = q0 + r;
        const bool row_ok = i < p.S;
        const uint32_t lane_off = uint32_t(quarter * 32) << 16;
        const int jlast = p.causal ? p.pos0 + i : p.L - 1;      // last visible key
        {   // this row's half of dCtx_h, rounded to tf32, into tensor memory: the A operand of T
            float4 x[HD / 8];                    // every load in flight before the first store
            if (p.dctx != nullptr) {
                const float4 *src = reinterpret_cast<const float4 *>(p.dctx + int64_t(row_ok ? i : 0) * (p.nh * HD) +
                                                                     h * HD + hf * (HD / 2));
#pragma unroll
                for (int k = 0; k < HD / 8; ++k) x[k] = row_ok ? src[k] : make_float4(0.f, 0.f, 0.f, 0.f);
            } else {
                // from the tf32 dCtx^T (already rounded; rounding again changes nothing): for
                // each column the warp's lanes read 32 consecutive rows, 128 contiguous bytes
                const float *src = p.dcT + int64_t(h * HD + hf * (HD / 2)) * p.ld_ct + (row_ok ? i : 0);
#pragma unroll
                for (int k = 0; k < HD / 8; ++k) {
                    const float *c4 = src + int64_t(4 * k) * p.ld_ct;
                    x[k] = row_ok ? make_float4(c4[0], c4[p.ld_ct], c4[2 * p.ld_ct], c4[3 * p.ld_ct])
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
#pragma unroll
            for (int c = 0; c < HD / 2; c += 16) {
                uint32_t v[16];
#pragma unroll
                for (int t = 0; t < 16; t += 4) {
                    const float4 y = x[(c + t) / 4];
                    v[t] = to_tf32(y.x);
                    v[t + 1] = to_tf32(y.y);
                    v[t + 2] = to_tf32(y.z);
                    v[t + 3] = to_tf32(y.w);
                }
                tmem_st16(tmem + Ly::TDC + uint32_t(hf * (HD / 2) + c) + lane_off, v);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&dcready);
        }
        // Key tiles alternate between the two groups of four warps (group hf takes the tiles
        // j = hf mod 2 and with them T / E buffer hf), each thread one query row and all of
        // the tile's columns, so that one group forms E_j while the other forms E_j+1.
        float D = 0.f;
        bool ok = true;
        for (int j = hf; j < nt; j += 2) {
            const int s = j % kQSlots, k0 = j * kQK;
            if (!mbar_wait(&kfull[s], (j / kQSlots) & 1, p.status, 26u) ||
                !mbar_wait(&tfull[j & 1], (j >> 1) & 1, p.status, 27u)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // T_j -> E_j in place, one 32-key atom at a time.  The buffer is free: T_j was
            // issued only after U_j-2 had read E_j-2 from it.
            const uint32_t tb = tmem + Ly::TT + uint32_t((j & 1) * kQK) + lane_off;
#pragma unroll 1
            for (int a = 0; a < Ly::NA; ++a) {
                uint32_t t[32];
                tmem_ld32(tb + uint32_t(32 * a), t);
                uint8_t *pt = sm + Ly::P(s) + a * Ly::P_ATOM;
                float pv[32];
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const float4 v = *reinterpret_cast<const float4 *>(pt + sw128_off(r, ch));
                    pv[4 * ch] = v.x;
                    pv[4 * ch + 1] = v.y;
                    pv[4 * ch + 2] = v.z;
                    pv[4 * ch + 3] = v.w;
                }
                const int ka = k0 + 32 * a;
                const bool diag = ka + 31 > jlast;               // masked keys in this row of the atom
                if (diag) {
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        if (ka + c > jlast) pv[c] = 0.f;
                }
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const float e = pv[c] * __uint_as_float(t[c]);
                    D += e;
                    t[c] = to_tf32(e);
                }
                // the P tile is the A operand of W += P K_j as staged (the MMA reads tf32);
                // masked keys of a diagonal tile are zeroed in place
                if (diag) {
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch)
                        st_shared_v4(pt + sw128_off(r, ch), __float_as_uint(pv[4 * ch]),
                                     __float_as_uint(pv[4 * ch + 1]), __float_as_uint(pv[4 * ch + 2]),
                                     __float_as_uint(pv[4 * ch + 3]));
                    fence_proxy_async();
                }
                tmem_st32(tb + uint32_t(32 * a), t);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&afull[j & 1]);
        }
        // D of the row: the two groups' shares meet in shared memory
        __shared__ float sD[2][kQM];
        sD[hf][r] = D;
        asm volatile("bar.sync 1, %0;" ::"r"(kEpiWarps * 32) : "memory");
        D = sD[0][r] + sD[1][r];
        if (p.D != nullptr && hf == 0 && i < p.S) p.D[int64_t(h) * p.S + i] = D;
        constexpr int half = HD / 2, q4 = HD / 4, nck = q4 / 16;
        // this row's (cos, sin) of its group's columns, loaded while the last MMAs run
        float4 cs_all[nck][8];
        {
            const float4 *rt4 = reinterpret_cast<const float4 *>(p.rt + int64_t(row_ok ? i : 0) * half);
#pragma unroll
            for (int ck = 0; ck < nck; ++ck)
#pragma unroll
                for (int t = 0; t < 8; ++t)
                    cs_all[ck][t] = p.rope ? rt4[(hf * q4 + 16 * ck) / 2 + t] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (ok && mbar_wait(&ufull, 0, p.status, 29u)) {
            tc_fence_after();
            float *out0 = p.dq + h * HD;
            // the rings are idle (every copy consumed, every MMA done): each warp turns its
            // 32-row blocks there so that the stores coalesce
            float *blk = reinterpret_cast<float *>(sm) + (warp - 2) * 32 * 33;
            const int c4 = (lane & 7) * 4, rl = lane >> 3;
#pragma unroll
            for (int ck = 0; ck < nck; ++ck) {                        // pairs (c, c + HD / 2)
                const int c = hf * q4 + 16 * ck;
                const float4 *cs = cs_all[ck];   // (cos, sin) of columns c .. c + 15, two per load
                uint32_t u1[16], u2[16], w1[16], w2[16];
                tmem_ld16(tmem + Ly::TU + uint32_t(c) + lane_off, u1);
                tmem_ld16(tmem + Ly::TU + uint32_t(c + half) + lane_off, u2);
                tmem_ld16(tmem + Ly::TW + uint32_t(c) + lane_off, w1);
                tmem_ld16(tmem + Ly::TW + uint32_t(c + half) + lane_off, w2);
                tmem_wait_ld();
                float y1[16], y2[16];
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    float a1 = p.scale * (__uint_as_float(u1[t]) - D * __uint_as_float(w1[t]));
                    float a2 = p.scale * (__uint_as_float(u2[t]) - D * __uint_as_float(w2[t]));
                    if (p.rope) {
                        const float4 q = cs[t / 2];
                        const float co = (t & 1) ? q.z : q.x, sn = (t & 1) ? q.w : q.y;
                        const float b1 = a1 * co + a2 * sn, b2 = -a1 * sn + a2 * co;
                        a1 = b1;
                        a2 = b2;
                    }
                    y1[t] = a1;
                    y2[t] = a2;
                }
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    blk[lane * 33 + t] = y1[t];
                    blk[lane * 33 + 16 + t] = y2[t];
                }
                __syncwarp();
#pragma unroll
                for (int k = 0; k < 8; ++k) {           // block column c4 is head column c + c4, or
                    const int rr = 4 * k + rl, ii = q0 + quarter * 32 + rr;   // c + half + c4 - 16
                    const float *a = blk + rr * 33 + c4;
                    if (ii < p.S)
                        *reinterpret_cast<float4 *>(out0 + int64_t(ii) * (p.nh * HD) + (c4 < 16 ? c + c4 : c + half + c4 - 16)) =
                            make_float4(a[0], a[1], a[2], a[3]);
                }
                __syncwarp();
            }
        }
        if (!ok) s_abort = 1;
    }
    // wind down: the MMA thread waited for its final commit, so no MMA is in flight;
    // after an abort, wait (bounded) for tile copies that were issued but not consumed
    tc_fence_before();
    __syncthreads();
    if (s_abort && threadIdx.x == 0) {
        for (int j = s_v_used; j < s_v_issued; ++j) mbar_wait(&vfull[j % kQSlots], (j / kQSlots) & 1, nullptr, 0u);
        for (int j = s_k_used; j < s_k_issued; ++j) mbar_wait(&kfull[j % kQSlots], (j / kQSlots) & 1, nullptr, 0u);
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Ly::COLS);
    }
}

// ------------------------------------------------------------------ dV

template <int HD>
struct DvLayout {
    // shared memory: rings of kVSlots slots: P tiles [kVQ queries][128 keys] (4 boxes) and
    // dCtx^T tiles [HD][kVQ queries] (the B operand)
    static constexpr int S_BYTES = kVQ * kVK * 4, B_BYTES = HD * kVQ * 4;
    static constexpr int B0 = kVSlots * S_BYTES, TOTAL = B0 + kVSlots * B_BYTES;
    // tensor memory: dV accumulator [128 keys][HD], then two P^T buffers [128 keys][kVQ] (A operand)
    static constexpr uint32_t TA = HD;
    static constexpr uint32_t COLS = (HD + 2 * kVQ) <= 128 ? 128 : 256;
};

template <int HD>
__global__ void __launch_bounds__(kAttnThreads, 2) attn_tc_dv_kernel(const __grid_constant__ AttnTcParams p) {
    using Ly = DvLayout<HD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    // sfull/sfree: P staging ring; bfull/bfree: dCtx^T ring; afull/afree: P^T in TMEM
    __shared__ uint64_t sfull[kVSlots], sfree[kVSlots], bfull[kVSlots], bfree[kVSlots], afull[2], afree[2], dfull;
    __shared__ uint32_t tmem_base;
    __shared__ int s_abort, s_s_issued, s_b_issued, s_b_used;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.x, G = p.nh / p.nkv, kvh = h / G, g = h % G;
    const int k0 = int(blockIdx.y) * kVK;                 // among the S newest keys (heaviest first)
    const int t0 = p.causal ? k0 / kVQ : 0;               // first query tile that sees key k0
    const int nw = (p.S + kVQ - 1) / kVQ - t0;            // query tiles of this CTA

    if (threadIdx.x == 0) {
        s_abort = 0;
        s_s_issued = s_b_issued = s_b_used = 0;
        for (int s = 0; s < kVSlots; ++s) {
            mbar_init(&sfull[s], 1);
            mbar_init(&sfree[s], kEpiWarps);
            mbar_init(&bfull[s], 1);
            mbar_init(&bfree[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&afull[b], kEpiWarps);
            mbar_init(&afree[b], 1);
        }
        mbar_init(&dfull, 1);
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base, Ly::COLS);
        tmem_relinquish();
    }
    fence_mbar_init();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tD = tmem_base;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer, kVSlots items ahead
        if (lane == 0) {
            for (int w = 0; w < nw; ++w) {
                const int s = w % kVSlots, qa = (t0 + w) * kVQ;
                if (w >= kVSlots && !mbar_wait(&sfree[s], (w / kVSlots - 1) & 1, p.status, 30u)) { s_abort = 1; break; }
                mbar_arrive_expect_tx(&sfull[s], Ly::S_BYTES);
                for (int b = 0; b < kVK / 32; ++b)
                    tma_load_3d(sm + s * Ly::S_BYTES + b * (kVQ * 128), &p.pv, p.pos0 + k0 + b * 32, qa, h, &sfull[s]);
                s_s_issued = w + 1;
                if (w >= kVSlots && !mbar_wait(&bfree[s], (w / kVSlots - 1) & 1, p.status, 36u)) { s_abort = 1; break; }
                mbar_arrive_expect_tx(&bfull[s], Ly::B_BYTES);
                tma_load_3d(sm + Ly::B0 + s * Ly::B_BYTES, &p.dct, qa, 0, h, &bfull[s]);
                s_b_issued = w + 1;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer: dV += P^T (TMEM) dCtx^T^T
        if (lane == 0) {
            constexpr uint32_t id = idesc_tf32(kVK, HD);
            bool ok = true;
            for (int w = 0; w < nw; ++w) {
                const int s = w % kVSlots;
                if (!mbar_wait(&afull[w & 1], (w >> 1) & 1, p.status, 31u) ||
                    !mbar_wait(&bfull[s], (w / kVSlots) & 1, p.status, 32u)) {
                    ok = false;
                    break;
                }
                s_b_used = w + 1;
                tc_fence_after();
                const uint64_t bd = sw128_desc(sm + Ly::B0 + s * Ly::B_BYTES);
                const uint32_t ta = tD + Ly::TA + uint32_t((w & 1) * kVQ);
#pragma unroll
                for (int k = 0; k < kVQ / 8; ++k)
                    mma_tf32_ts(tD, ta + uint32_t(8 * k), bd + 2 * k, id, (w > 0 || k > 0) ? 1u : 0u);
                mma_commit(&bfree[s]);
                mma_commit(&afree[w & 1]);
            }
            if (!ok) s_abort = 1;
            mma_commit(&dfull);
            mbar_wait(&dfull, 0, nullptr, 0u);
        }
    } else {
        // ------------------------------------------------ P^T writers, then the dV epilogue:
        // one key row and half of the queries (later: half of the columns) per thread
        constexpr int HQ = kVQ / 2;
        const int quarter = warp & 3, hf = (warp - 2) >> 2;
        const int r = quarter * 32 + lane, jj = k0 + r;        // key row of this thread
        const bool key_ok = jj < p.S;
        const int box = r >> 5, col = r & 31;
        const uint32_t lane_off = uint32_t(quarter * 32) << 16;
        bool ok = true;
        for (int w = 0; w < nw; ++w) {
            const int s = w % kVSlots, qa = (t0 + w) * kVQ + hf * HQ;
            if (!mbar_wait(&sfull[s], (w / kVSlots) & 1, p.status, 33u)) { ok = false; break; }
            const uint8_t *ps = sm + s * Ly::S_BYTES + box * (kVQ * 128) + (col & 3) * 4;
            static_assert(HQ == 16, "one 16-column tensor-memory store per writer");
            uint32_t pt[HQ];
#pragma unroll
            for (int qq = 0; qq < HQ; ++qq) {
                const float v = *reinterpret_cast<const float *>(ps + sw128_off(hf * HQ + qq, col >> 2));
                const bool vis = key_ok && (!p.causal || qa + qq >= jj);   // rows past S arrive as zeros
                pt[qq] = to_tf32(vis ? v : 0.f);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sfree[s]);               // staging slot read
            if (w >= 2 && !mbar_wait(&afree[w & 1], ((w - 2) >> 1) & 1, p.status, 34u)) { ok = false; break; }
            tc_fence_after();
            const uint32_t ta = tD + Ly::TA + uint32_t((w & 1) * kVQ + hf * HQ) + lane_off;
            tmem_st16(ta, pt);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&afull[w & 1]);
        }
        if (ok && mbar_wait(&dfull, 0, p.status, 35u)) {
            tc_fence_after();
            // Every copy into the staging ring has been consumed by now, so each warp turns
            // its 32 x 32 blocks there: lanes then run along columns and the stores coalesce.
            float *blk = reinterpret_cast<float *>(sm) + (warp - 2) * 32 * 33;
            const int64_t kvd = int64_t(p.nkv) * HD;
            float *out = p.dv + (G > 1 ? int64_t(g) * p.S * kvd : 0) + kvh * HD;
            const int c4 = (lane & 7) * 4, rl = lane >> 3;
#pragma unroll 1
            for (int c = hf * (HD / 2); c < (hf + 1) * (HD / 2); c += 32) {
                uint32_t v[32];
                tmem_ld32(tD + uint32_t(c) + lane_off, v);
                tmem_wait_ld();
#pragma unroll
                for (int t = 0; t < 32; ++t) blk[lane * 33 + t] = __uint_as_float(v[t]);
                __syncwarp();
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int rr = 4 * k + rl, key = k0 + quarter * 32 + rr;
                    const float *a = blk + rr * 33 + c4;
                    if (key < p.S)
                        *reinterpret_cast<float4 *>(out + int64_t(key) * kvd + c + c4) =
                            make_float4(a[0], a[1], a[2], a[3]);
                }
                __syncwarp();
            }
        }
        if (!ok) s_abort = 1;
    }
    tc_fence_before();
    __syncthreads();
    if (s_abort && threadIdx.x == 0) {
        // at most kVSlots copies per ring are in flight: the last ones issued
        for (int w = max(s_b_used, s_s_issued - kVSlots); w < s_s_issued; ++w)
            mbar_wait(&sfull[w % kVSlots], (w / kVSlots) & 1, nullptr, 0u);
        for (int w = max(s_b_used, s_b_issued - kVSlots); w < s_b_issued; ++w)
            mbar_wait(&bfull[w % kVSlots], (w / kVSlots) & 1, nullptr, 0u);
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tD, Ly::COLS);
    }
}

// ------------------------------------------------------------------ dK (exact input gradient)

// Key gradient of the S newest keys for the exact layer-input gradient: per head h and
// tile of 128 keys, over 32-query items w (causal: from the first item that sees key k0),
//   T^T_w = V_tile dCtx_w^T          tcgen05.mma, both operands in shared memory (V once)
//   dS^T  = P^T (.) (T^T - D_w)       writer warps, tf32 into tensor memory
//   dK   += dS^T q_w                  tcgen05.mma, A from tensor memory, q^T tile as B
// then scale dK (per-head partials added in head order when the group has several heads).
// A ring slot holds one item's P tile (4 boxes of 32 keys), tf32 dCtx rows and q^T tile,
// filled by one transaction and freed by ten arrivals: the eight writer warps once they
// have read P, and the commits of the item's two MMAs.  T^T_w+2 may take T^T_w's buffer as
// soon as the writers have read it; dS^T_w+2 waits for the dK MMA of item w.
template <int HD>
struct DkLayout {
    static constexpr int NB = HD / 32;                       // 128-byte atoms along head_dim
    static constexpr int V_BYTES = kVK * HD * 4;             // V tile [128 keys][HD], NB atoms
    static constexpr int P_BYTES = kVQ * kVK * 4;            // P item [32 queries][128 keys], 4 boxes
    static constexpr int C_BYTES = kVQ * HD * 4;             // dCtx rows [32 queries][HD], NB atoms
    static constexpr int Q_BYTES = HD * kVQ * 4;             // q^T [HD][32 queries], one atom
    static constexpr int SA = P_BYTES + C_BYTES;             // ring A slot: P and dCtx rows
    static constexpr int NS = 3;                             // slots of each ring
    static constexpr int A0 = V_BYTES, B0 = V_BYTES + NS * SA, TOTAL = B0 + NS * Q_BYTES;
    __host__ __device__ static constexpr int P(int s) { return A0 + s * SA; }
    __host__ __device__ static constexpr int C(int s) { return A0 + s * SA + P_BYTES; }
    __host__ __device__ static constexpr int Q(int s) { return B0 + s * Q_BYTES; }
    // tensor memory: dK [128 keys][HD], then T^T and dS^T double buffers [128 keys][32]
    static constexpr uint32_t TT = HD, TS = HD + 2 * kVQ;
    static constexpr uint32_t COLS = (HD + 4 * kVQ) <= 256 ? 256 : 512;
};

struct AttnTcDkParams {
    CUtensorMap v;              // Vr  {hd, L, nkv},   box {32, 128, 1}
    CUtensorMap pv;             // attn {L, S, nh},    box {32, 32, 1}
    CUtensorMap dcr;            // dCR {hd, nh, S},    box {32, 1, 32}  (tf32 dCtx rows)
    CUtensorMap qt;             // QT  {S, hd, nh},    box {32, hd, 1}  (tf32 q, transposed)
    const float *D;             // [nh, S]
    float *dk;                  // [S, nkv * hd], or per-head partials [nh / nkv][S, nkv * hd]
    int S, L, nh, nkv, pos0, causal;
    float scale;
    uint32_t *status;
};

// Key gradient of the S newest keys for the exact layer-input gradient: per head h and
// tile of 128 keys, over 32-query items w (causal: from the first item that sees key k0),
//   T^T_w = V_tile dCtx_w^T          tcgen05.mma, both operands in shared memory (V once)
//   dS^T  = P^T (.) (T^T - D_w)       writer warps, tf32 into tensor memory
//   dK   += dS^T q_w                  tcgen05.mma, A from tensor memory, q^T tile as B
// then scale dK (per-head partials added in head order when the group has several heads).
// Two rings, each filled by its own producer lane: A holds an item's P tile (4 boxes of
// 32 keys) and tf32 dCtx rows, freed once the writers have read P and T^T_w is formed; B
// holds its q^T tile, freed by the dK MMA.  The two writer groups take alternate items.
// T^T_w+2 may take T^T_w's buffer as soon as the writers have read it; dS^T_w+2 waits for
// the dK MMA of item w.
template <int HD>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_tc_dk_kernel(const __grid_constant__ AttnTcDkParams p) {
    using Ly = DkLayout<HD>;
    constexpr int NS = Ly::NS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    __shared__ uint64_t vfull, afullr[NS], afreer[NS], bfull[NS], bfree[NS], tfull[2], tfree[2], afull[2], afree[2],
        dfull;
    __shared__ uint32_t tmem_base;
    __shared__ int s_abort, s_a_issued, s_a_used, s_b_issued, s_b_used;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.x, G = p.nh / p.nkv, kvh = h / G, g = h % G;
    const int k0 = int(gridDim.y - 1 - blockIdx.y) * kVK;    // among the S newest keys (heaviest first)
    const int t0 = p.causal ? k0 / kVQ : 0;                   // first query item that sees key k0
    const int nw = (p.S + kVQ - 1) / kVQ - t0;

    if (threadIdx.x == 0) {
        s_abort = 0;
        s_a_issued = s_a_used = s_b_issued = s_b_used = 0;
        mbar_init(&vfull, 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(&afullr[s], 1);
            mbar_init(&afreer[s], kEpiWarps / 2 + 1);   // the item's writer group and its T^T MMA
            mbar_init(&bfull[s], 1);
            mbar_init(&bfree[s], 1);                    // its dK MMA
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tfree[b], kEpiWarps / 2);
            mbar_init(&afull[b], kEpiWarps / 2);
            mbar_init(&afree[b], 1);
        }
        mbar_init(&dfull, 1);
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base, Ly::COLS);
        tmem_relinquish();
    }
    fence_mbar_init();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tD = tmem_base;

    if (warp == 0) {
        // ------------------------------------------------ TMA producers: lane 0 V and ring A,
        // lane 1 ring B, NS items ahead each
        if (lane == 0) {
            mbar_arrive_expect_tx(&vfull, Ly::V_BYTES);
            for (int b = 0; b < Ly::NB; ++b)
                tma_load_3d(sm + b * (kVK * 128), &p.v, b * 32, p.pos0 + k0, kvh, &vfull);
            for (int w = 0; w < nw; ++w) {
                const int s = w % NS, qa = (t0 + w) * kVQ;
                if (w >= NS && !mbar_wait(&afreer[s], (w / NS - 1) & 1, p.status, 40u)) { s_abort = 1; break; }
                mbar_arrive_expect_tx(&afullr[s], Ly::SA);
                for (int b = 0; b < kVK / 32; ++b)
                    tma_load_3d(sm + Ly::P(s) + b * (kVQ * 128), &p.pv, p.pos0 + k0 + b * 32, qa, h, &afullr[s]);
                for (int b = 0; b < Ly::NB; ++b)
                    tma_load_3d(sm + Ly::C(s) + b * (kVQ * 128), &p.dcr, b * 32, h, qa, &afullr[s]);
                s_a_issued = w + 1;
            }
        } else if (lane == 1) {
            for (int w = 0; w < nw; ++w) {
                const int s = w % NS, qa = (t0 + w) * kVQ;
                if (w >= NS && !mbar_wait(&bfree[s], (w / NS - 1) & 1, p.status, 49u)) { s_abort = 1; break; }
                mbar_arrive_expect_tx(&bfull[s], Ly::Q_BYTES);
                tma_load_3d(sm + Ly::Q(s), &p.qt, qa, 0, h, &bfull[s]);
                s_b_issued = w + 1;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t id_t = idesc_tf32(kVK, kVQ), id_k = idesc_tf32(kVK, HD);
            auto mma_t = [&](int w) -> bool {              // T^T[w % 2] = V dCtx_w^T
                const int s = w % NS;
                if (!mbar_wait(&afullr[s], (w / NS) & 1, p.status, 41u)) return false;
                s_a_used = w + 1;
                tc_fence_after();
#pragma unroll
                for (int kb = 0; kb < Ly::NB; ++kb)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_tf32(tD + Ly::TT + uint32_t((w & 1) * kVQ), sw128_desc(sm + kb * (kVK * 128)) + 2 * k,
                                 sw128_desc(sm + Ly::C(s) + kb * (kVQ * 128)) + 2 * k, id_t, (kb | k) ? 1u : 0u);
                mma_commit(&afreer[s]);
                mma_commit(&tfull[w & 1]);
                return true;
            };
            bool ok = mbar_wait(&vfull, 0, p.status, 42u);
            tc_fence_after();
            ok = ok && (nw < 1 || mma_t(0)) && (nw < 2 || mma_t(1));
            for (int w = 0; ok && w < nw; ++w) {
                const int s = w % NS;
                if (!mbar_wait(&afull[w & 1], (w >> 1) & 1, p.status, 43u) ||
                    !mbar_wait(&bfull[s], (w / NS) & 1, p.status, 50u)) {
                    ok = false;
                    break;
                }
                s_b_used = w + 1;
                tc_fence_after();
                const uint64_t qd = sw128_desc(sm + Ly::Q(s));
#pragma unroll
                for (int k = 0; k < kVQ / 8; ++k)
                    mma_tf32_ts(tD, tD + Ly::TS + uint32_t((w & 1) * kVQ + 8 * k), qd + 2 * k, id_k,
                                (w > 0 || k > 0) ? 1u : 0u);
                mma_commit(&bfree[s]);
                mma_commit(&afree[w & 1]);
                // T^T_w+2 takes T^T_w's buffer: the writers read it before they filled dS^T_w
                if (w + 2 < nw) {
                    if (!mbar_wait(&tfree[w & 1], (w >> 1) & 1, p.status, 44u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (!(ok = mma_t(w + 2))) break;
                }
            }
            if (!ok) s_abort = 1;
            mma_commit(&dfull);
            mbar_wait(&dfull, 0, nullptr, 0u);
        }
    } else {
        // ------------------------------------------------ dS^T writers, then the dK epilogue:
        // the two groups of four warps take alternate items (group hf the items w = hf mod 2
        // and with them T^T / dS^T buffer hf), one key row (tensor-memory lane) and all 32
        // queries of the item per thread; the D values of the group's next item are loaded
        // while the current one is formed
        const int quarter = warp & 3, hf = (warp - 2) >> 2;
        const int r = quarter * 32 + lane, jj = k0 + r;        // key row of this thread
        const bool key_ok = jj < p.S;
        const int box = r >> 5, col = r & 31;
        const uint32_t lane_off = uint32_t(quarter * 32) << 16;
        const float *Dh = p.D + int64_t(h) * p.S;
        auto load_d = [&](int w, float (&dv)[kVQ]) {
            const int qa = (t0 + w) * kVQ;
#pragma unroll
            for (int qq = 0; qq < kVQ; ++qq) dv[qq] = (w < nw && qa + qq < p.S) ? __ldg(Dh + qa + qq) : 0.f;
        };
        float dv[kVQ], dvn[kVQ];
        load_d(hf, dv);
        bool ok = true;
        for (int w = hf; w < nw; w += 2) {
            const int s = w % NS, qa = (t0 + w) * kVQ;
            if (!mbar_wait(&afullr[s], (w / NS) & 1, p.status, 45u) ||
                !mbar_wait(&tfull[w & 1], (w >> 1) & 1, p.status, 46u)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t t[kVQ];
            tmem_ld32(tD + Ly::TT + uint32_t((w & 1) * kVQ) + lane_off, t);
            const uint8_t *ps = sm + Ly::P(s) + box * (kVQ * 128) + (col & 3) * 4;
            float pv[kVQ];
#pragma unroll
            for (int qq = 0; qq < kVQ; ++qq) pv[qq] = *reinterpret_cast<const float *>(ps + sw128_off(qq, col >> 2));
            load_d(w + 2, dvn);
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&tfree[w & 1]);                     // T^T_w read
                mbar_arrive(&afreer[s]);                        // P read
            }
            uint32_t ds[kVQ];
#pragma unroll
            for (int qq = 0; qq < kVQ; ++qq) {
                const bool vis = key_ok && qa + qq < p.S && (!p.causal || qa + qq >= jj);
                ds[qq] = to_tf32(vis ? pv[qq] * (__uint_as_float(t[qq]) - dv[qq]) : 0.f);
            }
            if (w >= 2 && !mbar_wait(&afree[w & 1], ((w - 2) >> 1) & 1, p.status, 47u)) { ok = false; break; }
            tc_fence_after();
            tmem_st32(tD + Ly::TS + uint32_t((w & 1) * kVQ) + lane_off, ds);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&afull[w & 1]);
#pragma unroll
            for (int qq = 0; qq < kVQ; ++qq) dv[qq] = dvn[qq];
        }
        if (ok && mbar_wait(&dfull, 0, p.status, 48u)) {
            tc_fence_after();
            // every copy into the rings has been consumed: each warp turns its 32 x 32 blocks
            // in ring A so that the stores coalesce
            float *blk = reinterpret_cast<float *>(sm + Ly::P(0)) + (warp - 2) * 32 * 33;
            const int64_t kvd = int64_t(p.nkv) * HD;
            float *out = p.dk + (G > 1 ? int64_t(g) * p.S * kvd : 0) + kvh * HD;
            const int c4 = (lane & 7) * 4, rl = lane >> 3;
#pragma unroll 1
            for (int c = hf * (HD / 2); c < (hf + 1) * (HD / 2); c += 32) {
                uint32_t v[32];
                tmem_ld32(tD + uint32_t(c) + lane_off, v);
                tmem_wait_ld();
#pragma unroll
                for (int q = 0; q < 32; ++q) blk[lane * 33 + q] = p.scale * __uint_as_float(v[q]);
                __syncwarp();
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int rr = 4 * k + rl, key = k0 + quarter * 32 + rr;
                    const float *a = blk + rr * 33 + c4;
                    if (key < p.S)
                        *reinterpret_cast<float4 *>(out + int64_t(key) * kvd + c + c4) =
                            make_float4(a[0], a[1], a[2], a[3]);
                }
                __syncwarp();
            }
        }
        if (!ok) s_abort = 1;
    }
    tc_fence_before();
    __syncthreads();
    if (s_abort && threadIdx.x == 0) {
        // the copies issued but not yet consumed (at most NS per ring, and V)
        mbar_wait(&vfull, 0, nullptr, 0u);
        for (int w = max(s_a_used, s_a_issued - NS); w < s_a_issued; ++w)
            mbar_wait(&afullr[w % NS], (w / NS) & 1, nullptr, 0u);
        for (int w = max(s_b_used, s_b_issued - NS); w < s_b_issued; ++w)
            mbar_wait(&bfull[w % NS], (w / NS) & 1, nullptr, 0u);
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tD, Ly::COLS);
    }
}

// dst = tf32 (round to nearest) copy of src, n floats (n % 4 == 0, 16-byte aligned)
__global__ void tf32_copy_kernel(const float4 *__restrict__ src, float4 *__restrict__ dst, int64_t n4) {
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += int64_t(gridDim.x) * blockDim.x) {
        const float4 x = src[i];
        dst[i] = make_float4(__uint_as_float(to_tf32(x.x)), __uint_as_float(to_tf32(x.y)), __uint_as_float(to_tf32(x.z)),
                             __uint_as_float(to_tf32(x.w)));
    }
}

// dV[jj, c] = sum over the group's heads g (in order) of part[g][jj, c]
__global__ void attn_tc_dv_sum_kernel(const float4 *__restrict__ part, float4 *__restrict__ dv, int64_t n4, int G) {
    constexpr int kMaxG = 8;                              // heads per KV head summed from registers
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < n4; e += 2 * stride) {
        const bool two = e + stride < n4;                 // two elements per thread
        float4 s0, s1;
        if (G <= kMaxG) {
            // every head's partial of both elements in flight at once, then the sums in
            // head order (the order the general loop below adds them in)
            float4 t0[kMaxG], t1[kMaxG];
#pragma unroll
            for (int g = 0; g < kMaxG; ++g) {
                t0[g] = g < G ? part[int64_t(g) * n4 + e] : z;
                t1[g] = g < G && two ? part[int64_t(g) * n4 + e + stride] : z;
            }
            s0 = t0[0];
            s1 = t1[0];
#pragma unroll
            for (int g = 1; g < kMaxG; ++g) {
                if (g >= G) break;
                s0.x += t0[g].x; s0.y += t0[g].y; s0.z += t0[g].z; s0.w += t0[g].w;
                s1.x += t1[g].x; s1.y += t1[g].y; s1.z += t1[g].z; s1.w += t1[g].w;
            }
        } else {
            s0 = part[e];
            s1 = two ? part[e + stride] : z;
            for (int g = 1; g < G; ++g) {
                const float4 t0 = part[int64_t(g) * n4 + e];
                const float4 t1 = two ? part[int64_t(g) * n4 + e + stride] : z;
                s0.x += t0.x; s0.y += t0.y; s0.z += t0.z; s0.w += t0.w;
                s1.x += t1.x; s1.y += t1.y; s1.z += t1.z; s1.w += t1.w;
            }
        }
        dv[e] = s0;
        if (two) dv[e + stride] = s1;
    }
}

// ------------------------------------------------------------------ recomputed attention

// The flash-style path: the attention weights are recomputed from q, the K cache and each
// query row's logsumexp instead of read from a materialised [nh, S, L] tensor.  After the
// prep (which also writes the tf32 K rows Kr):
//   dV kernel, per (head, tile of 128 cache keys), over 32-query items w:
//     S^T = K_tile q_w^T and T^T = V_tile dCtx_w^T            tcgen05.mma
//     P^T = exp(scale S^T - lse), masked, tf32, over S^T        writer warps
//     D_part[key tile, quarter][h, q] = sum over the quarter's 32 keys of P^T (.) T^T
//     dV += P^T dCtx_w                                          tcgen05.mma, A from tensor memory
//   D sum: D[h, i] = the partials of the visible key tiles in (tile, quarter) order, the
//     softmax-backward row sum sum_j P_ij dAttn_ij;
//   dQ kernel, per (head, tile of 128 queries), over 32-key tiles j:
//     S_j = q K_j^T and T_j = dCtx V_j^T                        tcgen05.mma
//     E_j = exp(scale S_j - lse) (T_j - D), masked, tf32, over T_j
//     dQ += E_j K_j                                             tcgen05.mma, A from tensor memory
//   then scale and RoPE backward as for the materialised path.
constexpr int kRK = 32;         // keys per recomputed-dQ tile
constexpr int kRBuf = 4;        // S / T buffer sets in tensor memory: the MMA thread keeps three ahead

struct AttnTcRcParams {
    CUtensorMap kr128, vr128;   // Kr, Vr {hd, L, nkv}, box {32, 128, 1}  dV: A of S^T, T^T (once)
    CUtensorMap qrow, crow;     // q, dCtx {hd, nh, S}, box {32, 1, 32}   dV: B of S^T, T^T
    CUtensorMap dct;            // dCT {S, hd, nh}, box {32, hd, 1}       dV: B of dV
    CUtensorMap kr32, vr32;     // Kr, Vr {hd, L, nkv}, box {32, 32, 1}   dQ: B of S, T
    CUtensorMap kt;             // Kt {L, hd, nkv}, box {32, hd, 1}       dQ: B of dQ
    const float *q, *dctx, *lse;
    float *Dpart, *D;           // [nkt * 4][nh][S], [nh][S]
    float *dq, *dv;             // dv: [S, nkv * hd], or per-head partials [nh / nkv][S, nkv * hd]
    const float2 *rt;           // RoPE table (rope only)
    int S, L, nh, nkv, pos0, causal, rope, nkt;
    float scale;
    uint32_t *status;
};

template <int HD>
struct DvRcLayout {
    static constexpr int NB = HD / 32;
    static constexpr int KV_BYTES = kVK * HD * 4;     // K or V rows [128 keys][HD]: NB atoms
    static constexpr int QI_BYTES = kVQ * HD * 4;     // q or dCtx rows [32][HD]: NB atoms
    static constexpr int CT_BYTES = HD * kVQ * 4;     // dCtx^T [HD][32]: one atom
    // ring A: an item's q and dCtx rows (freed once S^T and T^T are formed); ring B: its
    // dCtx^T (freed by its dV MMA)
    static constexpr int SA = 2 * QI_BYTES, NS = 2;
    static constexpr int K0 = 0, V0 = KV_BYTES, A0 = 2 * KV_BYTES, B0 = A0 + NS * SA, TOTAL = B0 + NS * CT_BYTES;
    __host__ __device__ static constexpr int Q(int s) { return A0 + s * SA; }
    __host__ __device__ static constexpr int C(int s) { return A0 + s * SA + QI_BYTES; }
    __host__ __device__ static constexpr int CT(int s) { return B0 + s * CT_BYTES; }
    // tensor memory: dV [128 keys][HD], then kRBuf sets of S^T (P^T written over it) and T^T
    static constexpr uint32_t TS = HD, TT = HD + kRBuf * kVQ;
    static constexpr uint32_t COLS = (HD + 2 * kRBuf * kVQ) <= 256 ? 256 : 512;
};

template <int HD>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_tc_dv_rc_kernel(const __grid_constant__ AttnTcRcParams p) {
    using Ly = DvRcLayout<HD>;
    constexpr int NB = Ly::NB, NS = Ly::NS;
    static_assert(HD + 2 * kRBuf * kVQ <= 512, "tensor memory");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    // kvfull: the K and V tiles; afull/afree, bfull/bfree: rings A and B; sfull: S^T and T^T of
    // an item formed; pfull: its P^T written; tfree: its dV MMA done (the buffer set is free)
    __shared__ uint64_t kvfull, afull[NS], afree[NS], bfull[NS], bfree[NS], sfull[kRBuf], pfull[kRBuf],
        tfree[kRBuf], dfull;
    __shared__ uint32_t tmem_base;
    __shared__ int s_abort, s_a_issued, s_a_used, s_b_issued, s_b_used;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.x, G = p.nh / p.nkv, kvh = h / G, g = h % G;
    const int k0 = int(blockIdx.y) * kVK;                           // cache keys k0 .. k0 + 127
    const int t0 = (p.causal ? max(0, k0 - p.pos0) : 0) / kVQ;      // first item that sees key k0
    const int nw = (p.S + kVQ - 1) / kVQ - t0;

    if (threadIdx.x == 0) {
        s_abort = 0;
        s_a_issued = s_a_used = s_b_issued = s_b_used = 0;
        mbar_init(&kvfull, 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(&afull[s], 1);
            mbar_init(&afree[s], 1);
            mbar_init(&bfull[s], 1);
            mbar_init(&bfree[s], 1);
        }
        for (int b = 0; b < kRBuf; ++b) {
            mbar_init(&sfull[b], 1);
            mbar_init(&pfull[b], kEpiWarps);
            mbar_init(&tfree[b], 1);
        }
        mbar_init(&dfull, 1);
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base, Ly::COLS);
        tmem_relinquish();
    }
    fence_mbar_init();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tD = tmem_base;

    if (warp == 0) {
        // ------------------------------------------------ TMA producers: lane 0 the K and V
        // tiles and ring A, lane 1 ring B
        if (lane == 0) {
            mbar_arrive_expect_tx(&kvfull, 2 * Ly::KV_BYTES);
            for (int b = 0; b < NB; ++b) {
                tma_load_3d(sm + Ly::K0 + b * (kVK * 128), &p.kr128, b * 32, k0, kvh, &kvfull);
                tma_load_3d(sm + Ly::V0 + b * (kVK * 128), &p.vr128, b * 32, k0, kvh, &kvfull);
            }
            for (int w = 0; w < nw; ++w) {
                const int s = w % NS, qa = (t0 + w) * kVQ;
                if (w >= NS && !mbar_wait(&afree[s], (w / NS - 1) & 1, p.status, 40u)) {
                    s_abort = 1;
                    break;
                }
                mbar_arrive_expect_tx(&afull[s], Ly::SA);
                for (int b = 0; b < NB; ++b) {
                    tma_load_3d(sm + Ly::Q(s) + b * (kVQ * 128), &p.qrow, b * 32, h, qa, &afull[s]);
                    tma_load_3d(sm + Ly::C(s) + b * (kVQ * 128), &p.crow, b * 32, h, qa, &afull[s]);
                }
                s_a_issued = w + 1;
            }
        } else if (lane == 1) {
            for (int w = 0; w < nw; ++w) {
                const int s = w % NS, qa = (t0 + w) * kVQ;
                if (w >= NS && !mbar_wait(&bfree[s], (w / NS - 1) & 1, p.status, 41u)) {
                    s_abort = 1;
                    break;
                }
                mbar_arrive_expect_tx(&bfull[s], Ly::CT_BYTES);
                tma_load_3d(sm + Ly::CT(s), &p.dct, qa, 0, h, &bfull[s]);
                s_b_issued = w + 1;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = idesc_tf32(kVK, kVQ), idV = idesc_tf32(kVK, HD);
            auto issue = [&](int w) -> bool {      // S^T_w and T^T_w into buffer set w % kRBuf
                const int s = w % NS, b = w % kRBuf;
                if (!mbar_wait(&afull[s], (w / NS) & 1, p.status, 42u)) return false;
                if (w >= kRBuf && !mbar_wait(&tfree[b], (w / kRBuf - 1) & 1, p.status, 43u)) return false;
                s_a_used = w + 1;
                tc_fence_after();
#pragma unroll
                for (int kb = 0; kb < NB; ++kb)
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t acc = (kb | k) ? 1u : 0u;
                        mma_tf32(tD + Ly::TS + uint32_t(b * kVQ), sw128_desc(sm + Ly::K0 + kb * (kVK * 128)) + 2 * k,
                                 sw128_desc(sm + Ly::Q(s) + kb * (kVQ * 128)) + 2 * k, idS, acc);
                        mma_tf32(tD + Ly::TT + uint32_t(b * kVQ), sw128_desc(sm + Ly::V0 + kb * (kVK * 128)) + 2 * k,
                                 sw128_desc(sm + Ly::C(s) + kb * (kVQ * 128)) + 2 * k, idS, acc);
                    }
                mma_commit(&afree[s]);
                mma_commit(&sfull[b]);
                return true;
            };
            bool ok = mbar_wait(&kvfull, 0, p.status, 44u);
            tc_fence_after();
            for (int w = 0; ok && w < min(nw, kRBuf - 1); ++w) ok = issue(w);
            for (int w = 0; ok && w < nw; ++w) {
                const int s = w % NS, b = w % kRBuf;
                if (!mbar_wait(&pfull[b], (w / kRBuf) & 1, p.status, 45u) ||
                    !mbar_wait(&bfull[s], (w / NS) & 1, p.status, 46u)) {
                    ok = false;
                    break;
                }
                s_b_used = w + 1;
                tc_fence_after();
                const uint64_t bd = sw128_desc(sm + Ly::CT(s));
#pragma unroll
                for (int k = 0; k < kVQ / 8; ++k)
                    mma_tf32_ts(tD, tD + Ly::TS + uint32_t(b * kVQ + 8 * k), bd + 2 * k, idV, (w > 0 || k > 0) ? 1u : 0u);
                mma_commit(&bfree[s]);
                mma_commit(&tfree[b]);
                // S^T / T^T of item w + 3 take the buffer set of item w - 1, whose dV MMA was
                // issued one item ago: the wait overlaps dV_w in the tensor pipe
                if (w + kRBuf - 1 < nw && !(ok = issue(w + kRBuf - 1))) break;
            }
            if (!ok) s_abort = 1;
            mma_commit(&dfull);
            mbar_wait(&dfull, 0, nullptr, 0u);
        }
    } else {
        // ------------------------------------------------ writers: one key row and half of the
        // item's queries per thread; then the dV epilogue
        const int quarter = warp & 3, hf = (warp - 2) >> 2;
        const int r = quarter * 32 + lane, key = k0 + r;
        const uint32_t lane_off = uint32_t(quarter * 32) << 16;
        const float *lse_h = p.lse + int64_t(h) * p.S;
        const float sl2 = p.scale * kLog2e;
        float *dpart = p.Dpart + (int64_t(int(blockIdx.y) * 4 + quarter) * p.nh + h) * p.S;
        // the query of the item's half whose sum over this warp's keys this lane ends with
        const int b4 = (lane >> 4) & 1, b3 = (lane >> 3) & 1, b2 = (lane >> 2) & 1, b1 = (lane >> 1) & 1;
        const int cq = 8 * b4 + 4 * b3 + 2 * b2 + b1;
        bool ok = true;
        for (int w = 0; w < nw; ++w) {
            const int b = w % kRBuf, qa = (t0 + w) * kVQ + hf * 16;
            float l[16];                                     // lse log2(e) of the half's queries
#pragma unroll
            for (int c = 0; c < 16; ++c) l[c] = qa + c < p.S ? __ldg(lse_h + qa + c) * kLog2e : 0.f;
            if (!mbar_wait(&sfull[b], (w / kRBuf) & 1, p.status, 47u)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sv[16], tv[16];
            tmem_ld16(tD + Ly::TS + uint32_t(b * kVQ + hf * 16) + lane_off, sv);
            tmem_ld16(tD + Ly::TT + uint32_t(b * kVQ + hf * 16) + lane_off, tv);
            tmem_wait_ld();
            float e[16];
            uint32_t pt[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const int qi = qa + c;
                const bool vis = qi < p.S && key < p.L && (!p.causal || key <= p.pos0 + qi);
                const float pv = vis ? ex2_approx(fmaf(sl2, __uint_as_float(sv[c]), -l[c])) : 0.f;
                e[c] = pv * __uint_as_float(tv[c]);
                pt[c] = to_tf32(pv);
            }
            tmem_st16(tD + Ly::TS + uint32_t(b * kVQ + hf * 16) + lane_off, pt);     // P^T over S^T
            // sum of e over the warp's 32 keys by halving exchanges: each level keeps half of
            // the queries and adds the partner's values of that half
            float v8[8], v4[4], v2[2];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float send = b4 ? e[i] : e[8 + i];
                v8[i] = (b4 ? e[8 + i] : e[i]) + __shfl_xor_sync(0xffffffffu, send, 16);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float send = b3 ? v8[i] : v8[4 + i];
                v4[i] = (b3 ? v8[4 + i] : v8[i]) + __shfl_xor_sync(0xffffffffu, send, 8);
            }
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const float send = b2 ? v4[i] : v4[2 + i];
                v2[i] = (b2 ? v4[2 + i] : v4[i]) + __shfl_xor_sync(0xffffffffu, send, 4);
            }
            float v1 = (b1 ? v2[1] : v2[0]) + __shfl_xor_sync(0xffffffffu, b1 ? v2[0] : v2[1], 2);
            v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
            if ((lane & 1) == 0 && qa + cq < p.S) dpart[qa + cq] = v1;
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&pfull[b]);
        }
        if (ok && mbar_wait(&dfull, 0, p.status, 48u)) {
            tc_fence_after();
            // the rings are idle (every copy consumed, every MMA done): each warp turns its
            // 32 x 32 blocks there so that the stores coalesce; only the S newest keys have dV
            float *blk = reinterpret_cast<float *>(sm) + (warp - 2) * 32 * 33;
            const int64_t kvd = int64_t(p.nkv) * HD;
            float *out = p.dv + (G > 1 ? int64_t(g) * p.S * kvd : 0) + kvh * HD;
            const int c4 = (lane & 7) * 4, rl = lane >> 3, first = p.L - p.S;
#pragma unroll 1
            for (int c = hf * (HD / 2); c < (hf + 1) * (HD / 2); c += 32) {
                uint32_t v[32];
                tmem_ld32(tD + uint32_t(c) + lane_off, v);
                tmem_wait_ld();
#pragma unroll
                for (int t = 0; t < 32; ++t) blk[lane * 33 + t] = __uint_as_float(v[t]);
                __syncwarp();
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int rr = 4 * k + rl, kk = k0 + quarter * 32 + rr;
                    const float *a = blk + rr * 33 + c4;
                    if (kk >= first && kk < p.L)
                        *reinterpret_cast<float4 *>(out + int64_t(kk - first) * kvd + c + c4) =
                            make_float4(a[0], a[1], a[2], a[3]);
                }
                __syncwarp();
            }
        }
        if (!ok) s_abort = 1;
    }
    tc_fence_before();
    __syncthreads();
    if (s_abort && threadIdx.x == 0) {
        mbar_wait(&kvfull, 0, nullptr, 0u);
        for (int w = max(s_a_used, s_a_issued - NS); w < s_a_issued; ++w)
            mbar_wait(&afull[w % NS], (w / NS) & 1, nullptr, 0u);
        for (int w = max(s_b_used, s_b_issued - NS); w < s_b_issued; ++w)
            mbar_wait(&bfull[w % NS], (w / NS) & 1, nullptr, 0u);
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tD, Ly::COLS);
    }
}

// D[h, i] = the partial row sums of the key tiles that row i sees, in (tile, quarter) order.
__global__ void attn_tc_dsum_kernel(const float *__restrict__ Dpart, float *__restrict__ D, int S, int nh, int nkt,
                                    int pos0, int causal) {
    const int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (e >= int64_t(nh) * S) return;
    const int h = int(e / S), i = int(e % S);
    const int lim = causal ? min(nkt, (pos0 + i) / kVK + 1) : nkt;      // tiles with first key <= pos0 + i
    const int64_t stride = int64_t(nh) * S;
    const float *src = Dpart + int64_t(h) * S + i;
    float acc = 0.f;
    for (int t0 = 0; t0 < lim; t0 += 4) {          // sixteen loads in flight, then the sum in order
        float v[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] = t0 + k / 4 < lim ? __ldg(src + int64_t(t0 * 4 + k) * stride) : 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) acc += v[k];
    }
    D[e] = acc;
}

template <int HD>
struct DqRcLayout {
    static constexpr int NB = HD / 32;
    static constexpr int Q_BYTES = kQM * HD * 4;      // q tile [128 rows][HD]: NB atoms (A of S)
    static constexpr int R_BYTES = kRK * HD * 4;      // K or V rows [32 keys][HD]: NB atoms
    static constexpr int KT_BYTES = HD * kRK * 4;     // K^T [HD][32 keys]: one atom
    // ring A: a tile's K and V rows (freed once S and T are formed); ring B: its K^T (freed
    // by its dQ MMA)
    static constexpr int SA = 2 * R_BYTES, NS = 3;
    static constexpr int A0 = Q_BYTES, B0 = A0 + NS * SA, TOTAL = B0 + NS * KT_BYTES;
    __host__ __device__ static constexpr int KR(int s) { return A0 + s * SA; }
    __host__ __device__ static constexpr int VR(int s) { return A0 + s * SA + R_BYTES; }
    __host__ __device__ static constexpr int KT(int s) { return B0 + s * KT_BYTES; }
    // tensor memory: dCtx (A of T), dQ, kRBuf sets of S and T (E written over T), [128][32] each
    static constexpr uint32_t TDC = 0, TQD = HD, TS = 2 * HD, TT = 2 * HD + kRBuf * kRK;
    static constexpr uint32_t COLS = (2 * HD + 2 * kRBuf * kRK) <= 256 ? 256 : 512;
};

template <int HD>
__global__ void __launch_bounds__(kAttnThreads, 1) attn_tc_dq_rc_kernel(const __grid_constant__ AttnTcRcParams p) {
    using Ly = DqRcLayout<HD>;
    constexpr int NB = Ly::NB, NS = Ly::NS;
    static_assert(2 * HD + 2 * kRBuf * kRK <= 512, "tensor memory");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    // afull/afree, bfull/bfree: rings A and B; qready: q in shared memory and dCtx in tensor
    // memory; sfull: S_j and T_j formed; efull: E_j written; tfree: dQ_j done
    __shared__ uint64_t afull[NS], afree[NS], bfull[NS], bfree[NS], qready, sfull[kRBuf], efull[kRBuf],
        tfree[kRBuf], dfull;
    __shared__ uint32_t tmem_base;
    __shared__ int s_abort, s_a_issued, s_a_used, s_b_issued, s_b_used;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.x, kvh = h / (p.nh / p.nkv);
    const int q0 = int(gridDim.y - 1 - blockIdx.y) * kQM;      // longest tiles first
    const int kend = p.causal ? min(p.L, p.pos0 + q0 + kQM) : p.L;
    const int nt = (kend + kRK - 1) / kRK;

    if (threadIdx.x == 0) {
        s_abort = 0;
        s_a_issued = s_a_used = s_b_issued = s_b_used = 0;
        for (int s = 0; s < NS; ++s) {
            mbar_init(&afull[s], 1);
            mbar_init(&afree[s], 1);
            mbar_init(&bfull[s], 1);
            mbar_init(&bfree[s], 1);
        }
        mbar_init(&qready, kEpiWarps);
        for (int b = 0; b < kRBuf; ++b) {
            mbar_init(&sfull[b], 1);
            mbar_init(&efull[b], kEpiWarps / 2);    // the four warps of the group that forms E_j
            mbar_init(&tfree[b], 1);
        }
        mbar_init(&dfull, 1);
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base, Ly::COLS);
        tmem_relinquish();
    }
    fence_mbar_init();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = tmem_base;

    if (warp == 0) {
        // ------------------------------------------------ TMA producers: lane 0 ring A, lane 1 ring B
        if (lane == 0) {
            for (int j = 0; j < nt; ++j) {
                const int s = j % NS, k0 = j * kRK;
                if (j >= NS && !mbar_wait(&afree[s], (j / NS - 1) & 1, p.status, 50u)) {
                    s_abort = 1;
                    break;
                }
                mbar_arrive_expect_tx(&afull[s], Ly::SA);
                for (int b = 0; b < NB; ++b) {
                    tma_load_3d(sm + Ly::KR(s) + b * (kRK * 128), &p.kr32, b * 32, k0, kvh, &afull[s]);
                    tma_load_3d(sm + Ly::VR(s) + b * (kRK * 128), &p.vr32, b * 32, k0, kvh, &afull[s]);
                }
                s_a_issued = j + 1;
            }
        } else if (lane == 1) {
            for (int j = 0; j < nt; ++j) {
                const int s = j % NS;
                if (j >= NS && !mbar_wait(&bfree[s], (j / NS - 1) & 1, p.status, 51u)) {
                    s_abort = 1;
                    break;
                }
                mbar_arrive_expect_tx(&bfull[s], Ly::KT_BYTES);
                tma_load_3d(sm + Ly::KT(s), &p.kt, j * kRK, 0, kvh, &bfull[s]);
                s_b_issued = j + 1;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = idesc_tf32(kQM, kRK), idQ = idesc_tf32(kQM, HD);
            auto issue = [&](int j) -> bool {      // S_j and T_j into buffer set j % kRBuf
                const int s = j % NS, b = j % kRBuf;
                if (!mbar_wait(&afull[s], (j / NS) & 1, p.status, 52u)) return false;
                if (j >= kRBuf && !mbar_wait(&tfree[b], (j / kRBuf - 1) & 1, p.status, 53u)) return false;
                s_a_used = j + 1;
                tc_fence_after();
#pragma unroll
                for (int kb = 0; kb < NB; ++kb)
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t acc = (kb | k) ? 1u : 0u;
                        mma_tf32(tm + Ly::TS + uint32_t(b * kRK), sw128_desc(sm + kb * (kQM * 128)) + 2 * k,
                                 sw128_desc(sm + Ly::KR(s) + kb * (kRK * 128)) + 2 * k, idS, acc);
                        mma_tf32_ts(tm + Ly::TT + uint32_t(b * kRK), tm + Ly::TDC + uint32_t(kb * 32 + k * 8),
                                    sw128_desc(sm + Ly::VR(s) + kb * (kRK * 128)) + 2 * k, idS, acc);
                    }
                mma_commit(&afree[s]);
                mma_commit(&sfull[b]);
                return true;
            };
            bool ok = mbar_wait(&qready, 0, p.status, 54u);
            tc_fence_after();
            for (int j = 0; ok && j < min(nt, kRBuf - 1); ++j) ok = issue(j);
            for (int j = 0; ok && j < nt; ++j) {
                const int s = j % NS, b = j % kRBuf;
                if (!mbar_wait(&efull[b], (j / kRBuf) & 1, p.status, 55u) ||
                    !mbar_wait(&bfull[s], (j / NS) & 1, p.status, 56u)) {
                    ok = false;
                    break;
                }
                s_b_used = j + 1;
                tc_fence_after();
                const uint64_t kd = sw128_desc(sm + Ly::KT(s));
#pragma unroll
                for (int k = 0; k < kRK / 8; ++k)
                    mma_tf32_ts(tm + Ly::TQD, tm + Ly::TT + uint32_t(b * kRK + 8 * k), kd + 2 * k, idQ,
                                (j > 0 || k > 0) ? 1u : 0u);
                mma_commit(&bfree[s]);
                mma_commit(&tfree[b]);
                // S_j+3 / T_j+3 take the buffer set of tile j - 1, whose dQ MMA was issued one
                // tile ago: the wait overlaps dQ_j in the tensor pipe
                if (j + kRBuf - 1 < nt && !(ok = issue(j + kRBuf - 1))) break;
            }
            if (!ok) s_abort = 1;
            mma_commit(&dfull);
            mbar_wait(&dfull, 0, nullptr, 0u);
        }
    } else {
        // ------------------------------------------------ writers: two groups of four warps
        // (one per TMEM lane quarter), one query row per thread
        const int quarter = warp & 3, hf = (warp - 2) >> 2;
        const int r = quarter * 32 + lane, i = q0 + r;
        const bool row_ok = i < p.S;
        const uint32_t lane_off = uint32_t(quarter * 32) << 16;
        const int jlast = p.causal ? p.pos0 + i : p.L - 1;      // last visible key
        {   // this row's half of q (tf32) into the q tile (the A operand of S, 128-byte
            // swizzled atoms of 32 columns) and of dCtx (tf32) into tensor memory (A of T)
            const int64_t ro = int64_t(row_ok ? i : 0) * (p.nh * HD) + h * HD + hf * (HD / 2);
            const float4 *qs = reinterpret_cast<const float4 *>(p.q + ro);
            const float4 *cs = reinterpret_cast<const float4 *>(p.dctx + ro);
            float4 xq[HD / 8], xc[HD / 8];
#pragma unroll
            for (int k = 0; k < HD / 8; ++k) {
                xq[k] = row_ok ? qs[k] : make_float4(0.f, 0.f, 0.f, 0.f);
                xc[k] = row_ok ? cs[k] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int k = 0; k < HD / 8; ++k) {
                const int col = hf * (HD / 2) + 4 * k;          // column of the row
                st_shared_v4(sm + (col >> 5) * (kQM * 128) + sw128_off(r, (col & 31) >> 2), to_tf32(xq[k].x),
                             to_tf32(xq[k].y), to_tf32(xq[k].z), to_tf32(xq[k].w));
            }
#pragma unroll
            for (int c = 0; c < HD / 2; c += 16) {
                uint32_t v[16];
#pragma unroll
                for (int t = 0; t < 16; t += 4) {
                    const float4 y = xc[(c + t) / 4];
                    v[t] = to_tf32(y.x);
                    v[t + 1] = to_tf32(y.y);
                    v[t + 2] = to_tf32(y.z);
                    v[t + 3] = to_tf32(y.w);
                }
                tmem_st16(tm + Ly::TDC + uint32_t(hf * (HD / 2) + c) + lane_off, v);
            }
            tmem_wait_st();
            fence_proxy_async();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&qready);
        }
        const float lse_i = row_ok ? __ldg(p.lse + int64_t(h) * p.S + i) * kLog2e : 0.f;   // in log2 units
        const float sl2 = p.scale * kLog2e;
        const float D_i = row_ok ? __ldg(p.D + int64_t(h) * p.S + i) : 0.f;
        // Key tiles alternate between the two groups of four warps
        bool ok = true;
        for (int j = hf; j < nt; j += 2) {
            const int b = j % kRBuf, ka = j * kRK;
            if (!mbar_wait(&sfull[b], (j / kRBuf) & 1, p.status, 57u)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sv[32], tv[32];
            tmem_ld32(tm + Ly::TS + uint32_t(b * kRK) + lane_off, sv);
            tmem_ld32(tm + Ly::TT + uint32_t(b * kRK) + lane_off, tv);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const bool vis = row_ok && ka + c <= jlast;
                const float pv = vis ? ex2_approx(fmaf(sl2, __uint_as_float(sv[c]), -lse_i)) : 0.f;
                tv[c] = to_tf32(pv * (__uint_as_float(tv[c]) - D_i));
            }
            tmem_st32(tm + Ly::TT + uint32_t(b * kRK) + lane_off, tv);       // E_j over T_j
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&efull[b]);
        }
        constexpr int half = HD / 2, q4 = HD / 4, nck = q4 / 16;
        // this row's (cos, sin) of its group's columns, loaded while the last MMAs run
        float4 cs_all[nck][8];
        {
            const float4 *rt4 = reinterpret_cast<const float4 *>(p.rt + int64_t(row_ok ? i : 0) * half);
#pragma unroll
            for (int ck = 0; ck < nck; ++ck)
#pragma unroll
                for (int t = 0; t < 8; ++t)
                    cs_all[ck][t] = p.rope ? rt4[(hf * q4 + 16 * ck) / 2 + t] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (ok && mbar_wait(&dfull, 0, p.status, 58u)) {
            tc_fence_after();
            float *out0 = p.dq + h * HD;
            float *blk = reinterpret_cast<float *>(sm) + (warp - 2) * 32 * 33;
            const int c4 = (lane & 7) * 4, rl = lane >> 3;
#pragma unroll
            for (int ck = 0; ck < nck; ++ck) {                        // pairs (c, c + HD / 2)
                const int c = hf * q4 + 16 * ck;
                const float4 *cs = cs_all[ck];
                uint32_t u1[16], u2[16];
                tmem_ld16(tm + Ly::TQD + uint32_t(c) + lane_off, u1);
                tmem_ld16(tm + Ly::TQD + uint32_t(c + half) + lane_off, u2);
                tmem_wait_ld();
                float y1[16], y2[16];
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    float a1 = p.scale * __uint_as_float(u1[t]), a2 = p.scale * __uint_as_float(u2[t]);
                    if (p.rope) {
                        const float4 qv = cs[t / 2];
                        const float co = (t & 1) ? qv.z : qv.x, sn = (t & 1) ? qv.w : qv.y;
                        const float b1 = a1 * co + a2 * sn, b2 = -a1 * sn + a2 * co;
                        a1 = b1;
                        a2 = b2;
                    }
                    y1[t] = a1;
                    y2[t] = a2;
                }
#pragma unroll
                for (int t = 0; t < 16; ++t) {
                    blk[lane * 33 + t] = y1[t];
                    blk[lane * 33 + 16 + t] = y2[t];
                }
                __syncwarp();
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int rr = 4 * k + rl, ii = q0 + quarter * 32 + rr;
                    const float *a = blk + rr * 33 + c4;
                    if (ii < p.S)
                        *reinterpret_cast<float4 *>(out0 + int64_t(ii) * (p.nh * HD) +
                                                    (c4 < 16 ? c + c4 : c + half + c4 - 16)) =
                            make_float4(a[0], a[1], a[2], a[3]);
                }
                __syncwarp();
            }
        }
        if (!ok) s_abort = 1;
    }
    tc_fence_before();
    __syncthreads();
    if (s_abort && threadIdx.x == 0) {
        for (int j = max(s_a_used, s_a_issued - NS); j < s_a_issued; ++j)
            mbar_wait(&afull[j % NS], (j / NS) & 1, nullptr, 0u);
        for (int j = max(s_b_used, s_b_issued - NS); j < s_b_issued; ++j)
            mbar_wait(&bfull[j % NS], (j / NS) & 1, nullptr, 0u);
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tm, Ly::COLS);
    }
}

// ------------------------------------------------------------------ host side

// fp32 3-D tensor map, 128-byte swizzle, zero fill out of range.  dims / box innermost
// first; strides in bytes of dims 1 and 2.
int make_map_f32_3d(CUtensorMap *m, const void *base, const uint64_t dims[3], const uint64_t strides[2],
                    const uint32_t box[3]) {
    EncodeTiled enc = encode_fn();
    TLB_REQUIRE(enc != nullptr, TLB_ECUDA, "attention (tcgen05): cuTensorMapEncodeTiled unavailable");
    const cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
    const cuuint64_t st[2] = {strides[0], strides[1]};
    const cuuint32_t bx[3] = {box[0], box[1], box[2]};
    const cuuint32_t es[3] = {1, 1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void *>(base), d, st, bx, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    TLB_REQUIRE(r == CUDA_SUCCESS, TLB_ECUDA, "attention (tcgen05): tensor map encoding failed (%d)", int(r));
    return TLB_OK;
}

struct TcAttnWs {
    size_t dCT, Kt, Vr, part, rt, Kr, Dpart, Dd, total;
    int64_t S4, L4;
};

// rc: the recomputed-attention path, which adds the K rows and the row-sum partials.
TcAttnWs tc_attn_layout(int64_t S, int64_t L, int nh, int nkv, int hd, bool rc = false) {
    auto r256 = [](size_t b) { return (b + 255) & ~size_t(255); };
    TcAttnWs w;
    w.S4 = (S + 3) & ~int64_t(3);
    w.L4 = (L + 3) & ~int64_t(3);
    w.dCT = 0;
    w.Kt = w.dCT + r256(size_t(nh) * hd * w.S4 * 4);
    w.Vr = w.Kt + r256(size_t(nkv) * hd * w.L4 * 4);
    w.part = w.Vr + r256(size_t(nkv) * L * hd * 4);
    w.rt = w.part + (nh > nkv ? r256(size_t(nh) * S * hd * 4) : 0);      // per-head dV sums
    w.Kr = w.rt + r256(size_t(S) * (hd / 2) * 8);                         // RoPE table
    const int64_t nkt = (L + kVK - 1) / kVK;
    w.Dpart = w.Kr + (rc ? r256(size_t(nkv) * L * hd * 4) : 0);
    w.Dd = w.Dpart + (rc ? r256(size_t(nkt) * 4 * nh * S * 4) : 0);
    w.total = w.Dd + (rc ? r256(size_t(nh) * S * 4) : 0);
    return w;
}

template <int HD>
int launch_attn_tc(const AttnArgs &a, const RopeFreqs &fr, void *scratch, uint32_t *status, cudaStream_t st) {
    const TcAttnWs w = tc_attn_layout(a.S, a.L, a.nh, a.nkv, HD);
    char *base = static_cast<char *>(scratch);
    float *dCT = reinterpret_cast<float *>(base + w.dCT);
    float *Kt = reinterpret_cast<float *>(base + w.Kt), *Vr = reinterpret_cast<float *>(base + w.Vr);
    const int nt_dc = a.dct_ready ? 0 : int(ceil_div(a.S, kPrepT)) * (a.nh * HD / kPrepT);   // dCtx^T tiles
    const int nt_kv = int(ceil_div(a.L, kPrepT)) * (a.nkv * HD / kPrepT);
    const int vec_kv = aligned16(a.k) && aligned16(a.v) && a.sh % 4 == 0 && a.sp % 4 == 0;
    float2 *rt = reinterpret_cast<float2 *>(base + w.rt);
    const int nt_rt = a.rope ? int(ceil_div(int64_t(a.S) * (HD / 2), int64_t(1024))) : 0;
    attn_tc_prep_kernel<<<unsigned(nt_dc + 2 * nt_kv + nt_rt), 256, 0, st>>>(a, dCT, Kt, Vr, int(w.S4), int(w.L4),
                                                                            nt_dc, nt_kv, vec_kv, fr, rt, nullptr);
    TLB_TRY(check_launch("attn_tc_prep"));

    AttnTcParams p;
    memset(&p, 0, sizeof(p));
    {
        const uint64_t d[3] = {uint64_t(HD), uint64_t(a.L), uint64_t(a.nkv)};
        const uint64_t s[2] = {uint64_t(HD) * 4, uint64_t(a.L) * HD * 4};
        const uint32_t b[3] = {32, uint32_t(kQK), 1};
        TLB_TRY(make_map_f32_3d(&p.v, Vr, d, s, b));
    }
    {
        const uint64_t d[3] = {uint64_t(a.L), uint64_t(a.S), uint64_t(a.nh)};
        const uint64_t s[2] = {uint64_t(a.L) * 4, uint64_t(a.S) * a.L * 4};
        const uint32_t bq[3] = {32, uint32_t(kQM), 1}, bv[3] = {32, uint32_t(kVQ), 1};
        TLB_TRY(make_map_f32_3d(&p.pq, a.attn, d, s, bq));
        TLB_TRY(make_map_f32_3d(&p.pv, a.attn, d, s, bv));
    }
    {
        const uint64_t d[3] = {uint64_t(a.L), uint64_t(HD), uint64_t(a.nkv)};
        const uint64_t s[2] = {uint64_t(w.L4) * 4, uint64_t(w.L4) * HD * 4};
        const uint32_t b[3] = {32, uint32_t(HD), 1};
        TLB_TRY(make_map_f32_3d(&p.kt, Kt, d, s, b));
    }
    {
        const uint64_t d[3] = {uint64_t(a.S), uint64_t(HD), uint64_t(a.nh)};
        const uint64_t s[2] = {uint64_t(w.S4) * 4, uint64_t(w.S4) * HD * 4};
        const uint32_t b[3] = {32, uint32_t(HD), 1};
        TLB_TRY(make_map_f32_3d(&p.dct, dCT, d, s, b));
    }
    const int G = a.nh / a.nkv;
    float *part = reinterpret_cast<float *>(base + w.part);
    p.dctx = a.dctx;
    p.dcT = dCT;
    p.ld_ct = int(w.S4);
    p.dq = a.dq;
    p.dv = G > 1 ? part : a.dv;
    p.S = a.S;
    p.L = a.L;
    p.nh = a.nh;
    p.nkv = a.nkv;
    p.pos0 = a.pos0;
    p.causal = a.causal;
    p.rope = a.rope;
    p.scale = a.scale;
    p.status = status;
    p.D = a.D;
    p.rt = rt;

    const int smq = DqLayout<HD>::TOTAL + 1024, smv = DvLayout<HD>::TOTAL + 1024;
    TLB_CUDA(cudaFuncSetAttribute(attn_tc_dq_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, smq));
    TLB_CUDA(cudaFuncSetAttribute(attn_tc_dv_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, smv));
    attn_tc_dq_kernel<HD><<<dim3(unsigned(a.nh), unsigned(ceil_div(a.S, kQM))), kAttnThreads, smq, st>>>(p);
    TLB_TRY(check_launch("attn_tc_dq"));
    attn_tc_dv_kernel<HD><<<dim3(unsigned(a.nh), unsigned(ceil_div(a.S, kVK))), kAttnThreads, smv, st>>>(p);
    TLB_TRY(check_launch("attn_tc_dv"));
    if (G == 1) return TLB_OK;
    const int64_t n4 = int64_t(a.S) * a.nkv * HD / 4;
    attn_tc_dv_sum_kernel<<<stream_grid(n4, 256), 256, 0, st>>>(reinterpret_cast<const float4 *>(part),
                                                                reinterpret_cast<float4 *>(a.dv), n4, G);
    return check_launch("attn_tc_dv_sum");
}

template <int HD>
int launch_attn_tc_dk(const AttnArgs &a, const float *q, const float *D, float *dk, void *scratch, void *extra,
                      uint32_t *status, cudaStream_t st) {
    const TcAttnWs w = tc_attn_layout(a.S, a.L, a.nh, a.nkv, HD);
    char *base = static_cast<char *>(scratch);
    const float *Vr = reinterpret_cast<const float *>(base + w.Vr);     // left by the attention prep
    float *part = reinterpret_cast<float *>(base + w.part);
    const int64_t qd = int64_t(a.nh) * HD;
    float *dCR = static_cast<float *>(extra);                            // [S, qd] tf32 dCtx
    float *QT = dCR + ((a.S * qd + 63) & ~int64_t(63));                  // [qd, S4] tf32 q, transposed
    const int64_t n4 = a.S * qd / 4;
    tf32_copy_kernel<<<stream_grid(n4, 256), 256, 0, st>>>(reinterpret_cast<const float4 *>(a.dctx),
                                                           reinterpret_cast<float4 *>(dCR), n4);
    TLB_TRY(check_launch("tf32_copy"));
    AttnArgs aq = a;               // the prep's first job transposes its dctx rows: give it q
    aq.dctx = q;
    const int nt_q = int(ceil_div(a.S, kPrepT)) * int(qd / kPrepT);
    const RopeFreqs no_rope{};
    attn_tc_prep_kernel<<<unsigned(nt_q), 256, 0, st>>>(aq, QT, nullptr, nullptr, int(w.S4), int(w.L4), nt_q, 0, 0,
                                                        no_rope, nullptr, nullptr);
    TLB_TRY(check_launch("attn_tc_prep_q"));

    AttnTcDkParams p;
    memset(&p, 0, sizeof(p));
    {
        const uint64_t d[3] = {uint64_t(HD), uint64_t(a.L), uint64_t(a.nkv)};
        const uint64_t s[2] = {uint64_t(HD) * 4, uint64_t(a.L) * HD * 4};
        const uint32_t b[3] = {32, uint32_t(kVK), 1};
        TLB_TRY(make_map_f32_3d(&p.v, Vr, d, s, b));
    }
    {
        const uint64_t d[3] = {uint64_t(a.L), uint64_t(a.S), uint64_t(a.nh)};
        const uint64_t s[2] = {uint64_t(a.L) * 4, uint64_t(a.S) * a.L * 4};
        const uint32_t b[3] = {32, uint32_t(kVQ), 1};
        TLB_TRY(make_map_f32_3d(&p.pv, a.attn, d, s, b));
    }
    {
        const uint64_t d[3] = {uint64_t(HD), uint64_t(a.nh), uint64_t(a.S)};
        const uint64_t s[2] = {uint64_t(HD) * 4, uint64_t(qd) * 4};
        const uint32_t b[3] = {32, 1, uint32_t(kVQ)};
        TLB_TRY(make_map_f32_3d(&p.dcr, dCR, d, s, b));
    }
    {
        const uint64_t d[3] = {uint64_t(a.S), uint64_t(HD), uint64_t(a.nh)};
        const uint64_t s[2] = {uint64_t(w.S4) * 4, uint64_t(w.S4) * HD * 4};
        const uint32_t b[3] = {32, uint32_t(HD), 1};
        TLB_TRY(make_map_f32_3d(&p.qt, QT, d, s, b));
    }
    const int G = a.nh / a.nkv;
    p.D = D;
    p.dk = G > 1 ? part : dk;
    p.S = a.S;
    p.L = a.L;
    p.nh = a.nh;
    p.nkv = a.nkv;
    p.pos0 = a.pos0;
    p.causal = a.causal;
    p.scale = a.scale;
    p.status = status;
    const int sm = DkLayout<HD>::TOTAL + 1024;
    TLB_CUDA(cudaFuncSetAttribute(attn_tc_dk_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, sm));
    attn_tc_dk_kernel<HD><<<dim3(unsigned(a.nh), unsigned(ceil_div(a.S, kVK))), kAttnThreads, sm, st>>>(p);
    TLB_TRY(check_launch("attn_tc_dk"));
    if (G == 1) return TLB_OK;
    const int64_t m4 = int64_t(a.S) * a.nkv * HD / 4;
    attn_tc_dv_sum_kernel<<<stream_grid(m4, 256), 256, 0, st>>>(reinterpret_cast<const float4 *>(part),
                                                                reinterpret_cast<float4 *>(dk), m4, G);
    return check_launch("attn_tc_dk_sum");
}

// The recomputed-attention path (attention weights from q, K and lse).
template <int HD>
int launch_attn_tc_rc(const AttnArgs &a, const RopeFreqs &fr, void *scratch, uint32_t *status, cudaStream_t st) {
    const TcAttnWs w = tc_attn_layout(a.S, a.L, a.nh, a.nkv, HD, true);
    char *base = static_cast<char *>(scratch);
    float *dCT = reinterpret_cast<float *>(base + w.dCT);
    float *Kt = reinterpret_cast<float *>(base + w.Kt), *Vr = reinterpret_cast<float *>(base + w.Vr);
    float *Kr = reinterpret_cast<float *>(base + w.Kr);
    float2 *rt = reinterpret_cast<float2 *>(base + w.rt);
    const int nt_dc = a.dct_ready ? 0 : int(ceil_div(a.S, kPrepT)) * (a.nh * HD / kPrepT);   // dCtx^T tiles
    const int nt_kv = int(ceil_div(a.L, kPrepT)) * (a.nkv * HD / kPrepT);
    const int nt_rt = a.rope ? int(ceil_div(int64_t(a.S) * (HD / 2), int64_t(1024))) : 0;
    const int vec_kv = aligned16(a.k) && aligned16(a.v) && a.sh % 4 == 0 && a.sp % 4 == 0;
    attn_tc_prep_kernel<<<unsigned(nt_dc + 3 * nt_kv + nt_rt), 256, 0, st>>>(a, dCT, Kt, Vr, int(w.S4), int(w.L4),
                                                                            nt_dc, nt_kv, vec_kv, fr, rt, Kr);
    TLB_TRY(check_launch("attn_tc_prep"));

    AttnTcRcParams p;
    memset(&p, 0, sizeof(p));
    {
        const uint64_t d[3] = {uint64_t(HD), uint64_t(a.L), uint64_t(a.nkv)};
        const uint64_t s[2] = {uint64_t(HD) * 4, uint64_t(a.L) * HD * 4};
        const uint32_t b128[3] = {32, uint32_t(kVK), 1}, b32[3] = {32, uint32_t(kRK), 1};
        TLB_TRY(make_map_f32_3d(&p.kr128, Kr, d, s, b128));
        TLB_TRY(make_map_f32_3d(&p.vr128, Vr, d, s, b128));
        TLB_TRY(make_map_f32_3d(&p.kr32, Kr, d, s, b32));
        TLB_TRY(make_map_f32_3d(&p.vr32, Vr, d, s, b32));
    }
    {
        const uint64_t d[3] = {uint64_t(HD), uint64_t(a.nh), uint64_t(a.S)};
        const uint64_t s[2] = {uint64_t(HD) * 4, uint64_t(a.nh) * HD * 4};
        const uint32_t b[3] = {32, 1, uint32_t(kVQ)};
        TLB_TRY(make_map_f32_3d(&p.qrow, a.q, d, s, b));
        TLB_TRY(make_map_f32_3d(&p.crow, a.dctx, d, s, b));
    }
    {
        const uint64_t d[3] = {uint64_t(a.S), uint64_t(HD), uint64_t(a.nh)};
        const uint64_t s[2] = {uint64_t(w.S4) * 4, uint64_t(w.S4) * HD * 4};
        const uint32_t b[3] = {32, uint32_t(HD), 1};
        TLB_TRY(make_map_f32_3d(&p.dct, dCT, d, s, b));
    }
    {
        const uint64_t d[3] = {uint64_t(a.L), uint64_t(HD), uint64_t(a.nkv)};
        const uint64_t s[2] = {uint64_t(w.L4) * 4, uint64_t(w.L4) * HD * 4};
        const uint32_t b[3] = {32, uint32_t(HD), 1};
        TLB_TRY(make_map_f32_3d(&p.kt, Kt, d, s, b));
    }
    const int G = a.nh / a.nkv;
    float *part = reinterpret_cast<float *>(base + w.part);
    p.q = a.q;
    p.dctx = a.dctx;
    p.lse = a.lse;
    p.Dpart = reinterpret_cast<float *>(base + w.Dpart);
    p.D = a.D != nullptr ? a.D : reinterpret_cast<float *>(base + w.Dd);
    p.dq = a.dq;
    p.dv = G > 1 ? part : a.dv;
    p.rt = rt;
    p.S = a.S;
    p.L = a.L;
    p.nh = a.nh;
    p.nkv = a.nkv;
    p.pos0 = a.pos0;
    p.causal = a.causal;
    p.rope = a.rope;
    p.nkt = int(ceil_div(int64_t(a.L), int64_t(kVK)));
    p.scale = a.scale;
    p.status = status;

    const int smv = DvRcLayout<HD>::TOTAL + 1024, smq = DqRcLayout<HD>::TOTAL + 1024;
    TLB_CUDA(cudaFuncSetAttribute(attn_tc_dv_rc_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, smv));
    TLB_CUDA(cudaFuncSetAttribute(attn_tc_dq_rc_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, smq));
    attn_tc_dv_rc_kernel<HD><<<dim3(unsigned(a.nh), unsigned(p.nkt)), kAttnThreads, smv, st>>>(p);
    TLB_TRY(check_launch("attn_tc_dv_rc"));
    const int64_t nd = int64_t(a.nh) * a.S;
    attn_tc_dsum_kernel<<<unsigned(ceil_div(nd, int64_t(256))), 256, 0, st>>>(p.Dpart, p.D, a.S, a.nh, p.nkt, a.pos0,
                                                                            a.causal);
    TLB_TRY(check_launch("attn_tc_dsum"));
    attn_tc_dq_rc_kernel<HD><<<dim3(unsigned(a.nh), unsigned(ceil_div(a.S, kQM))), kAttnThreads, smq, st>>>(p);
    TLB_TRY(check_launch("attn_tc_dq_rc"));
    if (G == 1) return TLB_OK;
    const int64_t n4 = int64_t(a.S) * a.nkv * HD / 4;
    attn_tc_dv_sum_kernel<<<stream_grid(n4, 256), 256, 0, st>>>(reinterpret_cast<const float4 *>(part),
                                                                reinterpret_cast<float4 *>(a.dv), n4, G);
    return check_launch("attn_tc_dv_sum");
}

}  // namespace

bool attn_tc_supported(int64_t S, int64_t L, int nh, int nkv, int hd) {
    // TMA reads attn rows from key L - S on: L and L - S multiples of 4 (16-byte starts)
    return S > 1 && S <= L && L % 4 == 0 && (L - S) % 4 == 0 && (hd == 64 || hd == 128) && nh <= 65535 &&
           nkv <= 65535 && nh % nkv == 0 && L < (int64_t(1) << 30);
}

size_t attn_tc_bytes(int64_t S, int64_t L, int nh, int nkv, int hd) {
    return tc_attn_layout(S, L, nh, nkv, hd).total;
}

size_t attn_tc_dk_bytes(int64_t S, int nh, int hd) {
    const int64_t qd = int64_t(nh) * hd, S4 = (S + 3) & ~int64_t(3);
    return size_t((S * qd + 63) & ~int64_t(63)) * 4 + size_t(qd) * S4 * 4;
}

int attn_tc_dk_launch(const AttnArgs &a, const float *q, const float *D, float *dk, void *scratch, void *extra,
                      uint32_t *status, cudaStream_t st) {
    if (a.S == 0) return TLB_OK;
    TLB_REQUIRE(attn_tc_supported(a.S, a.L, a.nh, a.nkv, a.hd), TLB_EUNSUPPORTED, "key gradient (tcgen05): shape");
    TLB_REQUIRE(aligned16(q) && aligned16(dk) && aligned16(a.dctx) && aligned16(extra), TLB_EUNSUPPORTED,
                "key gradient (tcgen05): q / dk / dctx / scratch not 16-byte aligned");
    return a.hd == 128 ? launch_attn_tc_dk<128>(a, q, D, dk, scratch, extra, status, st)
                       : launch_attn_tc_dk<64>(a, q, D, dk, scratch, extra, status, st);
}

int attn_tc_launch(const AttnArgs &a, float rope_base, void *scratch, uint32_t *status, cudaStream_t st) {
    if (a.S == 0) return TLB_OK;
    TLB_REQUIRE(attn_tc_supported(a.S, a.L, a.nh, a.nkv, a.hd), TLB_EUNSUPPORTED, "attention (tcgen05): shape");
    TLB_REQUIRE((reinterpret_cast<uintptr_t>(scratch) & 255u) == 0, TLB_EINVAL, "attention (tcgen05): scratch alignment");
    const bool rc = a.lse != nullptr;
    TLB_REQUIRE((rc ? aligned16(a.q) : aligned16(a.attn)) && aligned16(a.dq) && aligned16(a.dv) && aligned16(a.dctx),
                TLB_EUNSUPPORTED, "attention (tcgen05): attn or q / dq / dv / dctx not 16-byte aligned");
    TLB_REQUIRE(a.dctx != nullptr || (a.dct_ready && !rc), TLB_EINVAL,
                "attention (tcgen05): no dctx needs the stored weights and a ready dCtx^T");
    RopeFreqs fr;
    rope_freqs(fr, a.hd, rope_base);
    if (rc)
        return a.hd == 128 ? launch_attn_tc_rc<128>(a, fr, scratch, status, st)
                           : launch_attn_tc_rc<64>(a, fr, scratch, status, st);
    return a.hd == 128 ? launch_attn_tc<128>(a, fr, scratch, status, st) : launch_attn_tc<64>(a, fr, scratch, status, st);
}

size_t attn_tc_rc_bytes(int64_t S, int64_t L, int nh, int nkv, int hd) {
    return tc_attn_layout(S, L, nh, nkv, hd, true).total;
}

}  // namespace tlb
