// LoRA adapter gradients and their AdamW step ([RS] "LoRA Q backward" and
// "LoRA V backward", cpu_adamw, LoRA+ rate on B), s = alpha / rank:
//   gh[i, r] = s sum_o G[i, o] B[o, r]     (B before its update)
//   dB[o, r] = s sum_i G[i, o] h[i, r]     -> AdamW on B with lr * lr_b_mult
//   dA[r, c] = sum_i gh[i, r] x[i, c]      -> AdamW on A with lr
// sum dA^2 and sum dB^2 are added to sumsq[0] and sumsq[1].
//
// Two schedules:
//   * lora_launch: per-element reductions over S (three kernels); its only scratch is
//     gh.  Serves the allocation-free entry point.
//   * lora_seq_launch: tiled over 64-token x 128-column tiles with partial sums in a
//     workspace, for any S and for one or two adapters sharing x:
//       G pass   one read of each G tile gives the dB partial of its 64 tokens and the
//                gh partial of its 128 columns;
//       gh       gh = s * sum of the column-tile partials;
//       x pass   one read of each x tile gives the dA partials of every adapter;
//       AdamW    sums the token-tile partials of dA and dB, applies the update.
//     Every sum runs in a fixed order: the result does not depend on scheduling.
//     Rank-16 adapters of a layer whose attention ran on the tensor cores take the
//     tcgen05 G and x passes of lora_tc.cu over 128-token tiles instead; they write the
//     same partial-sum layouts, so the gh sum and the AdamW kernel serve both.
#include <algorithm>

#include <mutex>

#include "async.cuh"
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

// ------------------------------------------------------------------ tiled schedule

namespace {

constexpr int kLT = 64;          // tokens per tile
constexpr int kLO = 128;         // columns of G or x per tile
constexpr int kLP = kLO + 4;     // padded shared-memory row (float4-aligned)

struct LoraSide {
    const float *G, *h;          // [S, O], [S, rank]
    int O, n_ot, blk0, vecG;     // columns, column tiles, first G-pass block, 16-byte loads ok
    float s;
    tlb_lora l;
    float *part_b;               // [nrc_b][O][rank] (sized for n_rt)
    float *part_gh;              // [n_ot][S][rank]
    float *gh;                   // [S][rank]
    float *part_a;               // [nrc_a][rank][C] (sized for n_rt)
};

struct LoraSeqArgs {
    LoraSide side[2];
    const float *x;              // [S, C]
    const uint32_t *status;      // status block (optional): its step gate set skips AdamW
    int nside, S, C, rank, n_rt, vecx, vech;
    int tpc_b, nrc_b;            // G pass: row tiles per chunk, chunks (dB partials)
    int tpc_a, nrc_a;            // x pass: row tiles per chunk, chunks (dA partials)
};

// Zero-padded [kLT][kLP] tile of rows r0.. and columns c0.. of src [nrow, ncol] (leading dim ld).
__device__ __forceinline__ void load_tile(float *dst, const float *__restrict__ src, int64_t ld, int nrow,
                                          int ncol, int r0, int c0, bool vec) {
    if (vec) {
        for (int e = threadIdx.x; e < kLT * (kLO / 4); e += blockDim.x) {
            const int i = e / (kLO / 4), c = (e % (kLO / 4)) * 4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r0 + i < nrow && c0 + c < ncol)
                v = ld_stream(reinterpret_cast<const float4 *>(src + int64_t(r0 + i) * ld + c0 + c));
            *reinterpret_cast<float4 *>(dst + i * kLP + c) = v;
        }
    } else {
        for (int e = threadIdx.x; e < kLT * kLO; e += blockDim.x) {
            const int i = e / kLO, c = e % kLO;
            dst[i * kLP + c] = (r0 + i < nrow && c0 + c < ncol) ? src[int64_t(r0 + i) * ld + c0 + c] : 0.f;
        }
    }
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src, bool valid) {
    // 16 bytes global -> shared, zero-filled when !valid (no bytes are read then)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// Start copying the [kLT][kLP] tile at rows r0.., columns c0.. of src [nrow, ncol] (leading
// dim ld) with 16-byte cp.async when `vec`; else load it now.
__device__ __forceinline__ void issue_tile(float *dst, const float *__restrict__ src, int64_t ld, int nrow, int ncol,
                                           int r0, int c0, bool vec) {
    if (!vec) {
        load_tile(dst, src, ld, nrow, ncol, r0, c0, false);
        return;
    }
    for (int e = threadIdx.x; e < kLT * (kLO / 4); e += blockDim.x) {
        const int i = e / (kLO / 4), c = (e % (kLO / 4)) * 4;
        const bool ok = r0 + i < nrow && c0 + c < ncol;
        cp_async16(dst + i * kLP + c, ok ? src + int64_t(r0 + i) * ld + c0 + c : src, ok);
    }
}

// [kLT][RB] rows r0.. of a [nrow, R] matrix, zero-padded to RB columns.
template <int RB>
__device__ __forceinline__ void issue_rows(float *dst, const float *__restrict__ src, int nrow, int R, int r0,
                                           bool vec) {
    if (vec) {                                   // R == RB, 16-byte aligned rows
        for (int e = threadIdx.x; e < kLT * (RB / 4); e += blockDim.x) {
            const int i = e / (RB / 4), c = (e % (RB / 4)) * 4;
            const bool ok = r0 + i < nrow;
            cp_async16(dst + i * RB + c, ok ? src + int64_t(r0 + i) * RB + c : src, ok);
        }
    } else {
        for (int e = threadIdx.x; e < kLT * RB; e += blockDim.x) {
            const int i = e / RB, r = e % RB;
            dst[e] = (r < R && r0 + i < nrow) ? src[int64_t(r0 + i) * R + r] : 0.f;
        }
    }
}

// Block (column tile of one side, chunk of row tiles): one pass over its G tiles, staged
// two deep, gives the dB partial of the chunk (kept in registers across its tiles) and
// the gh partial of each tile.
template <int RB>
__global__ void __launch_bounds__(256) lora_gpass_kernel(LoraSeqArgs a) {
    extern __shared__ float4 sm4[];
    float *sG = reinterpret_cast<float *>(sm4);   // 2 x [kLT][kLP]
    float *sh = sG + 2 * kLT * kLP;               // 2 x [kLT][RB]
    float *sB = sh + 2 * kLT * RB;                // [kLO][RB]
    const int side = (a.nside > 1 && int(blockIdx.x) >= a.side[1].blk0) ? 1 : 0;
    const LoraSide &p = a.side[side];
    const int ot = int(blockIdx.x) - p.blk0, o0 = ot * kLO, R = a.rank, tid = threadIdx.x;
    const int rt0 = blockIdx.y * a.tpc_b, rt1 = min(rt0 + a.tpc_b, a.n_rt);
    const bool vecG = p.vecG != 0, vech = a.vech != 0;
    for (int e = tid; e < kLO * RB; e += 256) {
        const int o = e / RB, r = e % RB;
        sB[e] = (r < R && o0 + o < p.O) ? p.l.b[int64_t(o0 + o) * R + r] : 0.f;
    }
    issue_tile(sG, p.G, p.O, a.S, p.O, rt0 * kLT, o0, vecG);
    issue_rows<RB>(sh, p.h, a.S, R, rt0 * kLT, vech);
    cp_async_commit();
    constexpr int NB = RB / 2, NG = RB / 4;
    const int ob = tid % kLO, rbb = (tid / kLO) * NB;          // dB: (column, half of the ranks)
    const int ig = tid / 4, rbg = (tid % 4) * NG;              // gh: (token, quarter of the ranks)
    float accb[NB];
#pragma unroll
    for (int k = 0; k < NB; ++k) accb[k] = 0.f;
    for (int rt = rt0; rt < rt1; ++rt) {
        const int buf = (rt - rt0) & 1, r0 = rt * kLT;
        if (rt + 1 < rt1) {
            issue_tile(sG + (buf ^ 1) * kLT * kLP, p.G, p.O, a.S, p.O, r0 + kLT, o0, vecG);
            issue_rows<RB>(sh + (buf ^ 1) * kLT * RB, p.h, a.S, R, r0 + kLT, vech);
            cp_async_commit();
            cp_async_wait_one();
        } else {
            cp_async_wait_all();
        }
        __syncthreads();
        const float *g = sG + buf * kLT * kLP, *hh = sh + buf * kLT * RB;
#pragma unroll 4
        for (int i = 0; i < kLT; ++i) {
            const float gv = g[i * kLP + ob];
            const float4 *h4 = reinterpret_cast<const float4 *>(hh + i * RB + rbb);   // NB % 4 == 0 or NB == 2
            if constexpr (NB % 4 == 0) {
#pragma unroll
                for (int k = 0; k < NB / 4; ++k) {
                    const float4 v = h4[k];
                    accb[4 * k] = fmaf(gv, v.x, accb[4 * k]);
                    accb[4 * k + 1] = fmaf(gv, v.y, accb[4 * k + 1]);
                    accb[4 * k + 2] = fmaf(gv, v.z, accb[4 * k + 2]);
                    accb[4 * k + 3] = fmaf(gv, v.w, accb[4 * k + 3]);
                }
            } else {
#pragma unroll
                for (int k = 0; k < NB; ++k) accb[k] = fmaf(gv, hh[i * RB + rbb + k], accb[k]);
            }
        }
        float accg[NG];
#pragma unroll
        for (int k = 0; k < NG; ++k) accg[k] = 0.f;
#pragma unroll 4
        for (int o = 0; o < kLO; ++o) {
            const float gv = g[ig * kLP + o];
            if constexpr (NG % 4 == 0) {
#pragma unroll
                for (int k = 0; k < NG / 4; ++k) {
                    const float4 v = reinterpret_cast<const float4 *>(sB + o * RB + rbg)[k];
                    accg[4 * k] = fmaf(gv, v.x, accg[4 * k]);
                    accg[4 * k + 1] = fmaf(gv, v.y, accg[4 * k + 1]);
                    accg[4 * k + 2] = fmaf(gv, v.z, accg[4 * k + 2]);
                    accg[4 * k + 3] = fmaf(gv, v.w, accg[4 * k + 3]);
                }
            } else {
#pragma unroll
                for (int k = 0; k < NG; ++k) accg[k] = fmaf(gv, sB[o * RB + rbg + k], accg[k]);
            }
        }
        if (r0 + ig < a.S) {
            float *dst = p.part_gh + (int64_t(ot) * a.S + r0 + ig) * R;
#pragma unroll
            for (int k = 0; k < NG; ++k)
                if (rbg + k < R) dst[rbg + k] = accg[k];
        }
        __syncthreads();                           // buffer buf is refilled next iteration
    }
    if (o0 + ob < p.O) {
        float *dst = p.part_b + (int64_t(blockIdx.y) * p.O + o0 + ob) * R;
#pragma unroll
        for (int k = 0; k < NB; ++k)
            if (rbb + k < R) dst[rbb + k] = accb[k];
    }
}

// Rank-16 G pass with 4 x 4 register blocks (the layers' rank): per tile, dB as 128
// columns x 16 ranks = 32 column quads x 4 rank quads x 2 halves of the 64 rows, and
// gh as 64 rows x 16 ranks = 16 row groups x 4 rank quads x 4 column quarters; every
// float4 read from shared memory feeds four FMAs.  The halves / quarters meet in shared
// memory in a fixed order.
__global__ void __launch_bounds__(256) lora_gpass16_kernel(LoraSeqArgs a) {
    constexpr int RB = 16;
    extern __shared__ float4 sm4[];
    float *sG = reinterpret_cast<float *>(sm4);   // 2 x [kLT][kLP]
    float *sh = sG + 2 * kLT * kLP;               // 2 x [kLT][RB]
    float *sB = sh + 2 * kLT * RB;                // [kLO][RB]
    float *red = sB + kLO * RB;                   // [4][kLT][RB] gh quarters, then [2][kLO][RB] dB halves
    const int side = (a.nside > 1 && int(blockIdx.x) >= a.side[1].blk0) ? 1 : 0;
    const LoraSide &p = a.side[side];
    const int ot = int(blockIdx.x) - p.blk0, o0 = ot * kLO, R = a.rank, tid = threadIdx.x;
    const int rt0 = blockIdx.y * a.tpc_b, rt1 = min(rt0 + a.tpc_b, a.n_rt);
    const bool vecG = p.vecG != 0, vech = a.vech != 0;
    for (int e = tid; e < kLO * RB; e += 256) {
        const int o = e / RB, r = e % RB;
        sB[e] = (r < R && o0 + o < p.O) ? p.l.b[int64_t(o0 + o) * R + r] : 0.f;
    }
    issue_tile(sG, p.G, p.O, a.S, p.O, rt0 * kLT, o0, vecG);
    issue_rows<RB>(sh, p.h, a.S, R, rt0 * kLT, vech);
    cp_async_commit();
    // dB: column quad cq, rank quad rq, row half ih
    const int cq = tid & 31, rq = (tid >> 5) & 3, ih = tid >> 7;
    // gh: rows iq + 16 u (u = 0..3), rank quad gq, column quarter oq
    const int iq = tid & 15, gq = (tid >> 4) & 3, oq = tid >> 6;
    float accb[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int k = 0; k < 4; ++k) accb[u][k] = 0.f;
    for (int rt = rt0; rt < rt1; ++rt) {
        const int buf = (rt - rt0) & 1, r0 = rt * kLT;
        if (rt + 1 < rt1) {
            issue_tile(sG + (buf ^ 1) * kLT * kLP, p.G, p.O, a.S, p.O, r0 + kLT, o0, vecG);
            issue_rows<RB>(sh + (buf ^ 1) * kLT * RB, p.h, a.S, R, r0 + kLT, vech);
            cp_async_commit();
            cp_async_wait_one();
        } else {
            cp_async_wait_all();
        }
        __syncthreads();
        const float *g = sG + buf * kLT * kLP, *hh = sh + buf * kLT * RB;
#pragma unroll 4
        for (int i = ih * (kLT / 2); i < (ih + 1) * (kLT / 2); ++i) {
            const float4 gv = *reinterpret_cast<const float4 *>(g + i * kLP + 4 * cq);
            const float4 hv = *reinterpret_cast<const float4 *>(hh + i * RB + 4 * rq);
            const float gc[4] = {gv.x, gv.y, gv.z, gv.w}, hr[4] = {hv.x, hv.y, hv.z, hv.w};
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int k = 0; k < 4; ++k) accb[u][k] = fmaf(gc[u], hr[k], accb[u][k]);
        }
        float accg[4][4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int k = 0; k < 4; ++k) accg[u][k] = 0.f;
#pragma unroll 2
        for (int o = oq * (kLO / 4); o < (oq + 1) * (kLO / 4); o += 4) {
            float gr[4][4], bo[4][4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float4 v = *reinterpret_cast<const float4 *>(g + (iq + 16 * u) * kLP + o);
                gr[u][0] = v.x; gr[u][1] = v.y; gr[u][2] = v.z; gr[u][3] = v.w;
                const float4 w = *reinterpret_cast<const float4 *>(sB + (o + u) * RB + 4 * gq);
                bo[u][0] = w.x; bo[u][1] = w.y; bo[u][2] = w.z; bo[u][3] = w.w;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int v = 0; v < 4; ++v)
#pragma unroll
                    for (int k = 0; k < 4; ++k) accg[u][k] = fmaf(gr[u][v], bo[v][k], accg[u][k]);
        }
        // gh partial of the tile: sum the four column quarters in order
#pragma unroll
        for (int u = 0; u < 4; ++u)
            *reinterpret_cast<float4 *>(red + (oq * kLT + iq + 16 * u) * RB + 4 * gq) =
                make_float4(accg[u][0], accg[u][1], accg[u][2], accg[u][3]);
        __syncthreads();
        for (int e = tid; e < kLT * RB; e += 256) {
            const int i = e / RB, r = e % RB;
            const float v = red[e] + red[kLT * RB + e] + red[2 * kLT * RB + e] + red[3 * kLT * RB + e];
            if (r < R && r0 + i < a.S) p.part_gh[(int64_t(ot) * a.S + r0 + i) * R + r] = v;
        }
        __syncthreads();                           // buffer buf and red are reused next iteration
    }
    // dB partial of the chunk: sum the two row halves in order
#pragma unroll
    for (int u = 0; u < 4; ++u)
        *reinterpret_cast<float4 *>(red + (ih * kLO + 4 * cq + u) * RB + 4 * rq) =
            make_float4(accb[u][0], accb[u][1], accb[u][2], accb[u][3]);
    __syncthreads();
    for (int e = tid; e < kLO * RB; e += 256) {
        const int o = e / RB, r = e % RB;
        if (r < R && o0 + o < p.O)
            p.part_b[(int64_t(blockIdx.y) * p.O + o0 + o) * R + r] = red[e] + red[kLO * RB + e];
    }
}

// sum of p[k stride], k = 0 .. n - 1, in index order, sixteen loads in flight at a time
// (the tail batch included)
__device__ __forceinline__ float ordered_sum16(const float *p, int n, int64_t stride) {
    float acc = 0.f;
    for (int k = 0; k < n; k += 16) {
        const int m = min(16, n - k);
        float v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (j < m) v[j] = p[int64_t(k + j) * stride];
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (j < m) acc += v[j];
    }
    return acc;
}

// the same sum, B loads in flight at a time
template <int B>
__device__ __forceinline__ float ordered_sum(const float *p, int n, int64_t stride) {
    float acc = 0.f;
    int k = 0;
    for (; k + B <= n; k += B) {
        float v[B];
#pragma unroll
        for (int j = 0; j < B; ++j) v[j] = p[int64_t(k + j) * stride];
#pragma unroll
        for (int j = 0; j < B; ++j) acc += v[j];
    }
    for (; k < n; ++k) acc += p[int64_t(k) * stride];
    return acc;
}

__global__ void __launch_bounds__(256) lora_gh_sum_kernel(LoraSeqArgs a) {
    const int64_t n = int64_t(a.S) * a.rank;
    int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    int side = 0;
    if (e >= n) {
        side = 1;
        e -= n;
    }
    if (side >= a.nside || e >= n) return;
    const LoraSide &p = a.side[side];
    p.gh[e] = p.s * ordered_sum16(p.part_gh + e, p.n_ot, n);
}

// Block (column tile of x, chunk of row tiles): one pass over its x tiles, staged two
// deep, gives the dA partials of the chunk for every side (registers across its tiles).
template <int RB>
__global__ void __launch_bounds__(256) lora_xpass_kernel(LoraSeqArgs a) {
    extern __shared__ float4 sm4[];
    float *sx = reinterpret_cast<float *>(sm4);   // 2 x [kLT][kLP]
    float *sg = sx + 2 * kLT * kLP;               // 2 x [nside][kLT][RB]
    const int c0 = blockIdx.x * kLO, R = a.rank, tid = threadIdx.x;
    const int rt0 = blockIdx.y * a.tpc_a, rt1 = min(rt0 + a.tpc_a, a.n_rt);
    const bool vecx = a.vecx != 0, vech = a.vech != 0;
    auto issue = [&](int rt, int buf) {
        issue_tile(sx + buf * kLT * kLP, a.x, a.C, a.S, a.C, rt * kLT, c0, vecx);
        for (int sd = 0; sd < a.nside; ++sd)
            issue_rows<RB>(sg + (buf * 2 + sd) * kLT * RB, a.side[sd].gh, a.S, R, rt * kLT, vech);
        cp_async_commit();
    };
    issue(rt0, 0);
    constexpr int NB = RB / 2;
    const int c = tid % kLO, rb = (tid / kLO) * NB;
    float acc[2][NB];
#pragma unroll
    for (int sd = 0; sd < 2; ++sd)
#pragma unroll
        for (int k = 0; k < NB; ++k) acc[sd][k] = 0.f;
    for (int rt = rt0; rt < rt1; ++rt) {
        const int buf = (rt - rt0) & 1;
        if (rt + 1 < rt1) {
            issue(rt + 1, buf ^ 1);
            cp_async_wait_one();
        } else {
            cp_async_wait_all();
        }
        __syncthreads();
        const float *xs = sx + buf * kLT * kLP;
#pragma unroll
        for (int sd = 0; sd < 2; ++sd) {
            if (sd >= a.nside) break;
            const float *g = sg + (buf * 2 + sd) * kLT * RB;
#pragma unroll 4
            for (int i = 0; i < kLT; ++i) {
                const float xv = xs[i * kLP + c];
                if constexpr (NB % 4 == 0) {
#pragma unroll
                    for (int k = 0; k < NB / 4; ++k) {
                        const float4 v = reinterpret_cast<const float4 *>(g + i * RB + rb)[k];
                        acc[sd][4 * k] = fmaf(v.x, xv, acc[sd][4 * k]);
                        acc[sd][4 * k + 1] = fmaf(v.y, xv, acc[sd][4 * k + 1]);
                        acc[sd][4 * k + 2] = fmaf(v.z, xv, acc[sd][4 * k + 2]);
                        acc[sd][4 * k + 3] = fmaf(v.w, xv, acc[sd][4 * k + 3]);
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < NB; ++k) acc[sd][k] = fmaf(g[i * RB + rb + k], xv, acc[sd][k]);
                }
            }
        }
        __syncthreads();                           // buffer buf is refilled next iteration
    }
    if (c0 + c < a.C) {
#pragma unroll
        for (int sd = 0; sd < 2; ++sd) {
            if (sd >= a.nside) break;
            float *dst = a.side[sd].part_a + int64_t(blockIdx.y) * R * a.C + c0 + c;
#pragma unroll
            for (int k = 0; k < NB; ++k)
                if (rb + k < R) dst[int64_t(rb + k) * a.C] = acc[sd][k];
        }
    }
}

// Rank-16 x pass with 4 x 4 register blocks: dA of each side as 16 ranks x 128 columns =
// 4 rank quads x 32 column quads x 2 halves of the 64 rows; the halves meet in shared
// memory (in the x buffers, free after the last tile) in a fixed order.
__global__ void __launch_bounds__(256) lora_xpass16_kernel(LoraSeqArgs a) {
    constexpr int RB = 16;
    extern __shared__ float4 sm4[];
    float *sx = reinterpret_cast<float *>(sm4);   // 2 x [kLT][kLP]
    float *sg = sx + 2 * kLT * kLP;               // 2 x [nside][kLT][RB]
    const int c0 = blockIdx.x * kLO, R = a.rank, tid = threadIdx.x;
    const int rt0 = blockIdx.y * a.tpc_a, rt1 = min(rt0 + a.tpc_a, a.n_rt);
    const bool vecx = a.vecx != 0, vech = a.vech != 0;
    auto issue = [&](int rt, int buf) {
        issue_tile(sx + buf * kLT * kLP, a.x, a.C, a.S, a.C, rt * kLT, c0, vecx);
        for (int sd = 0; sd < a.nside; ++sd)
            issue_rows<RB>(sg + (buf * 2 + sd) * kLT * RB, a.side[sd].gh, a.S, R, rt * kLT, vech);
        cp_async_commit();
    };
    issue(rt0, 0);
    const int cq = tid & 31, rq = (tid >> 5) & 3, ih = tid >> 7;
    float acc[2][4][4];                            // [side][column][rank]
#pragma unroll
    for (int sd = 0; sd < 2; ++sd)
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[sd][u][k] = 0.f;
    for (int rt = rt0; rt < rt1; ++rt) {
        const int buf = (rt - rt0) & 1;
        if (rt + 1 < rt1) {
            issue(rt + 1, buf ^ 1);
            cp_async_wait_one();
        } else {
            cp_async_wait_all();
        }
        __syncthreads();
        const float *xs = sx + buf * kLT * kLP;
#pragma unroll 2
        for (int i = ih * (kLT / 2); i < (ih + 1) * (kLT / 2); ++i) {
            const float4 xv = *reinterpret_cast<const float4 *>(xs + i * kLP + 4 * cq);
            const float xc[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
            for (int sd = 0; sd < 2; ++sd) {
                if (sd >= a.nside) break;
                const float4 gv = *reinterpret_cast<const float4 *>(sg + ((buf * 2 + sd) * kLT + i) * RB + 4 * rq);
                const float gr[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int k = 0; k < 4; ++k) acc[sd][u][k] = fmaf(gr[k], xc[u], acc[sd][u][k]);
            }
        }
        __syncthreads();                           // buffer buf is refilled next iteration
    }
    // halves in order: red[ih][side][rank][column]
    float *red = sx;
#pragma unroll
    for (int sd = 0; sd < 2; ++sd)
#pragma unroll
        for (int k = 0; k < 4; ++k)
            *reinterpret_cast<float4 *>(red + ((ih * 2 + sd) * RB + 4 * rq + k) * kLO + 4 * cq) =
                make_float4(acc[sd][0][k], acc[sd][1][k], acc[sd][2][k], acc[sd][3][k]);
    __syncthreads();
    for (int sd = 0; sd < a.nside; ++sd) {
        float *dst = a.side[sd].part_a + int64_t(blockIdx.y) * R * a.C;
        for (int e = tid; e < RB * kLO; e += 256) {
            const int r = e / kLO, c = e % kLO;
            if (r < R && c0 + c < a.C)
                dst[int64_t(r) * a.C + c0 + c] = red[(sd * RB + r) * kLO + c] + red[((2 + sd) * RB + r) * kLO + c];
        }
    }
}

// One thread per parameter of [A_0 | B_0 | A_1 | B_1].
__global__ void __launch_bounds__(256) lora_seq_adamw_kernel(LoraSeqArgs a, AdamCoef ka, AdamCoef kb,
                                                             double *sumsq) {
    __shared__ float red[32];
    int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    float ssa = 0.f, ssb = 0.f;
    const bool step = a.status == nullptr || __ldcg(a.status + kStatusGate) == 0u;
    for (int sd = 0; sd < a.nside; ++sd) {
        const LoraSide &p = a.side[sd];
        const int64_t nA = int64_t(a.rank) * a.C, nB = int64_t(p.O) * a.rank;
        if (e < 0) break;
        // the parameter and its moments are loaded before the partial sums, so that both
        // rounds of loads are in flight together
        if (e < nA) {
            float w = 0.f, m = 0.f, v = 0.f;
            if (step) {
                w = p.l.a[e];
                m = p.l.m_a[e];
                v = p.l.v_a[e];
            }
            const float g = ordered_sum<8>(p.part_a + e, a.nrc_a, nA);
            if (p.l.grad_a) p.l.grad_a[e] = g;
            if (step) {
                p.l.a[e] = adam_elem(w, g, m, v, ka);
                p.l.m_a[e] = m;
                p.l.v_a[e] = v;
            }
            ssa = g * g;
            e = -1;
        } else if (e < nA + nB) {
            const int64_t f = e - nA;
            float w = 0.f, m = 0.f, v = 0.f;
            if (step) {
                w = p.l.b[f];
                m = p.l.m_b[f];
                v = p.l.v_b[f];
            }
            const float g = p.s * ordered_sum<8>(p.part_b + f, a.nrc_b, nB);
            if (p.l.grad_b) p.l.grad_b[f] = g;
            if (step) {
                p.l.b[f] = adam_elem(w, g, m, v, kb);
                p.l.m_b[f] = m;
                p.l.v_b[f] = v;
            }
            ssb = g * g;
            e = -1;
        } else {
            e -= nA + nB;
        }
    }
    if (sumsq) {
        const float ta = block_sum(ssa, red);
        const float tb = block_sum(ssb, red);
        if (threadIdx.x == 0) {
            if (ta != 0.f) atomicAdd(sumsq, double(ta));
            if (tb != 0.f) atomicAdd(sumsq + 1, double(tb));
        }
    }
}

struct SideBytes {
    size_t part_b, part_gh, gh, part_a, total;
};

SideBytes side_bytes(int64_t S, int out_dim, int in_dim, int rank) {
    auto r256 = [](size_t b) { return (b + 255) & ~size_t(255); };
    const int64_t n_rt = ceil_div(S, int64_t(kLT)), n_ot = ceil_div(int64_t(out_dim), int64_t(kLO));
    SideBytes b;
    b.part_b = r256(size_t(n_rt) * out_dim * rank * 4);
    b.part_gh = r256(size_t(n_ot) * S * rank * 4);
    b.gh = r256(size_t(S) * rank * 4);
    b.part_a = r256(size_t(n_rt) * rank * in_dim * 4);
    b.total = b.part_b + b.part_gh + b.gh + b.part_a;
    return b;
}

template <int RB>
int lora_seq_run(LoraSeqArgs a, int n_ot_total, const AdamCoef &ka, const AdamCoef &kb, double *sumsq,
                 cudaStream_t st, float *din, uint32_t *tc) {
    if constexpr (RB == 16) {
        // the tensor-core passes, with partial sums over chunks of 128-token tiles
        LoraTcJob tj[2] = {};
        for (int sd = 0; sd < a.nside; ++sd) {
            const LoraSide &p = a.side[sd];
            tj[sd] = LoraTcJob{p.G, p.h, p.l.b, p.gh, p.part_gh, p.part_b, p.part_a, p.O};
        }
        if (tc != nullptr && lora_tc_supported(a.S, a.C, a.rank, a.x, tj, a.nside)) {
            int tpc = 0;
            a.nrc_b = lora_tc_chunks(a.S, n_ot_total, tpc);
            TLB_TRY(lora_tc_gpass_launch(a.S, tj, a.nside, tpc, tc, st));
            const int64_t ngh = int64_t(a.nside) * a.S * a.rank;
            lora_gh_sum_kernel<<<unsigned(ceil_div(ngh, int64_t(256))), 256, 0, st>>>(a);
            TLB_TRY(check_launch("lora_gh_sum"));
            if (din != nullptr) {
                const float *gh[2] = {a.side[0].gh, a.side[1].gh};
                const float *A[2] = {a.side[0].l.a, a.side[1].l.a};
                TLB_TRY(lora_din_launch(a.S, a.C, a.rank, gh, A, a.nside, din, st));
            }
            a.nrc_a = lora_tc_chunks(a.S, int(ceil_div(a.C, kLO)), tpc);
            TLB_TRY(lora_tc_xpass_launch(a.S, a.C, a.x, tj, a.nside, tpc, tc, st));
            int64_t np = 0;
            for (int sd = 0; sd < a.nside; ++sd) np += int64_t(a.rank) * (a.C + a.side[sd].O);
            lora_seq_adamw_kernel<<<unsigned(ceil_div(np, int64_t(256))), 256, 0, st>>>(a, ka, kb, sumsq);
            return check_launch("lora_seq_adamw");
        }
    }
    // chunks of row tiles per block: at most two blocks per SM in each pass (one wave)
    const int target = 2 * num_sms();
    a.nrc_b = int(std::min<int64_t>(a.n_rt, std::max<int64_t>(1, target / n_ot_total)));
    a.tpc_b = int(ceil_div(a.n_rt, a.nrc_b));
    a.nrc_b = int(ceil_div(a.n_rt, a.tpc_b));
    const int n_ct = int(ceil_div(a.C, kLO));
    a.nrc_a = int(std::min<int64_t>(a.n_rt, std::max<int64_t>(1, target / n_ct)));
    a.tpc_a = int(ceil_div(a.n_rt, a.nrc_a));
    a.nrc_a = int(ceil_div(a.n_rt, a.tpc_a));
    const size_t smg = size_t(2 * kLT * kLP + 2 * kLT * RB + kLO * RB) * 4;
    const size_t smx = size_t(2 * kLT * kLP + 4 * kLT * RB) * 4;
    // two blocks per SM need the largest shared-memory carveout (the default split may
    // leave room for one, which turns each pass into two waves)
    {
        static std::once_flag once;
        cudaError_t err = cudaSuccess;
        std::call_once(once, [&] {
            const void *ks[] = {reinterpret_cast<const void *>(lora_gpass_kernel<4>),
                                reinterpret_cast<const void *>(lora_gpass_kernel<8>),
                                reinterpret_cast<const void *>(lora_gpass_kernel<16>),
                                reinterpret_cast<const void *>(lora_gpass_kernel<32>),
                                reinterpret_cast<const void *>(lora_gpass_kernel<64>),
                                reinterpret_cast<const void *>(lora_xpass_kernel<4>),
                                reinterpret_cast<const void *>(lora_xpass_kernel<8>),
                                reinterpret_cast<const void *>(lora_xpass_kernel<16>),
                                reinterpret_cast<const void *>(lora_xpass_kernel<32>),
                                reinterpret_cast<const void *>(lora_xpass_kernel<64>),
                                reinterpret_cast<const void *>(lora_gpass16_kernel),
                                reinterpret_cast<const void *>(lora_xpass16_kernel)};
            for (const void *k : ks) {
                const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                                                           int(cudaSharedmemCarveoutMaxShared));
                if (e != cudaSuccess && err == cudaSuccess) err = e;
            }
        });
        TLB_CUDA(err);
    }
    if (smg > 48 * 1024)
        TLB_CUDA(cudaFuncSetAttribute(lora_gpass_kernel<RB>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smg)));
    if (smx > 48 * 1024) {
        TLB_CUDA(cudaFuncSetAttribute(lora_xpass_kernel<RB>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smx)));
        if constexpr (RB == 16)
            TLB_CUDA(cudaFuncSetAttribute(lora_xpass16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smx)));
    }
    if constexpr (RB == 16) {
        const size_t sm16 = smg + size_t(4 * kLT * RB) * 4;
        TLB_CUDA(cudaFuncSetAttribute(lora_gpass16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sm16)));
        lora_gpass16_kernel<<<dim3(unsigned(n_ot_total), unsigned(a.nrc_b)), 256, sm16, st>>>(a);
    } else {
        lora_gpass_kernel<RB><<<dim3(unsigned(n_ot_total), unsigned(a.nrc_b)), 256, smg, st>>>(a);
    }
    TLB_TRY(check_launch("lora_gpass"));
    const int64_t ngh = int64_t(a.nside) * a.S * a.rank;
    lora_gh_sum_kernel<<<unsigned(ceil_div(ngh, int64_t(256))), 256, 0, st>>>(a);
    TLB_TRY(check_launch("lora_gh_sum"));
    if (din != nullptr) {      // the LoRA A paths of the exact input gradient, before AdamW moves A
        const float *gh[2] = {a.side[0].gh, a.side[1].gh};
        const float *A[2] = {a.side[0].l.a, a.side[1].l.a};
        TLB_TRY(lora_din_launch(a.S, a.C, a.rank, gh, A, a.nside, din, st));
    }
    if constexpr (RB == 16) lora_xpass16_kernel<<<dim3(unsigned(n_ct), unsigned(a.nrc_a)), 256, smx, st>>>(a);
    else lora_xpass_kernel<RB><<<dim3(unsigned(n_ct), unsigned(a.nrc_a)), 256, smx, st>>>(a);
    TLB_TRY(check_launch("lora_xpass"));
    int64_t np = 0;
    for (int sd = 0; sd < a.nside; ++sd) np += int64_t(a.rank) * (a.C + a.side[sd].O);
    lora_seq_adamw_kernel<<<unsigned(ceil_div(np, int64_t(256))), 256, 0, st>>>(a, ka, kb, sumsq);
    return check_launch("lora_seq_adamw");
}

}  // namespace

size_t lora_seq_bytes(int64_t S, int out_dim, int in_dim, int rank) {
    return side_bytes(S, out_dim, in_dim, rank).total;
}

int lora_seq_launch(int64_t S, int in_dim, int rank, float alpha, const float *x, const LoraJob *jobs, int njobs,
                    const tlb_adamw_cfg &adam, double *sumsq, cudaStream_t st, const uint32_t *status,
                    float *din, uint32_t *tc) {
    if (S == 0 || njobs == 0) return TLB_OK;
    TLB_REQUIRE(njobs <= 2, TLB_EINVAL, "lora: at most two adapters per call");
    TLB_REQUIRE(rank >= 1 && rank <= 64, TLB_EINVAL, "lora: rank must be in 1..64");
    const int64_t n_rt = ceil_div(S, int64_t(kLT));
    TLB_REQUIRE(n_rt <= 65535, TLB_EUNSUPPORTED, "lora: S = %lld too long", (long long)S);
    LoraSeqArgs a{};
    a.x = x;
    a.status = status;
    a.nside = njobs;
    a.S = int(S);
    a.C = in_dim;
    a.rank = rank;
    a.n_rt = int(n_rt);
    a.vecx = (in_dim % 4 == 0 && aligned16(x)) ? 1 : 0;
    // rows of h and gh stream with 16-byte copies when they are exactly one padded row
    const int rb = rank <= 4 ? 4 : rank <= 8 ? 8 : rank <= 16 ? 16 : rank <= 32 ? 32 : 64;
    a.vech = rank == rb ? 1 : 0;
    int blk = 0;
    for (int sd = 0; sd < njobs; ++sd) {
        const LoraJob &j = jobs[sd];
        LoraSide &p = a.side[sd];
        const SideBytes b = side_bytes(S, j.out_dim, in_dim, rank);
        char *base = static_cast<char *>(j.scratch);
        TLB_REQUIRE((reinterpret_cast<uintptr_t>(base) & 255u) == 0, TLB_EINVAL, "lora: scratch not 256-byte aligned");
        p.G = j.G;
        p.h = j.h;
        if (!aligned16(j.h)) a.vech = 0;
        p.O = j.out_dim;
        p.n_ot = int(ceil_div(int64_t(j.out_dim), int64_t(kLO)));
        p.blk0 = blk;
        p.vecG = (j.out_dim % 4 == 0 && aligned16(j.G)) ? 1 : 0;
        p.s = alpha / float(rank);
        p.l = j.l;
        p.part_b = reinterpret_cast<float *>(base);
        p.part_gh = reinterpret_cast<float *>(base + b.part_b);
        p.gh = reinterpret_cast<float *>(base + b.part_b + b.part_gh);
        p.part_a = reinterpret_cast<float *>(base + b.part_b + b.part_gh + b.gh);
        blk += p.n_ot;
    }
    const AdamCoef kb = adam_coef(adam, adam.lr_b_mult);
    const AdamCoef ka = adam_coef(adam, 1.0f);
    if (rank <= 4) return lora_seq_run<4>(a, blk, ka, kb, sumsq, st, din, tc);
    if (rank <= 8) return lora_seq_run<8>(a, blk, ka, kb, sumsq, st, din, tc);
    if (rank <= 16) return lora_seq_run<16>(a, blk, ka, kb, sumsq, st, din, tc);
    if (rank <= 32) return lora_seq_run<32>(a, blk, ka, kb, sumsq, st, din, tc);
    return lora_seq_run<64>(a, blk, ka, kb, sumsq, st, din, tc);
}


// ------------------------------------------------------------------ LoRA-A paths of d_in

namespace {

constexpr int kDinRows = 16;

struct LoraDinArgs {
    const float *gh[2];          // [S, rank] each: s G B with B before its update
    const float *A[2];           // [rank, C] each, before its update
    int njobs, S, C, rank;
    float *dn1;                  // [S, C], added into
};

// Block = 16 rows x 256 columns, one column per thread: the rows' gh values of both
// adapters in shared memory, then dn1[row, c] += sum_t sum_r gh_t[row, r] A_t[r, c].  A
// thread loads 16 of its A values at a time before it uses them (loads in flight), and
// each serves the block's 16 rows.
__global__ void __launch_bounds__(256) lora_din_kernel(LoraDinArgs a) {
    extern __shared__ float sgh[];                  // [kDinRows][njobs][rank]
    const int r0 = blockIdx.y * kDinRows;
    const int nrows = min(kDinRows, a.S - r0);
    const int per = a.njobs * a.rank;
    for (int e = threadIdx.x; e < kDinRows * per; e += blockDim.x) {
        const int row = e / per, t = (e % per) / a.rank, r = e % a.rank;
        sgh[e] = row < nrows ? (t == 0 ? a.gh[0] : a.gh[1])[int64_t(r0 + row) * a.rank + r] : 0.f;
    }
    __syncthreads();
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= a.C) return;
    float acc[kDinRows];
#pragma unroll
    for (int row = 0; row < kDinRows; ++row) acc[row] = 0.f;
    for (int t = 0; t < a.njobs; ++t) {
        const float *A = t == 0 ? a.A[0] : a.A[1];
        for (int rc = 0; rc < a.rank; rc += 16) {
            float av[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) av[k] = rc + k < a.rank ? __ldg(A + int64_t(rc + k) * a.C + c) : 0.f;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                if (rc + k >= a.rank) break;
                const float *g = sgh + t * a.rank + rc + k;
#pragma unroll
                for (int row = 0; row < kDinRows; ++row) acc[row] = fmaf(g[row * per], av[k], acc[row]);
            }
        }
    }
#pragma unroll
    for (int row = 0; row < kDinRows; ++row)      // constant bound: acc stays in registers
        if (row < nrows) a.dn1[int64_t(r0 + row) * a.C + c] += acc[row];
}

}  // namespace

int lora_din_launch(int64_t S, int in_dim, int rank, const float *const *gh, const float *const *A, int njobs,
                    float *dn1, cudaStream_t st) {
    if (S == 0 || njobs == 0) return TLB_OK;
    TLB_REQUIRE(njobs <= 2 && rank >= 1 && rank <= 64, TLB_EINVAL, "lora d_in: bad adapter count or rank");
    LoraDinArgs a{};
    for (int t = 0; t < njobs; ++t) {
        a.gh[t] = gh[t];
        a.A[t] = A[t];
    }
    a.njobs = njobs;
    a.S = int(S);
    a.C = in_dim;
    a.rank = rank;
    a.dn1 = dn1;
    const size_t sm = size_t(kDinRows) * njobs * rank * 4;
    lora_din_kernel<<<dim3(unsigned(ceil_div(in_dim, 256)), unsigned(ceil_div(S, int64_t(kDinRows)))), 256, sm,
                      st>>>(a);
    return check_launch("lora_din");
}

}  // namespace tlb
