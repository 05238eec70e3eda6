// LoRA adapter gradients on the tensor cores (tcgen05, kind::tf32) at rank 16, for the
// sequence layers whose attention backward runs on tcgen05 ([RS] "LoRA Q backward" and
// "LoRA V backward"; the scale s = alpha / rank is applied by the consumers of the
// partial sums, as for the CUDA-core passes):
//   G pass, per (adapter, 128-column tile of G, chunk of 128-token tiles t):
//     gh_part[tile][rows of t] = G_t B_tile       M 128 tokens,  N 16, K 128 columns
//     dB_part[chunk]          += G_t^T h_t        M 128 columns, N 16, K 128 tokens
//   x pass, per (128-column tile of x, chunk of 128-token tiles t):
//     dA_part[chunk]^T        += x_t^T [gh_0 | gh_1]_t    M 128 columns, N 16 per adapter
// G_t and x_t arrive by TMA as four 32-column boxes with 128-byte swizzle.  Sixteen writer
// warps round them to tf32 and write their transposes into tensor memory, the A operand
// of the token contractions (G_t also goes back rounded in place: the A operand of gh).
// The same warps write the small operands (B^T, h^T, gh^T) in the swizzled K-major
// layout.  The partial sums keep the layouts of the CUDA-core passes, so the gh sum and
// the AdamW kernel serve both.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"
#include "tc.cuh"

namespace tlb {

namespace {

constexpr int kTT = 128;                        // tokens per tile
constexpr int kCT = 128;                        // columns per tile
constexpr int kRk = 16;                         // rank
constexpr int kThreads = 576;                   // producer warp, MMA warp, 16 writer warps
constexpr int kWriters = 16;
constexpr int kWT = kTT / (kWriters / 4);       // tokens of a tile per writer warp (4 warps per lane quarter)
constexpr int kTileBytes = kTT * kCT * 4;       // 64 KB: four [128 rows][32 floats] boxes
constexpr int kBoxBytes = kTT * 128;
constexpr int kSlots = 3;                       // tiles of G or x staged ahead

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ uint32_t ld_shared_u32(const uint8_t *p) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)));
    return v;
}
__device__ __forceinline__ void st_shared_u32(uint8_t *p, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(smem_u32(p)), "r"(v) : "memory");
}

// Byte offset of element (row r, column k) of a K-major operand built of 32-column atoms
// of `rows` rows (128-byte rows, 128-byte swizzle), the layout TMA writes for a box of
// 32 floats by `rows` rows.
__device__ __forceinline__ uint32_t kmaj_off(int rows, int r, int k) {
    return uint32_t((k >> 5) * rows * 128 + r * 128) + (uint32_t(((k & 31) >> 2) ^ (r & 7)) << 4) +
           uint32_t((k & 3) * 4);
}

struct LoraTcSide {
    CUtensorMap g;              // G [S, O], box {32, 128}
    const float *h;             // [S, 16]
    const float *b;             // B [O, 16], before its update
    const float *gh;            // [S, 16] (x pass)
    float *part_gh;             // [n_ot][S][16]
    float *part_b;              // [nrc_b][O][16]
    float *part_a;              // [nrc_a][16][C]
    int O, blk0;
};

struct LoraTcParams {
    LoraTcSide side[2];
    CUtensorMap x;              // x [S, C], box {32, 128}
    int nside, S, C, tpc, n_tt;
    uint32_t *status;
};

// ------------------------------------------------------------------ G pass

struct GLayout {
    static constexpr int HT_BYTES = 4 * kRk * 128;            // [16 ranks][128 tokens]: four atoms
    static constexpr int HT0 = kSlots * kTileBytes, BT0 = HT0 + 2 * HT_BYTES, TOTAL = BT0 + HT_BYTES;
    // tensor memory: two G^T buffers [128 columns][128 tokens], two gh accumulators
    // [128 tokens][16], the dB accumulator [128 columns][16]
    static constexpr uint32_t TGT = 0, TGH = 2 * kTT, TDB = TGH + 2 * kRk, COLS = 512;
};

__global__ void __launch_bounds__(kThreads, 1) lora_tc_gpass_kernel(const __grid_constant__ LoraTcParams p) {
    using Ly = GLayout;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    // full / gfree: G slot landed / read by the gh MMA; ready: G_t rounded, G_t^T and h_t^T
    // written; tfree: the dB MMA of the tile done (h^T slot and G^T buffer free); ghfull /
    // ghfree: gh accumulator
    __shared__ uint64_t full[kSlots], gfree[kSlots], ready[2], tfree[2], ghfull[2], ghfree[2], dfull;
    __shared__ uint32_t tmem_base;
    __shared__ int s_abort, s_issued;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sd = (p.nside > 1 && int(blockIdx.x) >= p.side[1].blk0) ? 1 : 0;
    const LoraTcSide &q = p.side[sd];
    const int ot = int(blockIdx.x) - q.blk0, o0 = ot * kCT;
    const int t0 = int(blockIdx.y) * p.tpc, nt = min(p.tpc, p.n_tt - t0);

    if (threadIdx.x == 0) {
        s_abort = 0;
        s_issued = 0;
        for (int b = 0; b < kSlots; ++b) {
            mbar_init(&full[b], 1);
            mbar_init(&gfree[b], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ready[b], kWriters);
            mbar_init(&tfree[b], 1);
            mbar_init(&ghfull[b], 1);
            mbar_init(&ghfree[b], 4);
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
        // ------------------------------------------------ TMA producer, kSlots tiles ahead
        if (lane == 0) {
            for (int t = 0; t < nt; ++t) {
                const int b = t % kSlots;
                if (t >= kSlots && !mbar_wait(&gfree[b], (t / kSlots - 1) & 1, p.status, 80u)) {
                    s_abort = 1;
                    break;
                }
                mbar_arrive_expect_tx(&full[b], kTileBytes);
                for (int k = 0; k < 4; ++k)
                    tma_load_3d(sm + b * kTileBytes + k * kBoxBytes, &q.g, o0 + 32 * k, (t0 + t) * kTT, 0, &full[b]);
                s_issued = t + 1;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t id = idesc_tf32(128, kRk);
            bool ok = true;
            for (int t = 0; t < nt; ++t) {
                const int b = t & 1;
                if (!mbar_wait(&ready[b], (t >> 1) & 1, p.status, 81u) ||
                    (t >= 2 && !mbar_wait(&ghfree[b], ((t - 2) >> 1) & 1, p.status, 82u))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // gh_t = G_t B: A = G_t (shared memory, rounded in place), B = B^T
#pragma unroll
                for (int kb = 0; kb < 4; ++kb)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma_tf32(tm + Ly::TGH + uint32_t(b * kRk),
                                 sw128_desc(sm + (t % kSlots) * kTileBytes + kb * kBoxBytes) + 2 * k,
                                 sw128_desc(sm + Ly::BT0 + kb * (kRk * 128)) + 2 * k, id, (kb | k) ? 1u : 0u);
                mma_commit(&ghfull[b]);
                mma_commit(&gfree[t % kSlots]);
                // dB += G_t^T h_t: A = G_t^T (tensor memory), B = h_t^T
#pragma unroll
                for (int k = 0; k < kTT / 8; ++k)
                    mma_tf32_ts(tm + Ly::TDB, tm + Ly::TGT + uint32_t(b * kTT + 8 * k),
                                sw128_desc(sm + Ly::HT0 + b * Ly::HT_BYTES + (k >> 2) * (kRk * 128)) + 2 * (k & 3), id,
                                (t > 0 || k > 0) ? 1u : 0u);
                mma_commit(&tfree[b]);
            }
            if (!ok) s_abort = 1;
            mma_commit(&dfull);
            mbar_wait(&dfull, 0, nullptr, 0u);
        }
    } else {
        // ------------------------------------------------ writers: warp w owns tensor-memory
        // lanes 32 (w % 4) .. (tile columns of this thread) and a quarter hf of the tile's tokens
        const int qq = warp & 3, hf = (warp - 2) >> 2, wi = warp - 2;
        const int col = 32 * qq + lane;
        const uint32_t lane_off = uint32_t(32 * qq) << 16;
        {   // B^T, once: all loads in flight before the stores
            constexpr int NB = kRk * kCT / (kWriters * 32);
            float bv[NB];
#pragma unroll
            for (int k = 0; k < NB; ++k) {
                const int e = wi * 32 + lane + k * kWriters * 32, c = e >> 4, r = e & 15;
                bv[k] = o0 + c < q.O ? __ldg(q.b + int64_t(o0 + c) * kRk + r) : 0.f;
            }
#pragma unroll
            for (int k = 0; k < NB; ++k) {
                const int e = wi * 32 + lane + k * kWriters * 32, c = e >> 4, r = e & 15;
                st_shared_u32(sm + Ly::BT0 + kmaj_off(kRk, r, c), to_tf32(bv[k]));
            }
        }
        // h_t^T values of this thread (rows past S zero), loaded a tile ahead
        constexpr int NH = kRk * kTT / (kWriters * 32);
        float hv[NH];
        auto load_h = [&](int t) {
            const int s0 = (t0 + t) * kTT;
#pragma unroll
            for (int k = 0; k < NH; ++k) {
                const int e = wi * 32 + lane + k * kWriters * 32, s = e >> 4, r = e & 15;
                hv[k] = s0 + s < p.S ? __ldg(q.h + int64_t(s0 + s) * kRk + r) : 0.f;
            }
        };
        load_h(0);
        bool ok = true;
        for (int t = 0; t <= nt && ok; ++t) {
            if (t < nt) {
                const int b = t & 1;
                if (t >= 2 && !mbar_wait(&tfree[b], ((t - 2) >> 1) & 1, p.status, 83u)) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int k = 0; k < NH; ++k) {
                    const int e = wi * 32 + lane + k * kWriters * 32, s = e >> 4, r = e & 15;
                    st_shared_u32(sm + Ly::HT0 + b * Ly::HT_BYTES + kmaj_off(kRk, r, s), to_tf32(hv[k]));
                }
                if (t + 1 < nt) load_h(t + 1);
                if (!mbar_wait(&full[t % kSlots], (t / kSlots) & 1, p.status, 84u)) {
                    ok = false;
                    break;
                }
                uint8_t *gt = sm + (t % kSlots) * kTileBytes;
#pragma unroll 1
                for (int c16 = 0; c16 < kWT; c16 += 16) {
                    uint32_t v[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[j] = ld_shared_u32(gt + kmaj_off(kTT, hf * kWT + c16 + j, col));
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        v[j] = to_tf32(__uint_as_float(v[j]));
                        st_shared_u32(gt + kmaj_off(kTT, hf * kWT + c16 + j, col), v[j]);
                    }
                    tmem_st16(tm + Ly::TGT + uint32_t(b * kTT + hf * kWT + c16) + lane_off, v);
                }
                tmem_wait_st();
                fence_proxy_async();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ready[b]);
            }
            if (t > 0 && hf == 0) {
                // gh partial of the previous tile: one token row per thread
                const int u = t - 1, b = u & 1, s = (t0 + u) * kTT + col;
                if (!mbar_wait(&ghfull[b], (u >> 1) & 1, p.status, 85u)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                uint32_t v[16];
                tmem_ld16(tm + Ly::TGH + uint32_t(b * kRk) + lane_off, v);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ghfree[b]);
                if (s < p.S) {
                    float4 *dst = reinterpret_cast<float4 *>(q.part_gh + (int64_t(ot) * p.S + s) * kRk);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        dst[k] = make_float4(__uint_as_float(v[4 * k]), __uint_as_float(v[4 * k + 1]),
                                             __uint_as_float(v[4 * k + 2]), __uint_as_float(v[4 * k + 3]));
                }
            }
        }
        if (ok && hf == 0 && mbar_wait(&dfull, 0, p.status, 86u)) {
            // dB partial of the chunk: one column (row of B) per thread
            tc_fence_after();
            uint32_t v[16];
            tmem_ld16(tm + Ly::TDB + lane_off, v);
            tmem_wait_ld();
            if (o0 + col < q.O) {
                float4 *dst = reinterpret_cast<float4 *>(q.part_b + (int64_t(blockIdx.y) * q.O + o0 + col) * kRk);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    dst[k] = make_float4(__uint_as_float(v[4 * k]), __uint_as_float(v[4 * k + 1]),
                                         __uint_as_float(v[4 * k + 2]), __uint_as_float(v[4 * k + 3]));
            }
        }
        if (!ok) s_abort = 1;
    }
    tc_fence_before();
    __syncthreads();
    if (s_abort && threadIdx.x == 0)        // the last kSlots copies may still be in flight
        for (int t = max(0, s_issued - kSlots); t < s_issued; ++t)
            mbar_wait(&full[t % kSlots], (t / kSlots) & 1, nullptr, 0u);
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tm, Ly::COLS);
    }
}

// ------------------------------------------------------------------ x pass

struct XLayout {
    static constexpr int GT_BYTES = 4 * 32 * 128;             // [32 = 2 x 16 ranks][128 tokens]: four atoms
    static constexpr int GT0 = kSlots * kTileBytes, TOTAL = GT0 + 2 * GT_BYTES;
    // tensor memory: two x^T buffers [128 columns][128 tokens], the dA^T accumulator [128][32]
    static constexpr uint32_t TXT = 0, TDA = 2 * kTT, COLS = 512;
};

__global__ void __launch_bounds__(kThreads, 1) lora_tc_xpass_kernel(const __grid_constant__ LoraTcParams p) {
    using Ly = XLayout;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    // full / xfree: x slot landed / read by the writers; ready: x_t^T and gh_t^T written;
    // tfree: the MMA of the tile done (gh^T slot and x^T buffer free)
    __shared__ uint64_t full[kSlots], xfree[kSlots], ready[2], tfree[2], dfull;
    __shared__ uint32_t tmem_base;
    __shared__ int s_abort, s_issued;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c0 = int(blockIdx.x) * kCT;
    const int t0 = int(blockIdx.y) * p.tpc, nt = min(p.tpc, p.n_tt - t0);

    if (threadIdx.x == 0) {
        s_abort = 0;
        s_issued = 0;
        for (int b = 0; b < kSlots; ++b) {
            mbar_init(&full[b], 1);
            mbar_init(&xfree[b], kWriters);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ready[b], kWriters);
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
        if (lane == 0) {
            for (int t = 0; t < nt; ++t) {
                const int b = t % kSlots;
                if (t >= kSlots && !mbar_wait(&xfree[b], (t / kSlots - 1) & 1, p.status, 90u)) {
                    s_abort = 1;
                    break;
                }
                mbar_arrive_expect_tx(&full[b], kTileBytes);
                for (int k = 0; k < 4; ++k)
                    tma_load_3d(sm + b * kTileBytes + k * kBoxBytes, &p.x, c0 + 32 * k, (t0 + t) * kTT, 0, &full[b]);
                s_issued = t + 1;
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t id = idesc_tf32(128, kRk * p.nside);
            bool ok = true;
            for (int t = 0; t < nt; ++t) {
                const int b = t & 1;
                if (!mbar_wait(&ready[b], (t >> 1) & 1, p.status, 91u)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // dA^T += x_t^T [gh_0 | gh_1]_t: A = x_t^T (tensor memory), B = gh_t^T
#pragma unroll
                for (int k = 0; k < kTT / 8; ++k)
                    mma_tf32_ts(tm + Ly::TDA, tm + Ly::TXT + uint32_t(b * kTT + 8 * k),
                                sw128_desc(sm + Ly::GT0 + b * Ly::GT_BYTES + (k >> 2) * (32 * 128)) + 2 * (k & 3), id,
                                (t > 0 || k > 0) ? 1u : 0u);
                mma_commit(&tfree[b]);
            }
            if (!ok) s_abort = 1;
            mma_commit(&dfull);
            mbar_wait(&dfull, 0, nullptr, 0u);
        }
    } else {
        const int qq = warp & 3, hf = (warp - 2) >> 2, wi = warp - 2;
        const int col = 32 * qq + lane;
        const uint32_t lane_off = uint32_t(32 * qq) << 16;
        // gh_t^T values of this thread (rows 16 sd + r of adapter sd, rows past S zero),
        // loaded a tile ahead
        constexpr int NG = 2 * kRk * kTT / (kWriters * 32);
        float gv[NG];
        auto load_gh = [&](int t) {
            const int s0 = (t0 + t) * kTT;
#pragma unroll
            for (int k = 0; k < NG; ++k) {
                const int e = wi * 32 + lane + k * kWriters * 32, side = e / (kRk * kTT), f = e % (kRk * kTT);
                const int s = f >> 4, r = f & 15;
                gv[k] = side < p.nside && s0 + s < p.S ? __ldg(p.side[side].gh + int64_t(s0 + s) * kRk + r) : 0.f;
            }
        };
        load_gh(0);
        bool ok = true;
        for (int t = 0; t < nt; ++t) {
            const int b = t & 1;
            if (t >= 2 && !mbar_wait(&tfree[b], ((t - 2) >> 1) & 1, p.status, 92u)) {
                ok = false;
                break;
            }
#pragma unroll
            for (int k = 0; k < NG; ++k) {
                const int e = wi * 32 + lane + k * kWriters * 32, side = e / (kRk * kTT), f = e % (kRk * kTT);
                const int s = f >> 4, r = f & 15;
                st_shared_u32(sm + Ly::GT0 + b * Ly::GT_BYTES + kmaj_off(32, side * kRk + r, s), to_tf32(gv[k]));
            }
            if (t + 1 < nt) load_gh(t + 1);
            if (!mbar_wait(&full[t % kSlots], (t / kSlots) & 1, p.status, 93u)) {
                ok = false;
                break;
            }
            const uint8_t *xt = sm + (t % kSlots) * kTileBytes;
            static_assert(kWT == 32, "two 16-column tensor-memory stores per writer and tile");
            uint32_t v[2][16];
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
                for (int j = 0; j < 16; ++j) v[c][j] = ld_shared_u32(xt + kmaj_off(kTT, hf * kWT + 16 * c + j, col));
            __syncwarp();
            if (lane == 0) mbar_arrive(&xfree[t % kSlots]);      // the slot may be refilled
#pragma unroll
            for (int c = 0; c < 2; ++c) {
#pragma unroll
                for (int j = 0; j < 16; ++j) v[c][j] = to_tf32(__uint_as_float(v[c][j]));
                tmem_st16(tm + Ly::TXT + uint32_t(b * kTT + hf * kWT + 16 * c) + lane_off, v[c]);
            }
            tmem_wait_st();
            fence_proxy_async();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&ready[b]);
        }
        if (ok && hf == 0 && mbar_wait(&dfull, 0, p.status, 94u)) {
            // dA partial of the chunk: column c0 + col of every rank of every adapter
            tc_fence_after();
            for (int side = 0; side < p.nside; ++side) {
                uint32_t v[16];
                tmem_ld16(tm + Ly::TDA + uint32_t(side * kRk) + lane_off, v);
                tmem_wait_ld();
                if (c0 + col < p.C) {
                    float *dst = p.side[side].part_a + int64_t(blockIdx.y) * kRk * p.C + c0 + col;
#pragma unroll
                    for (int r = 0; r < kRk; ++r) dst[int64_t(r) * p.C] = __uint_as_float(v[r]);
                }
            }
        }
        if (!ok) s_abort = 1;
    }
    tc_fence_before();
    __syncthreads();
    if (s_abort && threadIdx.x == 0)
        for (int t = max(0, s_issued - kSlots); t < s_issued; ++t)
            mbar_wait(&full[t % kSlots], (t / kSlots) & 1, nullptr, 0u);
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tm, Ly::COLS);
    }
}

// fp32 [rows, cols] row-major as a 3-D tensor map {cols, rows, 1}, box {32, 128, 1},
// 128-byte swizzle, zero fill past the edges.
int map_rows(CUtensorMap *m, const float *base, int64_t rows, int64_t cols) {
    EncodeTiled enc = encode_fn();
    TLB_REQUIRE(enc != nullptr, TLB_ECUDA, "lora (tcgen05): cuTensorMapEncodeTiled unavailable");
    const cuuint64_t d[3] = {cuuint64_t(cols), cuuint64_t(rows), 1};
    const cuuint64_t st[2] = {cuuint64_t(cols) * 4, cuuint64_t(cols) * rows * 4};
    const cuuint32_t bx[3] = {32, kTT, 1};
    const cuuint32_t es[3] = {1, 1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float *>(base), d, st, bx, es,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    TLB_REQUIRE(r == CUDA_SUCCESS, TLB_ECUDA, "lora (tcgen05): tensor map encoding failed (%d)", int(r));
    return TLB_OK;
}

constexpr size_t kGSmem = size_t(GLayout::TOTAL) + 1024, kXSmem = size_t(XLayout::TOTAL) + 1024;

}  // namespace

bool lora_tc_supported(int64_t S, int in_dim, int rank, const float *x, const LoraTcJob *jobs, int njobs) {
    if (rank != kRk || S < 1 || S > (int64_t(1) << 30) || in_dim % 4 != 0 || !aligned16(x) || njobs < 1 || njobs > 2)
        return false;
    for (int j = 0; j < njobs; ++j)
        if (jobs[j].out_dim % 4 != 0 || !aligned16(jobs[j].G) || !aligned16(jobs[j].part_gh) ||
            !aligned16(jobs[j].part_b))
            return false;
    return true;
}

int lora_tc_chunks(int64_t S, int n_ct, int &tiles_per_chunk) {
    const int64_t n_tt = ceil_div(S, int64_t(kTT));
    int64_t nrc = std::max<int64_t>(1, std::min<int64_t>(n_tt, num_sms() / std::max(1, n_ct)));
    tiles_per_chunk = int(ceil_div(n_tt, nrc));
    return int(ceil_div(n_tt, int64_t(tiles_per_chunk)));
}

namespace {

int lora_tc_params(LoraTcParams &p, int64_t S, int in_dim, const float *x, const LoraTcJob *jobs, int njobs,
                   int tpc, uint32_t *status, bool gpass, int &n_blk) {
    memset(&p, 0, sizeof(p));
    p.nside = njobs;
    p.S = int(S);
    p.C = in_dim;
    p.tpc = tpc;
    p.n_tt = int(ceil_div(S, int64_t(kTT)));
    p.status = status;
    n_blk = 0;
    for (int j = 0; j < njobs; ++j) {
        LoraTcSide &q = p.side[j];
        if (gpass) TLB_TRY(map_rows(&q.g, jobs[j].G, S, jobs[j].out_dim));
        q.h = jobs[j].h;
        q.b = jobs[j].b;
        q.gh = jobs[j].gh;
        q.part_gh = jobs[j].part_gh;
        q.part_b = jobs[j].part_b;
        q.part_a = jobs[j].part_a;
        q.O = jobs[j].out_dim;
        q.blk0 = n_blk;
        n_blk += int(ceil_div(int64_t(q.O), int64_t(kCT)));
    }
    if (!gpass) TLB_TRY(map_rows(&p.x, x, S, in_dim));
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [] {
        err = cudaFuncSetAttribute(lora_tc_gpass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kGSmem));
        if (err == cudaSuccess)
            err = cudaFuncSetAttribute(lora_tc_xpass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kXSmem));
    });
    TLB_CUDA(err);
    return TLB_OK;
}

}  // namespace

int lora_tc_gpass_launch(int64_t S, const LoraTcJob *jobs, int njobs, int tiles_per_chunk, uint32_t *status,
                         cudaStream_t st) {
    LoraTcParams p;
    int n_ot = 0;
    TLB_TRY(lora_tc_params(p, S, 0, nullptr, jobs, njobs, tiles_per_chunk, status, true, n_ot));
    const int nrc = int(ceil_div(int64_t(p.n_tt), int64_t(tiles_per_chunk)));
    lora_tc_gpass_kernel<<<dim3(unsigned(n_ot), unsigned(nrc)), kThreads, kGSmem, st>>>(p);
    return check_launch("lora_tc_gpass");
}

int lora_tc_xpass_launch(int64_t S, int in_dim, const float *x, const LoraTcJob *jobs, int njobs,
                         int tiles_per_chunk, uint32_t *status, cudaStream_t st) {
    LoraTcParams p;
    int n_ot = 0;
    TLB_TRY(lora_tc_params(p, S, in_dim, x, jobs, njobs, tiles_per_chunk, status, false, n_ot));
    const int nrc = int(ceil_div(int64_t(p.n_tt), int64_t(tiles_per_chunk)));
    lora_tc_xpass_kernel<<<dim3(unsigned(ceil_div(int64_t(in_dim), int64_t(kCT))), unsigned(nrc)), kThreads, kXSmem,
                           st>>>(p);
    return check_launch("lora_tc_xpass");
}

}  // namespace tlb
