// Tensor-core (tcgen05) GEMM for the transposed-weight products of the sequence path:
//   C[M, N] (+)= alpha * A[M, K] . B[N, K]^T
// with A the bf16 output gradient (rows = tokens), B a bf16 weight stored [in, out]
// (= [N, K], K-major), fp32 accumulation in tensor memory ([FFN] W_down^T, W_gate^T,
// W_up^T products; [ATT] O-projection backward; [RS] gemm_backward_a).
//
// Persistent: one CTA per SM walks its share of the work, tile segment by tile segment
// (cta_group::1):
//   warp 0      TMA producer: 128x64 (A) and BNx64 (B) bf16 tiles, 128-byte swizzle,
//               into a STAGES-deep shared-memory ring guarded by mbarriers; the ring
//               runs on across units
//   warp 1      allocates 2 x BN TMEM columns (two accumulators); one thread issues
//               tcgen05.mma.kind::f16 (M = 128, N = BN, K = 16) four times per 64-wide
//               k block into the accumulator of the segment's parity; tcgen05.commit
//               frees each stage and, after a segment's last block, hands the
//               accumulator over
//   warps 2..9  epilogue: tcgen05.ld 32x32b.x32 (two warps per 32 TMEM lanes = rows, each
//               half of the columns); each 32 x 32 block turns in shared memory so that
//               lanes run along columns; scale, optional accumulate into C, coalesced fp32
//               stores (and an optional bf16 copy, or a tf32 transposed copy for the
//               attention), then release the accumulator, so one segment's epilogue
//               overlaps the next one's MMAs
// Paired form (BN = 256, clusters of two CTAs on one TPC, cta_group::2): the pair owns a
// 256 x 256 super-tile; each CTA loads its own 128 rows of A and its half (128 rows) of B
// into its own ring, the even CTA issues tcgen05.mma.cta_group::2 (M = 256, N = 256), which
// takes A and B halves from both CTAs' shared memory and leaves rows 0..127 in the even
// CTA's tensor memory and rows 128..255 in the odd one's.  Per CTA and k block that is
// 32 KB staged instead of 48 KB for the same 128 x 256 x 64 of work, which relieves the
// shared-memory traffic (TMA writes + MMA reads) that bounds the single-CTA form.  Both
// CTAs' copies count on the even CTA's full barrier; its commits free the stage and hand
// over the accumulators in both CTAs (multicast); both CTAs' epilogue warps release an
// accumulator on the even CTA's barrier.
// K may come from two segments (A0.B0^T + A1.B1^T, e.g. [dG | dU] . [W_gate | W_up]^T).
// Work is balanced stream-K style: the (tile, k block) iterations are split evenly over
// the CTAs; a tile done by one CTA is written by it, a tile shared by several is summed
// from their partial tiles by tc_fixup in CTA order.  Every mbarrier wait is bounded
// (status + wind-down).
#include <cuda.h>

#include <algorithm>
#include <cstring>
#include <vector>
#include <tuple>
#include <map>
#include <mutex>

#include "async.cuh"
#include "common.cuh"
#include "kernels.cuh"
#include "tc.cuh"

namespace tlb {

namespace {

constexpr int kBM = 128, kBK = 64;       // tile rows, k block (64 bf16 = 128 bytes)
constexpr int kStages = 4;               // ring depth, single-CTA form (48 KB stages)
constexpr int kStagesPair = 5;           // paired form (32 KB stages; a sixth slows the W_down^T epilogue)
template <bool PAIR> constexpr int stages_of() { return PAIR ? kStagesPair : kStages; }
// k-block time of the paired form relative to the single-CTA 128 x 256 form (planner)
constexpr double kPairRate = 0.75;
constexpr int kThreadsTC = 320;          // 10 warps: producer, MMA, 8 epilogue warps
constexpr int kEpiWarpsTC = 8;           // two per TMEM lane quarter, each half of the columns
constexpr int kMaxSeg = 3;               // K segments of one product

struct TcParams {
    CUtensorMap a[kMaxSeg];              // bf16 [M, K_seg], box 64 x 128
    CUtensorMap b[kMaxSeg];              // bf16 [N, K_seg], box 64 x BN
    int kb[kMaxSeg];                     // k blocks of each segment
    int nseg;
    int M, N;
    float alpha;
    float *out;                          // [M, N] fp32
    uint2 *obf;                          // mode 0: [M, N] bf16 copy of out (four per uint2), or null
    float *out_t;                        // mode 0, not accumulating: tf32 copy, transposed (ld_t), or null
    int64_t ld_t;
    int accumulate;
    float *partial;                      // [ctas][2][kBM * BN] fp32 partial tiles
    // epilogue: mode 0 writes out (+)= alpha acc; mode 1 treats alpha acc as dh and writes
    // the gated-activation backward dG, dU in bf16 ([FFN] ReLU^2 x Mul / [RS] SwiGLU)
    int mode, act;
    const float *gate, *up;              // [M, N] fp32 (mode 1); silu(gate) is recomputed
    uint2 *dg, *du;                      // [M, N] bf16, four per uint2 (mode 1)
    // schedule over the flattened (tile, k block) iterations, tiles numbered m fastest:
    // CTA c first runs the whole tiles [c dp, (c + 1) dp), then the stream-K share
    // [sk_base + sk_work c / ctas, sk_base + sk_work (c + 1) / ctas) of the rest.  In the
    // paired form a tile is a 256-row super-tile and c a CTA pair (ctas pairs).
    int dp;                              // whole tiles per CTA
    int ctas;
    int64_t sk_base, sk_work;
    uint32_t *status;
};

constexpr int kMaxFix = 256;
// Tiles shared by several CTAs (stream-K part): tile t is the sum of the partial tiles of
// CTAs c0..c1, CTA c0's in slot s0 (1 when c0 began in an earlier tile), the others in slot 0
// (paired form: super-tile t, pairs c0..c1, half h of it from CTA 2 c + h).
struct TcFixup {
    int n;
    int4 e[kMaxFix];                     // {tile, c0, c1, s0}
};

__host__ __device__ __forceinline__ int64_t sk_start(int64_t work, int ctas, int c) {
    return work * c / ctas;
}

// Epilogue of four columns col..col+3 (< N, col % 4 == 0) of one row; acc before alpha.
__device__ __forceinline__ void emit4(const TcParams &p, int row, int col, float4 acc) {
    const int64_t e = int64_t(row) * p.N + col;
    const float4 d = make_float4(p.alpha * acc.x, p.alpha * acc.y, p.alpha * acc.z, p.alpha * acc.w);
    if (p.mode == 0) {
        float4 y = d;
        if (p.accumulate) {
            const float4 c = *reinterpret_cast<const float4 *>(p.out + e);
            y.x += c.x; y.y += c.y; y.z += c.z; y.w += c.w;
        }
        if (p.out != nullptr) *reinterpret_cast<float4 *>(p.out + e) = y;
        if (p.obf != nullptr) p.obf[e / 4] = pack_bf16x4(y.x, y.y, y.z, y.w);
        if (p.out_t != nullptr) {
            float *t = p.out_t + int64_t(col) * p.ld_t + row;
            t[0] = __uint_as_float(to_tf32(y.x));
            t[p.ld_t] = __uint_as_float(to_tf32(y.y));
            t[2 * p.ld_t] = __uint_as_float(to_tf32(y.z));
            t[3 * p.ld_t] = __uint_as_float(to_tf32(y.w));
        }
        return;
    }
    const float4 g = ld_stream(reinterpret_cast<const float4 *>(p.gate + e));
    const float4 u = ld_stream(reinterpret_cast<const float4 *>(p.up + e));
    float4 og, ou;
    if (p.act == TLB_ACT_RELU2_MUL) {
        act_bwd_elem_bf16<TLB_ACT_RELU2_MUL>(g.x, u.x, d.x, og.x, ou.x);
        act_bwd_elem_bf16<TLB_ACT_RELU2_MUL>(g.y, u.y, d.y, og.y, ou.y);
        act_bwd_elem_bf16<TLB_ACT_RELU2_MUL>(g.z, u.z, d.z, og.z, ou.z);
        act_bwd_elem_bf16<TLB_ACT_RELU2_MUL>(g.w, u.w, d.w, og.w, ou.w);
    } else {
        act_bwd_elem_bf16<TLB_ACT_SILU_MUL>(g.x, u.x, d.x, og.x, ou.x);
        act_bwd_elem_bf16<TLB_ACT_SILU_MUL>(g.y, u.y, d.y, og.y, ou.y);
        act_bwd_elem_bf16<TLB_ACT_SILU_MUL>(g.z, u.z, d.z, og.z, ou.z);
        act_bwd_elem_bf16<TLB_ACT_SILU_MUL>(g.w, u.w, d.w, og.w, ou.w);
    }
    p.dg[e / 4] = pack_bf16x4(og.x, og.y, og.z, og.w);
    p.du[e / 4] = pack_bf16x4(ou.x, ou.y, ou.z, ou.w);
}

// Activation epilogue of one 32 x 32 block (rows rbase.., columns col0..) held in shared
// memory [32][33]: lanes are 8 column quads x 4 rows; every load of the block is issued
// before the first store, so the memory latency is paid once per block.  The SwiGLU form
// recomputes silu(gate) from the gate it loads anyway: a cached copy would add a third to
// the loads this epilogue is bound by.
template <int ACT>
__device__ __forceinline__ void act_block_t(const TcParams &p, int rbase, int col0, const float *blk, int lane) {
    const int c4 = (lane & 7) * 4, rl = lane >> 3;
    float4 g[8], u[8];
    bool ok[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int r = 4 * k + rl;
        ok[k] = rbase + r < p.M && col0 + c4 < p.N;
        const int64_t e = ok[k] ? int64_t(rbase + r) * p.N + col0 + c4 : 0;
        g[k] = ld_stream(reinterpret_cast<const float4 *>(p.gate + e));
        u[k] = ld_stream(reinterpret_cast<const float4 *>(p.up + e));
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int r = 4 * k + rl;
        if (!ok[k]) continue;
        const float *a = blk + r * 33 + c4;
        float4 og, ou;
        act_bwd_elem_bf16<ACT>(g[k].x, u[k].x, p.alpha * a[0], og.x, ou.x);
        act_bwd_elem_bf16<ACT>(g[k].y, u[k].y, p.alpha * a[1], og.y, ou.y);
        act_bwd_elem_bf16<ACT>(g[k].z, u[k].z, p.alpha * a[2], og.z, ou.z);
        act_bwd_elem_bf16<ACT>(g[k].w, u[k].w, p.alpha * a[3], og.w, ou.w);
        const int64_t e = int64_t(rbase + r) * p.N + col0 + c4;
        p.dg[e / 4] = pack_bf16x4(og.x, og.y, og.z, og.w);
        p.du[e / 4] = pack_bf16x4(ou.x, ou.y, ou.z, ou.w);
    }
}

__device__ __forceinline__ void act_block(const TcParams &p, int rbase, int col0, const float *blk, int lane) {
    if (p.act == TLB_ACT_RELU2_MUL) act_block_t<TLB_ACT_RELU2_MUL>(p, rbase, col0, blk, lane);
    else act_block_t<TLB_ACT_SILU_MUL>(p, rbase, col0, blk, lane);
}

// Plain epilogue of a warp's 32 x 32 block staged in shared memory (blk[r * 33 + c], before
// alpha): out (+)= alpha acc and the optional bf16 copy, with lanes along the columns
// (8 column quads x 4 rows per access), so every load and store is coalesced.
__device__ __forceinline__ void out_block(const TcParams &p, int rbase, int col0, const float *blk, int lane) {
    const int c4 = (lane & 7) * 4, rl = lane >> 3;
    const bool col_ok = col0 + c4 < p.N;                  // N % 4 == 0: the quad is whole
#pragma unroll 1
    for (int k0 = 0; k0 < 8 && p.out != nullptr; k0 += 4) {   // four loads of C in flight
        float4 c[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int r = 4 * (k0 + k) + rl;
            c[k] = (p.accumulate && col_ok && rbase + r < p.M)
                       ? *reinterpret_cast<const float4 *>(p.out + int64_t(rbase + r) * p.N + col0 + c4)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int r = 4 * (k0 + k) + rl;
            if (!col_ok || rbase + r >= p.M) continue;
            const float *a = blk + r * 33 + c4;
            float4 y = make_float4(p.alpha * a[0], p.alpha * a[1], p.alpha * a[2], p.alpha * a[3]);
            if (p.accumulate) {
                y.x += c[k].x; y.y += c[k].y; y.z += c[k].z; y.w += c[k].w;
            }
            const int64_t e = int64_t(rbase + r) * p.N + col0 + c4;
            *reinterpret_cast<float4 *>(p.out + e) = y;
            if (p.obf != nullptr) p.obf[e / 4] = pack_bf16x4(y.x, y.y, y.z, y.w);
        }
    }
    if (p.out_t != nullptr) {
        // the tf32 transposed copy (never accumulating: the value is alpha acc, as stored
        // above): four columns per step, eight lanes per column, four rows per lane, so each
        // column's 32 rows go out as 128 contiguous bytes.  Rows past M up to ld_t (a multiple
        // of 4) are padding of the copy.
        const int r4 = (lane & 7) * 4;
        if (rbase + r4 < p.M) {
#pragma unroll
            for (int cg = 0; cg < 8; ++cg) {
                const int c = cg * 4 + (lane >> 3);
                if (col0 + c >= p.N) continue;
                const float *a = blk + r4 * 33 + c;
                *reinterpret_cast<float4 *>(p.out_t + int64_t(col0 + c) * p.ld_t + rbase + r4) =
                    make_float4(__uint_as_float(to_tf32(p.alpha * a[0])), __uint_as_float(to_tf32(p.alpha * a[33])),
                                __uint_as_float(to_tf32(p.alpha * a[66])), __uint_as_float(to_tf32(p.alpha * a[99])));
            }
        }
    }
}

// A warp's 32 x 32 block of a partial tile (rows of BN floats), from shared memory, coalesced.
__device__ __forceinline__ void partial_block(float *o, int ld, const float *blk, int lane) {
    const int c4 = (lane & 7) * 4, rl = lane >> 3;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int r = 4 * k + rl;
        const float *a = blk + r * 33 + c4;
        *reinterpret_cast<float4 *>(o + int64_t(r) * ld + c4) = make_float4(a[0], a[1], a[2], a[3]);
    }
}

template <int M, int BN>
__device__ __forceinline__ uint32_t idesc_bf16() {
    return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

template <int BN, bool PAIR>
__global__ void __launch_bounds__(kThreadsTC, 1) tc_gemm_kernel(const __grid_constant__ TcParams p) {
    static_assert(!PAIR || BN == 256, "the paired form runs 256 x 256 super-tiles");
    constexpr int TM = PAIR ? 2 * kBM : kBM;                 // rows of a scheduled tile
    constexpr int BH = PAIR ? BN / 2 : BN;                   // rows of B this CTA stages
    constexpr int A_BYTES = kBM * kBK * 2, B_BYTES = BH * kBK * 2, STAGE = A_BYTES + B_BYTES;
    constexpr int kStages = stages_of<PAIR>();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t full[kStages], empty[kStages], accfull[2], accempty[2], done;
    __shared__ uint32_t tmem_base;
    __shared__ int s_abort, s_issued, s_consumed;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = PAIR ? int(cluster_rank()) : 0;        // this CTA's half of a super-tile
    const int cl = PAIR ? int(blockIdx.x >> 1) : int(blockIdx.x);
    const bool leader = rank == 0;                           // issues the MMAs

    // this CTA's (pair's) iterations: the whole tiles [c dp, (c + 1) dp), then its stream-K
    // range; cut at tile boundaries into segments
    const int tiles_m = (p.M + TM - 1) / TM;
    const int KB = p.kb[0] + (p.nseg > 1 ? p.kb[1] : 0) + (p.nseg > 2 ? p.kb[2] : 0);
    const int64_t a0 = int64_t(cl) * p.dp * KB, a1 = a0 + int64_t(p.dp) * KB;
    const int64_t b0 = p.sk_base + sk_start(p.sk_work, p.ctas, cl);
    const int64_t b1 = p.sk_base + sk_start(p.sk_work, p.ctas, cl + 1);
    const int64_t g0 = a0, g1 = a1 + (b1 - b0);               // local iteration count g1 - g0
    auto to_global = [&](int64_t g) { return g < a1 ? g : b0 + (g - a1); };
    // segment starting at local iteration g: tile, rows, columns, k blocks [kb0, kb1)
    auto segment = [&](int64_t g, int &m0, int &n0, int &kb0, int &kb1) {
        const int64_t gg = to_global(g), end = g < a1 ? a1 : b1;
        const int64_t t = gg / KB;
        kb0 = int(gg - t * KB);
        kb1 = int(std::min<int64_t>(KB, end - t * KB));
        m0 = int(t % tiles_m) * TM + rank * kBM;             // this CTA's rows
        n0 = int(t / tiles_m) * BN;
    };

    if (threadIdx.x == 0) {
        s_abort = 0;
        s_issued = s_consumed = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accfull[b], 1);
            mbar_init(&accempty[b], (PAIR ? 2 : 1) * kEpiWarpsTC);   // paired: both CTAs' warps
        }
        mbar_init(&done, 1);
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            tmem_alloc_pair(&tmem_base, 2 * BN);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(&tmem_base, 2 * BN);
            tmem_relinquish();
        }
    }
    fence_mbar_init();
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();              // the peer's barriers exist before any remote arrive
    tc_fence_after();
    const uint32_t tmem = tmem_base;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (ring continues across units)
        if (lane == 0) {
            int g = 0;
            bool ok = true;
            for (int64_t gs = g0; ok && gs < g1;) {
                int m0, n0, kb0, kb1;
                segment(gs, m0, n0, kb0, kb1);
                gs += kb1 - kb0;
                for (int kb = kb0; kb < kb1; ++kb, ++g) {
                    const int s = g % kStages;
                    if (g >= kStages && !mbar_wait(&empty[s], ((g / kStages) - 1) & 1, p.status, 10u)) {
                        ok = false;
                        break;
                    }
                    const int seg = kb < p.kb[0] ? 0 : (kb < p.kb[0] + p.kb[1] ? 1 : 2);
                    const int kx = (kb - (seg > 0 ? p.kb[0] : 0) - (seg > 1 ? p.kb[1] : 0)) * kBK;
                    uint8_t *sa = smem + s * STAGE;
                    if constexpr (PAIR) {
                        // both CTAs' copies count on the even CTA's full barrier
                        if (leader) mbar_arrive_expect_tx(&full[s], 2 * STAGE);
                        const uint32_t fb = cluster_addr(&full[s], 0);
                        tma_load_2d_pair(sa, &p.a[seg], kx, m0, fb);
                        tma_load_2d_pair(sa + A_BYTES, &p.b[seg], kx, n0 + rank * BH, fb);
                    } else {
                        mbar_arrive_expect_tx(&full[s], STAGE);
                        tma_load_2d(sa, &p.a[seg], kx, m0, &full[s]);
                        tma_load_2d(sa + A_BYTES, &p.b[seg], kx, n0, &full[s]);
                    }
                    s_issued = g + 1;
                }
            }
            if (!ok) s_abort = 1;
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer, accumulators alternate
        if (lane == 0 && leader) {
            const uint32_t idesc = idesc_bf16<TM, BN>();
            int g = 0, i = 0;
            bool ok = true;
            for (int64_t gs = g0; ok && gs < g1; ++i) {
                int m0, n0, kb0, kb1;
                segment(gs, m0, n0, kb0, kb1);
                gs += kb1 - kb0;
                const int b = i & 1;
                const uint32_t acc = tmem + uint32_t(b * BN);
                if (i >= 2 && !mbar_wait(&accempty[b], ((i >> 1) - 1) & 1, p.status, 13u)) { ok = false; break; }
                tc_fence_after();
                for (int kb = kb0; kb < kb1; ++kb, ++g) {
                    const int s = g % kStages;
                    if (!mbar_wait(&full[s], (g / kStages) & 1, p.status, 11u)) { ok = false; break; }
                    tc_fence_after();
                    const uint8_t *sa = smem + s * STAGE;
                    const uint64_t ad = sw128_desc(sa), bd = sw128_desc(sa + A_BYTES);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k) {  // 16 bf16 = 32 bytes = 2 descriptor units
                        if constexpr (PAIR)
                            mma_bf16_pair(acc, ad + 2 * k, bd + 2 * k, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
                        else
                            mma_bf16(acc, ad + 2 * k, bd + 2 * k, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
                    }
                    if constexpr (PAIR) mma_commit_pair(&empty[s], 3);   // frees the stage in both CTAs
                    else mma_commit(&empty[s]);
                    s_consumed = g + 1;
                }
                if (ok) {                             // this unit's MMAs done -> epilogue
                    if constexpr (PAIR) mma_commit_pair(&accfull[b], 3);
                    else mma_commit(&accfull[b]);
                }
            }
            if (!ok) s_abort = 1;
            // fires once every MMA issued above is complete
            if constexpr (PAIR) mma_commit_pair(&done, 1);
            else mma_commit(&done);
            mbar_wait(&done, 0, nullptr, 0u);
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2..9)
        const int q = warp & 3;                   // TMEM lane quarter this warp may read
        float *ep = reinterpret_cast<float *>(smem + kStages * STAGE);   // 8 x [32][33] transpose blocks
        int i = 0;
        for (int64_t gs = g0; gs < g1; ++i) {
            int m0, n0, kb0, kb1;
            segment(gs, m0, n0, kb0, kb1);
            const bool whole = kb0 == 0 && kb1 == KB;
            const int slot = to_global(gs) == b0 ? 0 : 1;   // first or last stream-K segment
            gs += kb1 - kb0;
            const int b = i & 1;
            if (!mbar_wait(&accfull[b], (i >> 1) & 1, p.status, 12u)) {
                s_abort = 1;
                break;
            }
            tc_fence_after();
            const int half = (warp - 2) >> 2;     // this warp's half of the tile's columns
            float *blk = ep + (warp - 2) * 32 * 33;
            for (int j = half * (BN / 64); j < (half + 1) * (BN / 64); ++j) {
                uint32_t v[32];
                tmem_ld32(tmem + uint32_t(b * BN) + (uint32_t(q * 32) << 16) + uint32_t(j * 32), v);
                tmem_wait_ld();
                const int col0 = n0 + j * 32;
                // the warp's 32 x 32 block (one row per lane) goes through shared memory so
                // that lanes run along columns and every global access is coalesced
#pragma unroll
                for (int t = 0; t < 32; ++t) blk[lane * 33 + t] = __uint_as_float(v[t]);
                __syncwarp();
                if (!whole)         // partial tile of this CTA, tile-local [kBM][BN]
                    partial_block(p.partial + ((int64_t(blockIdx.x) * 2 + slot) * kBM + q * 32) * BN + j * 32, BN,
                                  blk, lane);   // paired: blockIdx.x = 2 pair + half
                else if (p.mode == 1)
                    act_block(p, m0 + q * 32, col0, blk, lane);
                else
                    out_block(p, m0 + q * 32, col0, blk, lane);
                __syncwarp();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (PAIR) mbar_arrive_cluster(cluster_addr(&accempty[b], 0));
                else mbar_arrive(&accempty[b]);
            }
        }
    }
    // wind down: the MMA thread waited for its final commit, so no MMA is in flight;
    // after an abort, also wait (bounded) for the tile copies that were issued but never
    // consumed, so nothing lands in shared memory after exit
    tc_fence_before();
    __syncthreads();
    if (s_abort && threadIdx.x == 0 && leader) {
        for (int g = s_consumed; g < s_issued; ++g) mbar_wait(&full[g % kStages], (g / kStages) & 1, nullptr, 0u);
    }
    __syncthreads();
    // paired: neither CTA leaves or frees its tensor memory while the other's commits or
    // arrivals may still reach it.  (After an abort, which a wait that ran out has already
    // reported, the bounded wait above covers the even CTA's own copies; the odd CTA's count
    // on the even CTA's barrier and are not awaited separately.)
    if constexpr (PAIR) cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        if constexpr (PAIR) tmem_dealloc_pair(tmem, 2 * BN);
        else tmem_dealloc(tmem, 2 * BN);
    }
}

// Stream-K fixup: a tile shared by CTAs c0..c1 is the sum, in CTA order, of their partial
// tiles; out (+)= alpha * sum.  Block (entry, y) does rows [y kBM / gridDim.y, ...) of it.
template <int BN, bool PAIR>
__global__ void __launch_bounds__(256) tc_fixup_kernel(const __grid_constant__ TcParams p,
                                                       const __grid_constant__ TcFixup f) {
    constexpr int TM = PAIR ? 2 * kBM : kBM;
    const int4 en = f.e[blockIdx.x];
    const int tiles_m = (p.M + TM - 1) / TM;
    const int m0 = (en.x % tiles_m) * TM, n0 = (en.x / tiles_m) * BN;
    const int rows = TM / gridDim.y, r0 = blockIdx.y * rows;
    for (int e = threadIdx.x; e < rows * (BN / 4); e += blockDim.x) {
        const int r = r0 + e / (BN / 4), c4 = (e % (BN / 4)) * 4;
        const int h = r / kBM, lr = r % kBM;               // half of a super-tile, row in it
        auto part = [&](int c) {
            const int slot = c == en.y ? en.w : 0;
            const int64_t cta = PAIR ? 2 * int64_t(c) + h : c;
            return *reinterpret_cast<const float4 *>(p.partial + ((cta * 2 + slot) * kBM + lr) * BN + c4);
        };
        // CTA order, up to eight partial tiles' loads in flight at a time
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c = en.y; c <= en.z; c += 8) {
            const int n = min(8, en.z - c + 1);
            float4 v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (u < n) v[u] = part(c + u);
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (u < n) {
                    acc.x += v[u].x; acc.y += v[u].y; acc.z += v[u].z; acc.w += v[u].w;
                }
        }
        const int row = m0 + r, col = n0 + c4;
        if (row >= p.M || col >= p.N) continue;
        emit4(p, row, col, acc);
    }
}

// fp32 [rows, cols] -> bf16 (round to nearest even), 4 at a time
__global__ void to_bf16_kernel(const float4 *__restrict__ x, uint2 *__restrict__ y, int64_t n4) {
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n4; i += 4 * stride) {          // four loads in flight per thread
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = x[i + u * stride];
#pragma unroll
        for (int u = 0; u < 4; ++u) y[i + u * stride] = pack_bf16x4(v[u].x, v[u].y, v[u].z, v[u].w);
    }
    for (; i < n4; i += stride) {
        const float4 v = x[i];
        y[i] = pack_bf16x4(v.x, v.y, v.z, v.w);
    }
}

// ---------------------------------------------------------------- host side

// bf16 [rows, cols] row-major, box cols 64 x rows box_rows, 128-byte swizzle, zero fill.
int make_map(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int box_rows) {
    EncodeTiled enc = encode_fn();
    TLB_REQUIRE(enc != nullptr, TLB_ECUDA, "tcgen05 GEMM: cuTensorMapEncodeTiled unavailable");
    const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(cols) * 2};
    const cuuint32_t box[2] = {cuuint32_t(kBK), cuuint32_t(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    TLB_REQUIRE(r == CUDA_SUCCESS, TLB_ECUDA, "tcgen05 GEMM: tensor map encoding failed (%d)", int(r));
    return TLB_OK;
}

template <int BN, bool PAIR>
int launch_tc(const TcParams &p, cudaStream_t st) {
    constexpr int smem = stages_of<PAIR>() * (kBM * kBK * 2 + (PAIR ? BN / 2 : BN) * kBK * 2) +
                         kEpiWarpsTC * 32 * 33 * 4 + 1024;
    static_assert(smem <= 227 * 1024 - 256, "shared memory of one CTA");
    auto k = tc_gemm_kernel<BN, PAIR>;
    TLB_CUDA(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    if constexpr (PAIR) {                             // clusters of two CTAs, one pair per TPC
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(unsigned(2 * p.ctas));
        cfg.blockDim = dim3(kThreadsTC);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        TLB_CUDA(cudaLaunchKernelEx(&cfg, k, p));
    } else {
        k<<<p.ctas, kThreadsTC, smem, st>>>(p);
    }
    TLB_TRY(check_launch("tcgen05 gemm"));
    // tiles of the stream-K part that more than one CTA touched
    const int64_t KB = p.kb[0] + (p.nseg > 1 ? p.kb[1] : 0) + (p.nseg > 2 ? p.kb[2] : 0);
    TcFixup f;
    f.n = 0;
    int c = 0;
    for (int64_t t = p.sk_base / KB; p.sk_work > 0 && t < (p.sk_base + p.sk_work) / KB; ++t) {
        const int64_t ta = t * KB - p.sk_base, tb = ta + KB;     // within the stream-K range
        while (c + 1 < p.ctas && sk_start(p.sk_work, p.ctas, c + 1) <= ta) ++c;
        int c1 = c;
        while (c1 + 1 < p.ctas && sk_start(p.sk_work, p.ctas, c1 + 1) < tb) ++c1;
        if (c1 > c) {
            TLB_REQUIRE(f.n < kMaxFix, TLB_EUNSUPPORTED, "tcgen05 GEMM: too many shared tiles");
            f.e[f.n++] = make_int4(int(t), c, c1, sk_start(p.sk_work, p.ctas, c) < ta ? 1 : 0);
        }
    }
    if (f.n == 0) return TLB_OK;
    tc_fixup_kernel<BN, PAIR><<<dim3(unsigned(f.n), PAIR ? 64 : 32), 256, 0, st>>>(p, f);
    return check_launch("tcgen05 gemm fixup");
}

}  // namespace

TcPlan tc_plan(int64_t M, int64_t N, int64_t K) {
    // 256 x 256 super-tiles on persistent CTA pairs, or 128 x 256 / 128 x 128 tiles on
    // persistent CTAs.  Candidates: `dp` whole tiles per CTA (pair), the remaining tiles
    // shared stream-K style by the `ctas` CTAs (pairs).
    // Cost: the busiest CTA's k blocks (one 128 x BN x 64 MMA block each, at the rate
    // these kernels reach: 128-wide tiles about 1.4 times slower per flop), plus 8 us
    // per stream-K segment of the busiest CTA (each ends in a TMEM drain into a partial
    // tile), the partial-tile traffic and a fixup launch when tiles are shared.  The
    // constants are fitted to measured plans of the S = 512 and S = 2048 layer products:
    // an even split (every CTA inside one tile) beats a finer uneven one.  Plans are cached.
    static std::mutex mu;
    static std::map<std::tuple<int64_t, int64_t, int64_t, int>, TcPlan> cache;
    const int nsm = num_sms();
    const auto key = std::make_tuple(M, N, K, nsm);
    {
        std::lock_guard<std::mutex> lk(mu);
        auto it = cache.find(key);
        if (it != cache.end()) return it->second;
    }
    TcPlan best{N > 128 ? 256 : 128, 1, 0, 0, 0};
    double best_cost = 1e300;
    for (int form = 0; form < 3; ++form) {
        // 0: paired 256 x 256 super-tiles, 1: single 128 x 256, 2: single 128 x 128
        const bool pair = form == 0;
        const int bn = form == 2 ? 128 : 256;
        if (bn == 256 && N <= 128) continue;
        if (pair && (M <= kBM || nsm < 2)) continue;
        const int64_t tm = pair ? 2 * kBM : kBM;
        const int units = pair ? nsm / 2 : nsm;
        const int64_t tiles = ceil_div(N, bn) * ceil_div(M, tm), KB = ceil_div(K, kBK);
        // s per k block of a CTA's 128 x bn share; 128-wide tiles stage A twice as often per
        // flop, the paired form stages half of B
        const double t_kb = 2.0 * kBM * bn * kBK / (1.3e15 / nsm) * (bn == 128 ? 1.4 : pair ? kPairRate : 1.0);
        const double tile_io = (pair ? 2.0 : 1.0) * 2.0 * kBM * bn * 4 / 6.0e12;   // s per partial tile written + read
        auto consider = [&](int64_t ctas, int64_t dp) {
            if (ctas < 1 || ctas > units || dp < 0 || dp * ctas > tiles) return;
            const int64_t skw = (tiles - dp * ctas) * KB;
            int64_t shared = 0;
            for (int64_t c = 1; c < ctas && skw > 0; ++c)
                if (sk_start(skw, int(ctas), int(c)) % KB != 0) ++shared;
            int64_t segs = 0;   // stream-K segments of the busiest CTA
            for (int64_t c = 0; c < ctas && skw > 0; ++c) {
                const int64_t a = sk_start(skw, int(ctas), int(c)), b = sk_start(skw, int(ctas), int(c + 1));
                if (b > a) segs = std::max<int64_t>(segs, (b - 1) / KB - a / KB + 1);
            }
            const double cost = double(dp * KB + ceil_div(skw, ctas)) * t_kb + double(segs) * 8e-6 +
                                (shared > 0 ? 2.0 * shared * tile_io + 3e-6 : 0.0);
            if (cost < best_cost) {
                best_cost = cost;
                best = TcPlan{bn, int(ctas), int(dp), int(shared), pair ? 1 : 0};
            }
        };
        std::vector<int64_t> cand = {units};
        for (int64_t s = 1; s <= 8; ++s) cand.push_back(std::min<int64_t>(tiles * s, units));
        for (int64_t d = 1; d <= 8; ++d) cand.push_back(std::max<int64_t>(1, std::min<int64_t>(units, ceil_div(tiles, d))));
        for (int64_t ctas : cand) {
            consider(ctas, tiles / ctas);
            consider(ctas, tiles / ctas - 1);
            consider(ctas, 0);
        }
    }
    std::lock_guard<std::mutex> lk(mu);
    cache[key] = best;
    return best;
}

size_t tc_partial_bytes(int64_t M, int64_t N, int64_t K) {
    // sized for two partial tiles per CTA whatever the split of K into segments
    const TcPlan pl = tc_plan(M, N, K);
    return size_t(pl.ctas) * (pl.pair ? 2 : 1) * 2 * kBM * pl.bn * 4;
}

int tc_convert_bf16(const float *x, void *y, int64_t n, cudaStream_t st) {
    if (n == 0) return TLB_OK;
    TLB_REQUIRE(n % 4 == 0 && aligned16(x) && aligned16(y), TLB_EUNSUPPORTED, "bf16 conversion: n %% 4 or alignment");
    to_bf16_kernel<<<stream_grid(n / 4, 256), 256, 0, st>>>(reinterpret_cast<const float4 *>(x),
                                                            reinterpret_cast<uint2 *>(y), n / 4);
    return check_launch("to_bf16");
}

bool tc_supported(int64_t M, int64_t N, int64_t K) {
    // TMA: row strides multiples of 16 bytes (K % 8 for bf16); the fp32 epilogue uses float4
    return M > 0 && N > 0 && K > 0 && K % 8 == 0 && N % 4 == 0 && M < (int64_t(1) << 31) && N < (1 << 30);
}

int tc_gemm(const TcOperand *seg, int nseg, int64_t M, int64_t N, float alpha, float *out, bool accumulate,
            float *partial, uint32_t *status, cudaStream_t st, const TcActEpilogue *act, void *out_bf16,
            float *out_t, int64_t ld_t) {
    TLB_REQUIRE(nseg >= 1 && nseg <= kMaxSeg, TLB_EINVAL, "tcgen05 GEMM: 1 to 3 K segments");
    int64_t K = 0;
    for (int i = 0; i < nseg; ++i) K += seg[i].K;
    const TcPlan pl = tc_plan(M, N, K);
    TLB_REQUIRE(partial != nullptr, TLB_EINVAL, "tcgen05 GEMM: needs a partial-tile buffer");
    if (act != nullptr) {
        TLB_REQUIRE(!accumulate && N % 4 == 0 && aligned16(act->gate) && aligned16(act->up) &&
                        aligned16(act->dgate) && aligned16(act->dup),
                    TLB_EUNSUPPORTED, "tcgen05 GEMM: activation epilogue operands");
    } else {
        TLB_REQUIRE(aligned16(out) && (out_bf16 == nullptr || aligned16(out_bf16)), TLB_EUNSUPPORTED,
                    "tcgen05 GEMM: output alignment");
        TLB_REQUIRE(out != nullptr || (out_t != nullptr && out_bf16 == nullptr), TLB_EINVAL,
                    "tcgen05 GEMM: no output (out may be null only beside the transposed copy)");
    }
    TLB_REQUIRE(act == nullptr || out_bf16 == nullptr, TLB_EINVAL, "tcgen05 GEMM: bf16 copy of an activation epilogue");
    TLB_REQUIRE(out_t == nullptr || (act == nullptr && !accumulate && ld_t >= M && ld_t % 4 == 0 && aligned16(out_t)),
                TLB_EINVAL, "tcgen05 GEMM: transposed copy needs the plain, non-accumulating epilogue, ld_t >= M, "
                            "ld_t %% 4 == 0 and 16-byte alignment");
    TcParams p;
    memset(&p, 0, sizeof(p));
    for (int i = 0; i < nseg; ++i) {
        TLB_REQUIRE(aligned16(seg[i].a) && aligned16(seg[i].b) && seg[i].K % 8 == 0, TLB_EUNSUPPORTED,
                    "tcgen05 GEMM: operand alignment");
        TLB_TRY(make_map(&p.a[i], seg[i].a, M, seg[i].K, kBM));
        TLB_TRY(make_map(&p.b[i], seg[i].b, N, seg[i].K, pl.pair ? pl.bn / 2 : pl.bn));
        p.kb[i] = int(ceil_div(seg[i].K, kBK));
    }
    p.nseg = nseg;
    p.M = int(M);
    p.N = int(N);
    p.alpha = alpha;
    p.out = out;
    p.obf = static_cast<uint2 *>(out_bf16);
    p.out_t = out_t;
    p.ld_t = ld_t;
    p.accumulate = accumulate ? 1 : 0;
    p.partial = partial;
    if (act != nullptr) {
        p.mode = 1;
        p.act = act->act;
        p.gate = act->gate;
        p.up = act->up;
        p.dg = static_cast<uint2 *>(act->dgate);
        p.du = static_cast<uint2 *>(act->dup);
    }
    const int64_t KB = p.kb[0] + (nseg > 1 ? p.kb[1] : 0) + (nseg > 2 ? p.kb[2] : 0), tiles = ceil_div(N, pl.bn) * ceil_div(M, pl.pair ? 2 * kBM : kBM);
    p.ctas = pl.ctas;
    p.dp = pl.dp;
    p.sk_base = int64_t(pl.dp) * pl.ctas * KB;
    p.sk_work = (tiles - int64_t(pl.dp) * pl.ctas) * KB;
    p.status = status;
    if (pl.pair) return launch_tc<256, true>(p, st);
    return pl.bn == 256 ? launch_tc<256, false>(p, st) : launch_tc<128, false>(p, st);
}

}  // namespace tlb
