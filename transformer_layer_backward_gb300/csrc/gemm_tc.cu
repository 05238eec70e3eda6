// Tensor-core (tcgen05) GEMM for the transposed-weight products of the sequence path:
//   C[M, N] (+)= alpha * A[M, K] . B[N, K]^T
// with A the bf16 output gradient (rows = tokens), B a bf16 weight stored [in, out]
// (= [N, K], K-major), fp32 accumulation in tensor memory ([FFN] W_down^T, W_gate^T,
// W_up^T products; [ATT] O-projection backward; [RS] gemm_backward_a).
//
// One CTA computes one 128 x BN tile (cta_group::1):
//   warp 0      TMA producer: 128x64 (A) and BNx64 (B) bf16 tiles, 128-byte swizzle,
//               into a STAGES-deep shared-memory ring guarded by mbarriers
//   warp 1      allocates BN TMEM columns; one thread issues tcgen05.mma.kind::f16
//               (M = 128, N = BN, K = 16) four times per 64-wide k block, and
//               tcgen05.commit frees each stage when its MMAs have completed
//   warps 2..5  epilogue: tcgen05.ld 32x32b.x32 (each warp its 32 TMEM lanes = rows),
//               scale, optional accumulate into C, fp32 stores
// K may come from two segments (A0.B0^T + A1.B1^T, e.g. [dG | dU] . [W_gate | W_up]^T)
// and may be split over gridDim.z CTAs, which then write fp32 partial tiles to a
// workspace that tc_reduce sums.  Every mbarrier wait is bounded (status + wind-down).
#include <cuda.h>

#include <cstring>
#include <mutex>

#include "async.cuh"
#include "common.cuh"
#include "kernels.cuh"
#include "tc.cuh"

namespace tlb {

namespace {

constexpr int kBM = 128, kBK = 64;       // tile rows, k block (64 bf16 = 128 bytes)
constexpr int kStages = 4;
constexpr int kThreadsTC = 192;          // 6 warps

struct TcParams {
    CUtensorMap a[2];                    // bf16 [M, K_seg], box 64 x 128
    CUtensorMap b[2];                    // bf16 [N, K_seg], box 64 x BN
    int kb[2];                           // k blocks of each segment
    int nseg;
    int M, N;
    float alpha;
    float *out;                          // [M, N] fp32 when splits == 1
    int accumulate;
    float *partial;                      // [splits, M, N] fp32 when splits > 1
    uint32_t *status;
};

template <int BN>
__device__ __forceinline__ uint32_t idesc_bf16() {
    return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(BN >> 3) << 17) | (uint32_t(kBM >> 4) << 24);
}

template <int BN>
__global__ void __launch_bounds__(kThreadsTC, 1) tc_gemm_kernel(const __grid_constant__ TcParams p) {
    constexpr int A_BYTES = kBM * kBK * 2, B_BYTES = BN * kBK * 2, STAGE = A_BYTES + B_BYTES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t full[kStages], empty[kStages], tmem_full;
    __shared__ uint32_t tmem_base;
    __shared__ int s_abort, s_issued, s_consumed;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BN, m0 = blockIdx.y * kBM;

    // k blocks of this CTA (split over gridDim.z)
    const int KB = p.kb[0] + (p.nseg > 1 ? p.kb[1] : 0);
    const int kb0 = int(int64_t(KB) * blockIdx.z / gridDim.z), kb1 = int(int64_t(KB) * (blockIdx.z + 1) / gridDim.z);

    if (threadIdx.x == 0) {
        s_abort = 0;
        s_issued = s_consumed = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&tmem_full, 1);
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base, BN);
        tmem_relinquish();
    }
    fence_mbar_init();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_d = tmem_base;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            for (int kb = kb0; kb < kb1; ++kb) {
                const int i = kb - kb0, s = i % kStages;
                if (!mbar_wait(&empty[s], ((i / kStages) & 1) ^ 1, p.status, 10u)) { s_abort = 1; break; }
                const int seg = kb < p.kb[0] ? 0 : 1;
                const int kx = (seg == 0 ? kb : kb - p.kb[0]) * kBK;
                uint8_t *sa = smem + s * STAGE;
                mbar_arrive_expect_tx(&full[s], STAGE);
                tma_load_2d(sa, &p.a[seg], kx, m0, &full[s]);
                tma_load_2d(sa + A_BYTES, &p.b[seg], kx, n0, &full[s]);
                s_issued = i + 1;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16<BN>();
            for (int kb = kb0; kb < kb1; ++kb) {
                const int i = kb - kb0, s = i % kStages;
                if (!mbar_wait(&full[s], (i / kStages) & 1, p.status, 11u)) { s_abort = 1; break; }
                tc_fence_after();
                const uint8_t *sa = smem + s * STAGE;
                const uint64_t ad = sw128_desc(sa), bd = sw128_desc(sa + A_BYTES);
#pragma unroll
                for (int k = 0; k < kBK / 16; ++k)   // 16 bf16 = 32 bytes = 2 descriptor units
                    mma_bf16(tmem_d, ad + 2 * k, bd + 2 * k, idesc, (i > 0 || k > 0) ? 1u : 0u);
                mma_commit(&empty[s]);
                s_consumed = i + 1;
            }
            mma_commit(&tmem_full);               // all MMAs of this CTA done -> epilogue
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2..5)
        const int q = warp & 3;                   // TMEM lane quarter this warp may read
        const int row = m0 + q * 32 + lane;
        const bool ok = mbar_wait(&tmem_full, 0, p.status, 12u);
        tc_fence_after();
        if (ok && kb1 > kb0) {
            for (int j = 0; j < BN / 32; ++j) {
                uint32_t v[32];
                tmem_ld32(tmem_d + (uint32_t(q * 32) << 16) + uint32_t(j * 32), v);
                tmem_wait_ld();
                const int col0 = n0 + j * 32;
                if (row >= p.M || col0 >= p.N) continue;
                if (gridDim.z == 1) {
                    float *o = p.out + int64_t(row) * p.N + col0;
                    if (col0 + 32 <= p.N && (p.N & 3) == 0) {
#pragma unroll
                        for (int t = 0; t < 32; t += 4) {
                            float4 r = make_float4(p.alpha * __uint_as_float(v[t]), p.alpha * __uint_as_float(v[t + 1]),
                                                   p.alpha * __uint_as_float(v[t + 2]),
                                                   p.alpha * __uint_as_float(v[t + 3]));
                            if (p.accumulate) {
                                const float4 c = *reinterpret_cast<const float4 *>(o + t);
                                r.x += c.x; r.y += c.y; r.z += c.z; r.w += c.w;
                            }
                            *reinterpret_cast<float4 *>(o + t) = r;
                        }
                    } else {
                        for (int t = 0; t < 32 && col0 + t < p.N; ++t)
                            o[t] = p.alpha * __uint_as_float(v[t]) + (p.accumulate ? o[t] : 0.f);
                    }
                } else {
                    float *o = p.partial + (int64_t(blockIdx.z) * p.M + row) * p.N + col0;
                    if (col0 + 32 <= p.N && (p.N & 3) == 0) {
#pragma unroll
                        for (int t = 0; t < 32; t += 4)
                            *reinterpret_cast<float4 *>(o + t) = make_float4(
                                __uint_as_float(v[t]), __uint_as_float(v[t + 1]), __uint_as_float(v[t + 2]),
                                __uint_as_float(v[t + 3]));
                    } else {
                        for (int t = 0; t < 32 && col0 + t < p.N; ++t) o[t] = __uint_as_float(v[t]);
                    }
                }
            }
        }
    }
    // wind down: every MMA this CTA issued has completed once tmem_full fired (the
    // epilogue waited for it); after an abort, also wait (bounded) for the tile copies
    // that were issued but never consumed, so nothing lands in shared memory after exit
    tc_fence_before();
    __syncthreads();
    if (s_abort && threadIdx.x == 0) {
        for (int i = s_consumed; i < s_issued; ++i) mbar_wait(&full[i % kStages], (i / kStages) & 1, nullptr, 0u);
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_d, BN);
    }
}

// out[m, n] (+)= alpha * sum_z partial[z, m, n]
__global__ void tc_reduce_kernel(const float4 *__restrict__ part, float4 *out, int64_t mn4, int splits, float alpha,
                                 int accumulate) {
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < mn4; i += int64_t(gridDim.x) * blockDim.x) {
        float4 s = part[i];
        for (int z = 1; z < splits; ++z) {
            const float4 t = part[int64_t(z) * mn4 + i];
            s.x += t.x; s.y += t.y; s.z += t.z; s.w += t.w;
        }
        s.x *= alpha; s.y *= alpha; s.z *= alpha; s.w *= alpha;
        if (accumulate) {
            const float4 c = out[i];
            s.x += c.x; s.y += c.y; s.z += c.z; s.w += c.w;
        }
        out[i] = s;
    }
}

// fp32 [rows, cols] -> bf16 (round to nearest even), 4 at a time
__global__ void to_bf16_kernel(const float4 *__restrict__ x, uint2 *__restrict__ y, int64_t n4) {
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += int64_t(gridDim.x) * blockDim.x) {
        const float4 v = x[i];
        const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
        y[i] = make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
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

template <int BN>
int launch_tc(const TcParams &p, int splits, cudaStream_t st) {
    constexpr int smem = kStages * (kBM * kBK * 2 + BN * kBK * 2) + 1024;
    auto k = tc_gemm_kernel<BN>;
    TLB_CUDA(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    dim3 grid(unsigned(ceil_div(p.N, BN)), unsigned(ceil_div(p.M, kBM)), unsigned(splits));
    k<<<grid, kThreadsTC, smem, st>>>(p);
    return check_launch("tcgen05 gemm");
}

}  // namespace

TcPlan tc_plan(int64_t M, int64_t N, int64_t K) {
    // pick the tile width and K split that minimise (waves x work per CTA): one CTA per
    // SM fits (the 4-stage ring takes 132-197 KB of shared memory)
    const int nsm = num_sms();
    const int64_t KB = ceil_div(K, kBK);
    TcPlan best{256, 1};
    double best_cost = 1e300;
    for (int bn : {256, 128}) {
        const int64_t tiles = ceil_div(N, bn) * ceil_div(M, kBM);
        for (int sp = 1; sp <= kMaxSplits; ++sp) {
            if (sp > 1 && KB / sp < 8) break;
            const int64_t ctas = tiles * sp;
            const double waves = double(ceil_div(ctas, nsm));
            const double cost = waves * (double(bn) * double(ceil_div(KB, sp)) + 2048.0) + (sp > 1 ? 64.0 * sp : 0.0);
            if (cost < best_cost) {
                best_cost = cost;
                best = TcPlan{bn, sp};
            }
        }
    }
    return best;
}

size_t tc_partial_bytes(int64_t M, int64_t N, int64_t K) {
    const TcPlan pl = tc_plan(M, N, K);
    return pl.splits > 1 ? size_t(pl.splits) * M * N * 4 : 0;
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
            float *partial, uint32_t *status, cudaStream_t st) {
    TLB_REQUIRE(nseg == 1 || nseg == 2, TLB_EINVAL, "tcgen05 GEMM: 1 or 2 K segments");
    const int64_t K = seg[0].K + (nseg > 1 ? seg[1].K : 0);
    const TcPlan pl = tc_plan(M, N, K);
    TLB_REQUIRE(pl.splits == 1 || partial != nullptr, TLB_EINVAL, "tcgen05 GEMM: split K needs a partial buffer");
    TLB_REQUIRE(aligned16(out), TLB_EUNSUPPORTED, "tcgen05 GEMM: output alignment");
    TcParams p;
    memset(&p, 0, sizeof(p));
    for (int i = 0; i < nseg; ++i) {
        TLB_REQUIRE(aligned16(seg[i].a) && aligned16(seg[i].b) && seg[i].K % 8 == 0, TLB_EUNSUPPORTED,
                    "tcgen05 GEMM: operand alignment");
        TLB_TRY(make_map(&p.a[i], seg[i].a, M, seg[i].K, kBM));
        TLB_TRY(make_map(&p.b[i], seg[i].b, N, seg[i].K, pl.bn));
        p.kb[i] = int(ceil_div(seg[i].K, kBK));
    }
    p.nseg = nseg;
    p.M = int(M);
    p.N = int(N);
    p.alpha = alpha;
    p.out = out;
    p.accumulate = accumulate ? 1 : 0;
    p.partial = partial;
    p.status = status;
    TLB_TRY(pl.bn == 256 ? launch_tc<256>(p, pl.splits, st) : launch_tc<128>(p, pl.splits, st));
    if (pl.splits > 1) {
        const int64_t mn4 = M * N / 4;
        tc_reduce_kernel<<<stream_grid(mn4, 256), 256, 0, st>>>(reinterpret_cast<const float4 *>(partial),
                                                                reinterpret_cast<float4 *>(out), mn4, pl.splits,
                                                                alpha, accumulate ? 1 : 0);
        TLB_TRY(check_launch("tcgen05 gemm reduce"));
    }
    return TLB_OK;
}

}  // namespace tlb
