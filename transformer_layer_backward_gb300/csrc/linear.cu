// Input gradient of a linear layer whose weight is stored [in, out]:
//   dX[s, i] (+)= scale * sum_o dY[s, o] * W[i, o]
// ([FFN] W_down^T / W_gate^T / W_up^T products, [ATT] O-projection backward,
//  [RS] gemm_backward_a).  Every output is the dot product of one contiguous
// weight row with one row of dY, so both operands are read along K.
//
//  * S == 1 (single-token decode): a GEMV.  Each warp owns R weight rows and
//    streams them with 128-bit loads; dY sits in shared memory.  Ternary int8
//    weights are decoded exactly with a byte permute and one subtraction.
//  * S > 1: a tiled CUDA-core GEMM (64x64 tiles, fp32 accumulation).  bf16
//    weights take the tensor-core path in gemm_tc.cu when it applies.
#include "common.cuh"
#include "kernels.cuh"

namespace tlb {

// ------------------------------------------------------------------ GEMV (S == 1)

template <int WT>
struct Elem;
template <> struct Elem<TLB_W_F32> { static constexpr int size = 4; };
template <> struct Elem<TLB_W_BF16> { static constexpr int size = 2; };
template <> struct Elem<TLB_W_TERNARY_I8> { static constexpr int size = 1; };
template <> struct Elem<TLB_W_TERNARY_2B> { static constexpr int size = 0; };   // four weights per byte

// Dot product of one 16-byte chunk of a weight row with EPC floats of x.
template <int WT>
__device__ __forceinline__ float chunk_dot(uint4 w, const float *x) {
    if constexpr (WT == TLB_W_F32) {
        return __uint_as_float(w.x) * x[0] + __uint_as_float(w.y) * x[1] +
               __uint_as_float(w.z) * x[2] + __uint_as_float(w.w) * x[3];
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

constexpr int kGemvWarps = 8;

// y[r] (+)= scale * W[r, :] . x for rows r of W [rows, cols]; row bytes a multiple of 16.
template <int WT, int R>
__global__ void __launch_bounds__(kGemvWarps * 32)
gemv_rows_kernel(const void *__restrict__ W, const float *__restrict__ x, float *y, int rows, int cols,
                 float scale, int accumulate) {
    extern __shared__ float4 smem4[];
    float *sx = reinterpret_cast<float *>(smem4);
    for (int c = threadIdx.x; c < cols; c += blockDim.x) sx[c] = x[c];
    __syncthreads();
    constexpr int EPC = 16 / Elem<WT>::size;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r0 = (blockIdx.x * kGemvWarps + warp) * R;
    if (r0 >= rows) return;
    const int nch = cols / EPC;
    const size_t row_bytes = size_t(cols) * Elem<WT>::size;
    const char *wb = reinterpret_cast<const char *>(W);
    float acc[R];
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r] = 0.f;
    for (int ch = lane; ch < nch; ch += 32) {
        uint4 w[R];
#pragma unroll
        for (int r = 0; r < R; ++r)
            w[r] = (r0 + r < rows) ? ld_stream_u4(wb + size_t(r0 + r) * row_bytes + size_t(ch) * 16)
                                   : make_uint4(0, 0, 0, 0);
        float xv[EPC];
#pragma unroll
        for (int e = 0; e < EPC; e += 4) {
            const float4 t = *reinterpret_cast<const float4 *>(sx + ch * EPC + e);
            xv[e] = t.x;
            xv[e + 1] = t.y;
            xv[e + 2] = t.z;
            xv[e + 3] = t.w;
        }
#pragma unroll
        for (int r = 0; r < R; ++r) acc[r] += chunk_dot<WT>(w[r], xv);
    }
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const float s = warp_sum(acc[r]);
        if (lane == 0 && r0 + r < rows) y[r0 + r] = (accumulate ? y[r0 + r] : 0.f) + scale * s;
    }
}

// Any shape / alignment: one warp per row, element loads.
template <int WT>
__global__ void gemv_rows_generic_kernel(const void *__restrict__ W, const float *__restrict__ x, float *y,
                                         int rows, int cols, float scale, int accumulate) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x * (blockDim.x >> 5) + warp;
    if (r >= rows) return;
    float acc = 0.f;
    for (int c = lane; c < cols; c += 32) acc += weight_at<WT>(W, int64_t(r) * cols + c) * x[c];
    acc = warp_sum(acc);
    if (lane == 0) y[r] = (accumulate ? y[r] : 0.f) + scale * acc;
}

template <int WT>
static int launch_gemv(const void *W, const float *x, float *y, int rows, int cols, float scale,
                       int accumulate, cudaStream_t st) {
    constexpr int R = 4;
    const size_t row_bytes = size_t(cols) * Elem<WT>::size;
    const size_t smem = size_t(cols) * sizeof(float);
    // packed ternary rows: the decode chain's streaming kernels serve S = 1 layers; this
    // standalone product reads them one weight at a time
    bool chunked = false;
    if constexpr (Elem<WT>::size > 0) {
        if (row_bytes % 16 == 0 && aligned16(W) && smem <= 200 * 1024) {
            if (smem > 48 * 1024)
                TLB_CUDA(cudaFuncSetAttribute(gemv_rows_kernel<WT, R>,
                                              cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)));
            const int grid = int(ceil_div(rows, kGemvWarps * R));
            gemv_rows_kernel<WT, R><<<grid, kGemvWarps * 32, smem, st>>>(W, x, y, rows, cols, scale, accumulate);
            chunked = true;
        }
    }
    if (!chunked) {
        gemv_rows_generic_kernel<WT><<<unsigned(ceil_div(rows, 8)), 256, 0, st>>>(W, x, y, rows, cols,
                                                                               scale, accumulate);
    }
    return check_launch("gemv");
}

// ------------------------------------------------------------------ CUDA-core GEMM (S > 1)

// C[M, N] (+)= alpha * A[M, K] . B[N, K]^T, A float, B of storage type WT.
template <int WT>
__global__ void __launch_bounds__(256)
gemm_nt_simt_kernel(const float *__restrict__ A, const void *__restrict__ B, float *C, int M, int N,
                    int K, float alpha, int accumulate) {
    __shared__ __align__(16) float As[16][68];
    __shared__ __align__(16) float Bs[16][68];
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
    const int lr = tid >> 2, lk = (tid & 3) * 4;
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    for (int k0 = 0; k0 < K; k0 += 16) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int k = k0 + lk + e;
            const int m = m0 + lr, n = n0 + lr;
            As[lk + e][lr] = (m < M && k < K) ? A[int64_t(m) * K + k] : 0.f;
            Bs[lk + e][lr] = (n < N && k < K) ? weight_at<WT>(B, int64_t(n) * K + k) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            const float4 a = *reinterpret_cast<const float4 *>(&As[kk][ty * 4]);
            const float4 b = *reinterpret_cast<const float4 *>(&Bs[kk][tx * 4]);
            const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty * 4 + i;
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n >= N) continue;
            float* c = C + int64_t(m) * N + n;
            *c = (accumulate ? *c : 0.f) + alpha * acc[i][j];
        }
    }
}

template <int WT>
static int launch_gemm_simt(const float *A, const void *B, float *C, int M, int N, int K, float alpha,
                            int accumulate, cudaStream_t st) {
    dim3 grid(unsigned(ceil_div(N, 64)), unsigned(ceil_div(M, 64)));
    gemm_nt_simt_kernel<WT><<<grid, 256, 0, st>>>(A, B, C, M, N, K, alpha, accumulate);
    return check_launch("gemm_nt_simt");
}

// Workspace of the tensor-core path: [status 256 B][bf16 copy of dY][stream-K partial tiles].
size_t linear_ws_bytes(int wtype, int64_t S, int64_t out_dim, int64_t in_dim) {
    if (wtype != TLB_W_BF16 || S <= 1 || !tc_supported(S, in_dim, out_dim)) return kStatusBytes;
    return kStatusBytes + ((size_t(S) * out_dim * 2 + 255) & ~size_t(255)) + tc_partial_bytes(S, in_dim, out_dim);
}

int linear_t_launch(int wtype, const void *W, float scale, const float *dY, int64_t S, int64_t out_dim,
                    int64_t in_dim, float *dX, bool accumulate, cudaStream_t st, void *ws, size_t ws_bytes) {
    if (S == 0 || in_dim == 0) return TLB_OK;
    TLB_REQUIRE(S < (1 << 30) && out_dim < (1 << 30) && in_dim < (1 << 30), TLB_EUNSUPPORTED,
                "linear backward: dimension >= 2^30");
    const int acc = accumulate ? 1 : 0;
    if (S == 1) {
        switch (wtype) {
            case TLB_W_F32: return launch_gemv<TLB_W_F32>(W, dY, dX, int(in_dim), int(out_dim), scale, acc, st);
            case TLB_W_BF16: return launch_gemv<TLB_W_BF16>(W, dY, dX, int(in_dim), int(out_dim), scale, acc, st);
            case TLB_W_TERNARY_2B:
                return launch_gemv<TLB_W_TERNARY_2B>(W, dY, dX, int(in_dim), int(out_dim), scale, acc, st);
            default: return launch_gemv<TLB_W_TERNARY_I8>(W, dY, dX, int(in_dim), int(out_dim), scale, acc, st);
        }
    }
    if (wtype == TLB_W_BF16 && ws != nullptr && tc_supported(S, in_dim, out_dim) && aligned16(dY) &&
        aligned16(W) && aligned16(dX) && ws_bytes >= linear_ws_bytes(wtype, S, out_dim, in_dim)) {
        char *w = static_cast<char *>(ws);
        void *a = w + kStatusBytes;
        float *part = reinterpret_cast<float *>(w + kStatusBytes + ((size_t(S) * out_dim * 2 + 255) & ~size_t(255)));
        TLB_TRY(tc_convert_bf16(dY, a, S * out_dim, st));
        const TcOperand op{a, W, out_dim};
        return tc_gemm(&op, 1, S, in_dim, scale, dX, accumulate, part, reinterpret_cast<uint32_t *>(w), st);
    }
    switch (wtype) {
        case TLB_W_F32:
            return launch_gemm_simt<TLB_W_F32>(dY, W, dX, int(S), int(in_dim), int(out_dim), scale, acc, st);
        case TLB_W_BF16:
            return launch_gemm_simt<TLB_W_BF16>(dY, W, dX, int(S), int(in_dim), int(out_dim), scale, acc, st);
        case TLB_W_TERNARY_2B:
            return launch_gemm_simt<TLB_W_TERNARY_2B>(dY, W, dX, int(S), int(in_dim), int(out_dim), scale, acc,
                                                      st);
        default:
            return launch_gemm_simt<TLB_W_TERNARY_I8>(dY, W, dX, int(S), int(in_dim), int(out_dim), scale,
                                                      acc, st);
    }
}

}  // namespace tlb
