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
    float *part_b;               // [n_rt][O][rank]
    float *part_gh;              // [n_ot][S][rank]
    float *gh;                   // [S][rank]
    float *part_a;               // [n_rt][rank][C]
};

struct LoraSeqArgs {
    LoraSide side[2];
    const float *x;              // [S, C]
    int nside, S, C, rank, n_rt, vecx;
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

template <int RB>
__global__ void __launch_bounds__(256) lora_gpass_kernel(LoraSeqArgs a) {
    extern __shared__ float4 sm4[];
    float *sG = reinterpret_cast<float *>(sm4);   // [kLT][kLP]
    float *sh = sG + kLT * kLP;                   // [kLT][RB]
    float *sB = sh + kLT * RB;                    // [kLO][RB]
    const int side = (a.nside > 1 && int(blockIdx.x) >= a.side[1].blk0) ? 1 : 0;
    const LoraSide &p = a.side[side];
    const int ot = int(blockIdx.x) - p.blk0, rt = blockIdx.y;
    const int r0 = rt * kLT, o0 = ot * kLO, R = a.rank, tid = threadIdx.x;
    for (int e = tid; e < kLT * RB; e += 256) {
        const int i = e / RB, r = e % RB;
        sh[e] = (r < R && r0 + i < a.S) ? p.h[int64_t(r0 + i) * R + r] : 0.f;
    }
    for (int e = tid; e < kLO * RB; e += 256) {
        const int o = e / RB, r = e % RB;
        sB[e] = (r < R && o0 + o < p.O) ? p.l.b[int64_t(o0 + o) * R + r] : 0.f;
    }
    load_tile(sG, p.G, p.O, a.S, p.O, r0, o0, p.vecG != 0);
    __syncthreads();
    {   // dB partial [128 columns][RB]: thread = (column, half of the ranks)
        constexpr int NB = RB / 2;
        const int o = tid % kLO, rb = (tid / kLO) * NB;
        float acc[NB];
#pragma unroll
        for (int k = 0; k < NB; ++k) acc[k] = 0.f;
#pragma unroll 4
        for (int i = 0; i < kLT; ++i) {
            const float g = sG[i * kLP + o];
#pragma unroll
            for (int k = 0; k < NB; ++k) acc[k] = fmaf(g, sh[i * RB + rb + k], acc[k]);
        }
        if (o0 + o < p.O) {
            float *dst = p.part_b + (int64_t(rt) * p.O + o0 + o) * R;
#pragma unroll
            for (int k = 0; k < NB; ++k)
                if (rb + k < R) dst[rb + k] = acc[k];
        }
    }
    {   // gh partial [64 tokens][RB]: thread = (token, quarter of the ranks)
        constexpr int NG = RB / 4;
        const int i = tid / 4, rb = (tid % 4) * NG;
        float acc[NG];
#pragma unroll
        for (int k = 0; k < NG; ++k) acc[k] = 0.f;
#pragma unroll 4
        for (int o = 0; o < kLO; ++o) {
            const float g = sG[i * kLP + o];
#pragma unroll
            for (int k = 0; k < NG; ++k) acc[k] = fmaf(g, sB[o * RB + rb + k], acc[k]);
        }
        if (r0 + i < a.S) {
            float *dst = p.part_gh + (int64_t(ot) * a.S + r0 + i) * R;
#pragma unroll
            for (int k = 0; k < NG; ++k)
                if (rb + k < R) dst[rb + k] = acc[k];
        }
    }
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
    float acc = 0.f;
    for (int ot = 0; ot < p.n_ot; ++ot) acc += p.part_gh[int64_t(ot) * n + e];
    p.gh[e] = p.s * acc;
}

template <int RB>
__global__ void __launch_bounds__(256) lora_xpass_kernel(LoraSeqArgs a) {
    extern __shared__ float4 sm4[];
    float *sx = reinterpret_cast<float *>(sm4);   // [kLT][kLP]
    float *sg = sx + kLT * kLP;                   // [nside][kLT][RB]
    const int ct = blockIdx.x, rt = blockIdx.y;
    const int c0 = ct * kLO, r0 = rt * kLT, R = a.rank, tid = threadIdx.x;
    for (int sd = 0; sd < a.nside; ++sd)
        for (int e = tid; e < kLT * RB; e += 256) {
            const int i = e / RB, r = e % RB;
            sg[sd * kLT * RB + e] = (r < R && r0 + i < a.S) ? a.side[sd].gh[int64_t(r0 + i) * R + r] : 0.f;
        }
    load_tile(sx, a.x, a.C, a.S, a.C, r0, c0, a.vecx != 0);
    __syncthreads();
    constexpr int NB = RB / 2;
    const int c = tid % kLO, rb = (tid / kLO) * NB;
    for (int sd = 0; sd < a.nside; ++sd) {
        const float *g = sg + sd * kLT * RB;
        float acc[NB];
#pragma unroll
        for (int k = 0; k < NB; ++k) acc[k] = 0.f;
#pragma unroll 4
        for (int i = 0; i < kLT; ++i) {
            const float xv = sx[i * kLP + c];
#pragma unroll
            for (int k = 0; k < NB; ++k) acc[k] = fmaf(g[i * RB + rb + k], xv, acc[k]);
        }
        if (c0 + c < a.C) {
            float *dst = a.side[sd].part_a + int64_t(rt) * R * a.C + c0 + c;
#pragma unroll
            for (int k = 0; k < NB; ++k)
                if (rb + k < R) dst[int64_t(rb + k) * a.C] = acc[k];
        }
    }
}

// One thread per parameter of [A_0 | B_0 | A_1 | B_1].
__global__ void __launch_bounds__(256) lora_seq_adamw_kernel(LoraSeqArgs a, AdamCoef ka, AdamCoef kb,
                                                             double *sumsq) {
    __shared__ float red[32];
    int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    float ssa = 0.f, ssb = 0.f;
    for (int sd = 0; sd < a.nside; ++sd) {
        const LoraSide &p = a.side[sd];
        const int64_t nA = int64_t(a.rank) * a.C, nB = int64_t(p.O) * a.rank;
        if (e < 0) break;
        if (e < nA) {
            float g = 0.f;
            for (int rt = 0; rt < a.n_rt; ++rt) g += p.part_a[int64_t(rt) * nA + e];
            if (p.l.grad_a) p.l.grad_a[e] = g;
            float m = p.l.m_a[e], v = p.l.v_a[e];
            p.l.a[e] = adam_elem(p.l.a[e], g, m, v, ka);
            p.l.m_a[e] = m;
            p.l.v_a[e] = v;
            ssa = g * g;
            e = -1;
        } else if (e < nA + nB) {
            const int64_t f = e - nA;
            float g = 0.f;
            for (int rt = 0; rt < a.n_rt; ++rt) g += p.part_b[int64_t(rt) * nB + f];
            g *= p.s;
            if (p.l.grad_b) p.l.grad_b[f] = g;
            float m = p.l.m_b[f], v = p.l.v_b[f];
            p.l.b[f] = adam_elem(p.l.b[f], g, m, v, kb);
            p.l.m_b[f] = m;
            p.l.v_b[f] = v;
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
int lora_seq_run(const LoraSeqArgs &a, int n_ot_total, const AdamCoef &ka, const AdamCoef &kb, double *sumsq,
                 cudaStream_t st) {
    const size_t smg = size_t(kLT * kLP + kLT * RB + kLO * RB) * 4;
    const size_t smx = size_t(kLT * kLP + 2 * kLT * RB) * 4;
    if (smg > 48 * 1024)
        TLB_CUDA(cudaFuncSetAttribute(lora_gpass_kernel<RB>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smg)));
    if (smx > 48 * 1024)
        TLB_CUDA(cudaFuncSetAttribute(lora_xpass_kernel<RB>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smx)));
    lora_gpass_kernel<RB><<<dim3(unsigned(n_ot_total), unsigned(a.n_rt)), 256, smg, st>>>(a);
    TLB_TRY(check_launch("lora_gpass"));
    const int64_t ngh = int64_t(a.nside) * a.S * a.rank;
    lora_gh_sum_kernel<<<unsigned(ceil_div(ngh, int64_t(256))), 256, 0, st>>>(a);
    TLB_TRY(check_launch("lora_gh_sum"));
    lora_xpass_kernel<RB><<<dim3(unsigned(ceil_div(a.C, kLO)), unsigned(a.n_rt)), 256, smx, st>>>(a);
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
                    const tlb_adamw_cfg &adam, double *sumsq, cudaStream_t st) {
    if (S == 0 || njobs == 0) return TLB_OK;
    TLB_REQUIRE(njobs <= 2, TLB_EINVAL, "lora: at most two adapters per call");
    TLB_REQUIRE(rank >= 1 && rank <= 64, TLB_EINVAL, "lora: rank must be in 1..64");
    const int64_t n_rt = ceil_div(S, int64_t(kLT));
    TLB_REQUIRE(n_rt <= 65535, TLB_EUNSUPPORTED, "lora: S = %lld too long", (long long)S);
    LoraSeqArgs a{};
    a.x = x;
    a.nside = njobs;
    a.S = int(S);
    a.C = in_dim;
    a.rank = rank;
    a.n_rt = int(n_rt);
    a.vecx = (in_dim % 4 == 0 && aligned16(x)) ? 1 : 0;
    int blk = 0;
    for (int sd = 0; sd < njobs; ++sd) {
        const LoraJob &j = jobs[sd];
        LoraSide &p = a.side[sd];
        const SideBytes b = side_bytes(S, j.out_dim, in_dim, rank);
        char *base = static_cast<char *>(j.scratch);
        TLB_REQUIRE((reinterpret_cast<uintptr_t>(base) & 255u) == 0, TLB_EINVAL, "lora: scratch not 256-byte aligned");
        p.G = j.G;
        p.h = j.h;
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
    if (rank <= 4) return lora_seq_run<4>(a, blk, ka, kb, sumsq, st);
    if (rank <= 8) return lora_seq_run<8>(a, blk, ka, kb, sumsq, st);
    if (rank <= 16) return lora_seq_run<16>(a, blk, ka, kb, sumsq, st);
    if (rank <= 32) return lora_seq_run<32>(a, blk, ka, kb, sumsq, st);
    return lora_seq_run<64>(a, blk, ka, kb, sumsq, st);
}

}  // namespace tlb
