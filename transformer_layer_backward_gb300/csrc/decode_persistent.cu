// Single-token (decode) layer backward as ONE persistent cooperative kernel.
//
// The work is the chain of the FFN backward ([FFN] "Backward (reverse)"), the
// attention backward ([ATT] "Gradient Flow") and the LoRA update ([RS] LoRA blocks,
// cpu_adamw).  Every step depends on a reduction over the previous step's whole
// output, so a multi-kernel version pays a launch, a prologue and a memory latency
// per step while HBM idles.  Here one block per SM runs all phases, separated by
// grid barriers, and the weight rows of the three transposed-weight GEMVs stream into
// shared memory through TMA bulk copies (cp.async.bulk + mbarrier).  Each GEMV warp
// owns two shared-memory slots: while it computes on one, the copy of its next item
// lands in the other, and as soon as an item is consumed the warp starts the copy of
// the item after next -- which belongs to the next phase once the current one is
// done.  So the weights of phase p+1 arrive while the grid barrier and the prologue
// of phase p+1 run, and HBM streams W_down, W_gate | W_up and W_O back to back.
//
//   phase 1  dF   = s_d W_down dOut                      (+ partial sums for the sub-norm)
//   phase 2  dG, dU (sub-norm RMSNorm bwd + gated-activation bwd, per block), then
//            dN2  = s_g W_gate dG + s_u W_up dU   (items: two rows x one column range)
//   phase 3  dR1  = dOut + RMSNorm_bwd(r1, g_ffn, dN2), then dSub = s_o W_O dR1
//   phase 4  per (KV head, 64 keys): dCtx (sub-norm bwd), one pass over K and V:
//            dA = dCtx_h . V[j], U += P dA K[j], W += P K[j], D += P dA per head, so
//            that dQ_h = scale (U_h - D_h W_h) summed over chunks; the chunk holding the
//            current position also forms dV and gh_v
//   phase 5  per head: dQ from the chunk sums, RoPE backward -> dQpre, gh_q
//   phase 6  dB = s G h^T, dA = gh x^T for both adapters, AdamW with LoRA+ on B
//
// Every item of the GEMV phases uses each loaded vector chunk for several weight rows
// (shared-memory bandwidth, not HBM, would otherwise bound the decode), and the dot
// products run on packed f32x2 FMAs with independent accumulators.
//
// Grid barriers count on one monotonic 64-bit word of the workspace (release-add to
// arrive, acquire-load to wait).  Waits are bounded: a timed-out mbarrier or barrier
// records TLB_ETIMEOUT in the workspace status block and the kernel winds down
// (waiting, bounded, for its own copies in flight); the workspace must then be zeroed
// before it is used again.
#include "async.cuh"
#include "common.cuh"
#include "decode.cuh"
#include "kernels.cuh"

#include <algorithm>
#include <atomic>

namespace tlb {

// Test hook (tlb_debug_skip_barrier_arrival): the block of the next persistent call that
// skips its arrival at the third grid barrier, or -1.
static std::atomic<int> g_skip_arrival{-1};

namespace {

constexpr int kPW = 16;                 // warps per block
constexpr int kPT = kPW * 32;
constexpr int kMaxRowsPerItem = 8;
constexpr int kKeysPerItem = 64;        // attention keys per (KV head, chunk) item
constexpr int kMaxBlockRows = 256;      // phase-2 rows per block held in shared memory
constexpr int kSlotsPerWarp = 1;        // shared-memory slots (items in flight) per GEMV warp

struct PArgs {
    DecodeArgs d;
    uint32_t *status;                   // workspace status block
    unsigned long long *gbar;           // [0] grid-barrier arrivals of this call, [1] blocks done;
                                        // the last block done puts both back to zero
    int skip_block;                     // test hook: this block skips its arrival at barrier 3 (-1: none)
    float2 *pp;                         // per-block partial sums, 3 x nblocks
    int nblocks, ngemv, slot_bytes, xbytes;
    int rpi;                            // rows per item in phases 1 and 3
    int nsplit;                         // column ranges of a phase-2 row pair
    int achunks;                        // ceil(L / kKeysPerItem)
    RopeFreqs fr;
};

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_add_u64(unsigned long long *p, unsigned long long v) {
    asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Barrier k (1-based) of this call: every block adds 1 to the monotonic counter and
// waits until it reaches base + k * nblocks.
__device__ __forceinline__ bool grid_sync(const PArgs &p, int k, unsigned long long base, int *s_abort) {
    __syncthreads();
    if (threadIdx.x == 0 && !*s_abort) {
        __threadfence();
        if (!(k == 3 && int(blockIdx.x) == p.skip_block)) red_release_add_u64(p.gbar, 1ull);
        const unsigned long long target = base + (unsigned long long)k * p.nblocks;
        if (ld_acquire_u64(p.gbar) < target) {
            const long long t0 = clock64();
            while (ld_acquire_u64(p.gbar) < target) {
                if (clock64() - t0 > kWaitLimitCycles) {
                    report_timeout(p.status, 100u + unsigned(k));
                    *s_abort = 1;
                    break;
                }
            }
        }
        __threadfence();
    }
    __syncthreads();
    return *s_abort == 0;
}

// Rows [b * R / nb, (b + 1) * R / nb) of an R-row phase belong to block b.
__device__ __forceinline__ void block_rows(int R, int b, int nb, int &r0, int &r1) {
    r0 = int(int64_t(R) * b / nb);
    r1 = int(int64_t(R) * (b + 1) / nb);
}

struct ItemMap {
    int n1, n2, n3;                       // items of phases 1..3 of this block
    int a0, a1, b0, b1, c0, c1;           // row ranges of phases 1..3
};

__device__ __forceinline__ ItemMap item_map(const PArgs &p) {
    ItemMap m;
    block_rows(p.d.I, blockIdx.x, p.nblocks, m.a0, m.a1);
    block_rows(p.d.H, blockIdx.x, p.nblocks, m.b0, m.b1);
    block_rows(p.d.qd, blockIdx.x, p.nblocks, m.c0, m.c1);
    m.n1 = (m.a1 - m.a0 + p.rpi - 1) / p.rpi;
    m.n2 = ((m.b1 - m.b0 + 1) / 2) * p.nsplit;
    m.n3 = (m.c1 - m.c0 + p.rpi - 1) / p.rpi;
    return m;
}

// Lane 0: start the bulk copy of item g (block-local numbering over phases 1..3).
template <int WT>
__device__ __forceinline__ void issue_item(const PArgs &p, const ItemMap &m, int g, char *slot, uint64_t *bar) {
    constexpr int ES = 16 / EPC<WT>::v;
    const DecodeArgs &d = p.d;
    fence_proxy_async();
    if (g < m.n1) {
        const int r0 = m.a0 + g * p.rpi;
        const int k = min(p.rpi, m.a1 - r0);
        const uint32_t rb = uint32_t(d.H) * ES;
        mbar_arrive_expect_tx(bar, rb * k);
        tma_load_1d(slot, static_cast<const char *>(d.w_down) + size_t(r0) * rb, rb * k, bar);
    } else if (g < m.n1 + m.n2) {
        // rows h, h + 1 (k2 of them) of W_gate then of W_up, column range q of each:
        // slot = [W_gate row h | W_gate row h+1 | W_up row h | W_up row h+1]
        const int j = g - m.n1;
        const int h = m.b0 + 2 * (j / p.nsplit), q = j % p.nsplit;
        const int k2 = min(2, m.b1 - h);
        const uint32_t rb = uint32_t(d.I) * ES;            // full row bytes
        const uint32_t pb = rb / p.nsplit;                  // bytes of one column range
        mbar_arrive_expect_tx(bar, 2 * k2 * pb);
        for (int r = 0; r < k2; ++r) {
            const size_t off = size_t(h + r) * rb + size_t(q) * pb;
            tma_load_1d(slot + r * pb, static_cast<const char *>(d.w_gate) + off, pb, bar);
            tma_load_1d(slot + (2 + r) * pb, static_cast<const char *>(d.w_up) + off, pb, bar);
        }
    } else {
        const int r0 = m.c0 + (g - m.n1 - m.n2) * p.rpi;
        const int k = min(p.rpi, m.c1 - r0);
        const uint32_t rb = uint32_t(d.H) * ES;
        mbar_arrive_expect_tx(bar, rb * k);
        tma_load_1d(slot, static_cast<const char *>(d.w_o) + size_t(r0) * rb, rb * k, bar);
    }
}

__device__ __forceinline__ unsigned long long f2pack(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float f2sum(unsigned long long v) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return lo + hi;
}
__device__ __forceinline__ unsigned long long f2fma(unsigned long long a, unsigned long long b, unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ unsigned long long f2add(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Weight pair j (elements 2j, 2j+1) of a 16-byte chunk, as packed floats.
template <int WT>
__device__ __forceinline__ unsigned long long wpair(uint4 w, int j) {
    const uint32_t q[4] = {w.x, w.y, w.z, w.w};
    if constexpr (WT == TLB_W_F32) {
        return f2pack(__uint_as_float(q[2 * j]), __uint_as_float(q[2 * j + 1]));
    } else if constexpr (WT == TLB_W_BF16) {
        return f2pack(bf16_lo(q[j]), bf16_hi(q[j]));
    } else {
        // int8 -> float: byte biased into the mantissa of 2^23, then 2^23 + 128 removed (exact)
        const uint32_t u = q[j >> 1] ^ 0x80808080u;
        const uint32_t s0 = (j & 1) ? 0x7652u : 0x7650u, s1 = (j & 1) ? 0x7653u : 0x7651u;
        const unsigned long long raw = f2pack(__uint_as_float(__byte_perm(u, 0x4B000000u, s0)),
                                              __uint_as_float(__byte_perm(u, 0x4B000000u, s1)));
        return f2add(raw, 0xCB000080CB000080ull);   // (-8388736, -8388736)
    }
}

// One warp: k (<= R) rows of nch 16-byte chunks in shared memory (row stride rb bytes),
// starting at chunk ch0 of the full vector, dotted with the swizzled vector x; the k
// sums (times scale) go to every lane.  Each vector chunk is read once for all rows.
template <int WT, int R>
__device__ __forceinline__ void dot_rows(const char *slot, int k, int nch, uint32_t rb, int ch0, const float *x,
                                         float scale, float *out) {
    constexpr int E = EPC<WT>::v, P = E / 4;
    const int lane = threadIdx.x & 31;
    unsigned long long acc[R][2];
#pragma unroll
    for (int r = 0; r < R; ++r) acc[r][0] = acc[r][1] = 0ull;
    for (int c = lane; c < nch; c += 32) {
        ulonglong2 xv[P];
#pragma unroll
        for (int q = 0; q < P; ++q) xv[q] = reinterpret_cast<const ulonglong2 *>(x)[xunit<WT>((ch0 + c) * P + q)];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (r < k) {
                const uint4 w = *reinterpret_cast<const uint4 *>(slot + r * rb + c * 16);
#pragma unroll
                for (int j = 0; j < E / 2; ++j) {
                    const unsigned long long xp = (j & 1) ? xv[j >> 1].y : xv[j >> 1].x;
                    acc[r][j & 1] = f2fma(wpair<WT>(w, j), xp, acc[r][j & 1]);
                }
            }
        }
    }
#pragma unroll
    for (int r = 0; r < R; ++r) out[r] = scale * warp_sum(f2sum(acc[r][0]) + f2sum(acc[r][1]));
}

// Sum of nb partials (every thread gets it).
__device__ __forceinline__ float2 sum_pp(const float2 *pp, int nb, float2 *red) {
    float2 acc = make_float2(0.f, 0.f);
    for (int i = threadIdx.x; i < nb; i += blockDim.x) {
        const float2 t = __ldcg(pp + i);
        acc.x += t.x;
        acc.y += t.y;
    }
    return block_sum2(acc, red);
}

__device__ __forceinline__ void coef(float2 s, int n, float eps, float &rinv, float &c) {
    const float ms = s.y / float(n) + eps;
    rinv = rsqrtf(ms);
    c = s.x / float(n) / ms;
}

template <int WT, int VPL>
__device__ __forceinline__ void persistent_body(const PArgs &p) {
    constexpr int GM = 16 / VPL;                 // heads per KV group held in registers
    constexpr int ES = 16 / EPC<WT>::v;
    extern __shared__ float4 smem4[];
    __shared__ uint64_t mbar[kSlotsPerWarp * kPW];
    __shared__ float2 red[32];
    __shared__ int s_abort;
    __shared__ unsigned long long s_base;
    __shared__ float2 s_acc[kPW];
    __shared__ float racc[kMaxBlockRows];
    const DecodeArgs &d = p.d;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    char *smem = reinterpret_cast<char *>(smem4);
    float *sX = reinterpret_cast<float *>(smem);
    char *slots = smem + p.xbytes;
    const bool gemv_warp = warp < p.ngemv;

    if (threadIdx.x == 0) {
        s_abort = 0;
        s_base = 0;   // every call finds the counter at zero (the last block of the previous one reset it)
    }
    if (lane == 0 && gemv_warp)
        for (int i = 0; i < kSlotsPerWarp; ++i) mbar_init(&mbar[kSlotsPerWarp * warp + i], 1);
    fence_mbar_init();
    __syncthreads();
    const unsigned long long base = s_base;

    const ItemMap m = item_map(p);
    const int total = m.n1 + m.n2 + m.n3;
    // the first items of each GEMV warp: the weights start streaming right away
    if (gemv_warp && lane == 0) {
        for (int i = 0; i < kSlotsPerWarp; ++i) {
            const int g = warp + i * p.ngemv;
            const int sidx = kSlotsPerWarp * warp + i;
            if (g < total) issue_item<WT>(p, m, g, slots + size_t(sidx) * p.slot_bytes, &mbar[sidx]);
        }
    }
    if (blockIdx.x == 0 && threadIdx.x < 2 * d.rank) d.gh[threadIdx.x] = 0.f;   // gh_q | gh_v accumulators
    // phase 1 vector: dOut
    {
        const float4 *x4 = reinterpret_cast<const float4 *>(d.d_hidden);
        for (int u = threadIdx.x; u < (d.H >> 2); u += blockDim.x) reinterpret_cast<float4 *>(sX)[xunit<WT>(u)] = x4[u];
    }
    __syncthreads();

    int it = 0;              // index of this warp's next item (its global number is warp + it * ngemv)
    bool ok = true;
    // ---------------------------------------------------------------- phases 1..3: GEMVs
    for (int phase = 1; phase <= 3; ++phase) {
        float rinv = 1.f, c = 0.f;
        if (phase == 2) {
            if (!grid_sync(p, 1, base, &s_abort)) { ok = false; break; }
            const bool sub = d.flags & TLB_SUB_NORM;
            if (sub) coef(sum_pp(p.pp, p.nblocks, red), d.I, d.eps, rinv, c);
            const bool cache = d.act == TLB_ACT_SILU_MUL && (d.flags & TLB_USE_SILU_CACHE);
            float *sG = sX, *sU = sX + d.I;
            const int n4 = d.I >> 2;
            for (int i = threadIdx.x; i < n4; i += blockDim.x) {
                const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
                const float4 df = __ldcg(reinterpret_cast<const float4 *>(d.dF) + i);
                const float4 hd = sub ? reinterpret_cast<const float4 *>(d.hidden)[i] : z;
                const float4 gm = sub ? reinterpret_cast<const float4 *>(d.g_sub_ffn)[i] : z;
                const float4 ga = reinterpret_cast<const float4 *>(d.gate)[i];
                const float4 uu = reinterpret_cast<const float4 *>(d.up)[i];
                const float4 sl = cache ? reinterpret_cast<const float4 *>(d.silu_gate)[i] : z;
                const float dfv[4] = {df.x, df.y, df.z, df.w}, hdv[4] = {hd.x, hd.y, hd.z, hd.w};
                const float gmv[4] = {gm.x, gm.y, gm.z, gm.w}, gav[4] = {ga.x, ga.y, ga.z, ga.w};
                const float uuv[4] = {uu.x, uu.y, uu.z, uu.w}, slv[4] = {sl.x, sl.y, sl.z, sl.w};
                float og[4], ou[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float dh = sub ? rinv * (dfv[e] * gmv[e] - hdv[e] * c) : dfv[e];
                    const float gg = gav[e], u = uuv[e];
                    if (d.act == TLB_ACT_RELU2_MUL) {
                        const float r = fmaxf(gg, 0.f);
                        og[e] = dh * u * 2.f * r;
                        ou[e] = dh * r * r;
                    } else {
                        const float sig = 1.f / (1.f + expf(-gg));
                        const float y = gg * sig;
                        og[e] = dh * u * (sig * (1.f + gg - y));
                        ou[e] = dh * (cache ? slv[e] : y);
                    }
                }
                reinterpret_cast<float4 *>(sG)[xunit<WT>(i)] = make_float4(og[0], og[1], og[2], og[3]);
                reinterpret_cast<float4 *>(sU)[xunit<WT>(i)] = make_float4(ou[0], ou[1], ou[2], ou[3]);
            }
            for (int i = threadIdx.x; i < m.b1 - m.b0; i += blockDim.x) racc[i] = 0.f;
            __syncthreads();
        } else if (phase == 3) {
            if (!grid_sync(p, 2, base, &s_abort)) { ok = false; break; }
            const bool pre = d.flags & TLB_PRE_NORM, resid = d.flags & TLB_RESIDUAL;
            if (pre) coef(sum_pp(p.pp + p.nblocks, p.nblocks, red), d.H, d.eps, rinv, c);
            const int n4 = d.H >> 2;
            for (int i = threadIdx.x; i < n4; i += blockDim.x) {
                const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
                const float4 dn = __ldcg(reinterpret_cast<const float4 *>(d.dN2) + i);
                const float4 r = pre ? reinterpret_cast<const float4 *>(d.r1)[i] : z;
                const float4 gm = pre ? reinterpret_cast<const float4 *>(d.g_ffn)[i] : z;
                const float4 dO = resid ? reinterpret_cast<const float4 *>(d.d_hidden)[i] : z;
                float4 v;
                v.x = (pre ? rinv * (dn.x * gm.x - r.x * c) : dn.x) + dO.x;
                v.y = (pre ? rinv * (dn.y * gm.y - r.y * c) : dn.y) + dO.y;
                v.z = (pre ? rinv * (dn.z * gm.z - r.z * c) : dn.z) + dO.z;
                v.w = (pre ? rinv * (dn.w * gm.w - r.w * c) : dn.w) + dO.w;
                reinterpret_cast<float4 *>(sX)[xunit<WT>(i)] = v;
                if (blockIdx.x == 0) reinterpret_cast<float4 *>(d.dR1)[i] = v;
            }
            __syncthreads();
        }
        const int gend = phase == 1 ? m.n1 : (phase == 2 ? m.n1 + m.n2 : total);
        const int gbeg = phase == 1 ? 0 : (phase == 2 ? m.n1 : m.n1 + m.n2);
        float2 acc = make_float2(0.f, 0.f);     // (sum y g z, sum z^2) of phases 1 and 3, lane 0
        if (gemv_warp) {
            for (int g = warp + it * p.ngemv; g < gend; g = warp + it * p.ngemv) {
                const int sidx = kSlotsPerWarp * warp + (it % kSlotsPerWarp);
                char *slot = slots + size_t(sidx) * p.slot_bytes;
                if (!mbar_wait(&mbar[sidx], (it / kSlotsPerWarp) & 1, p.status, 1u)) { ok = false; break; }
                float out[kMaxRowsPerItem];
                int row0 = 0, k = 0;
                if (phase == 2) {
                    const int j = g - m.n1;
                    row0 = m.b0 + 2 * (j / p.nsplit);
                    k = min(2, m.b1 - row0);
                    const int q = j % p.nsplit;
                    const int cols = d.I / p.nsplit;
                    const uint32_t pb = uint32_t(cols) * ES;
                    const int nch = cols / EPC<WT>::v;
                    float o2[2];
                    dot_rows<WT, 2>(slot, k, nch, pb, q * nch, sX, d.s_gate, out);
                    dot_rows<WT, 2>(slot + 2 * pb, k, nch, pb, q * nch, sX + d.I, d.s_up, o2);
                    out[0] += o2[0];
                    out[1] += o2[1];
                } else {
                    const int base_r = phase == 1 ? m.a0 : m.c0;
                    const int lim = phase == 1 ? m.a1 : m.c1;
                    row0 = base_r + (g - gbeg) * p.rpi;
                    k = min(p.rpi, lim - row0);
                    dot_rows<WT, kMaxRowsPerItem>(slot, k, d.H / EPC<WT>::v, uint32_t(d.H) * ES, 0, sX,
                                                  phase == 1 ? d.s_down : d.s_o, out);
                }
                __syncwarp();
                if (lane == 0) {
                    const int gn = g + kSlotsPerWarp * p.ngemv;
                    if (gn < total) issue_item<WT>(p, m, gn, slot, &mbar[sidx]);
                    if (phase == 2) {
                        atomicAdd(&racc[row0 - m.b0], out[0]);
                        if (k > 1) atomicAdd(&racc[row0 + 1 - m.b0], out[1]);
                    } else {
                        float *y = phase == 1 ? d.dF : d.dSub;
                        const float *gam = phase == 1 ? d.g_sub_ffn : d.g_sub_attn;
                        const float *z = phase == 1 ? d.hidden : d.ctx;
#pragma unroll
                        for (int r = 0; r < kMaxRowsPerItem; ++r) {
                            if (r < k) {
                                y[row0 + r] = out[r];
                                if (gam != nullptr) {
                                    const float zz = z[row0 + r];
                                    acc.x += out[r] * gam[row0 + r] * zz;
                                    acc.y += zz * zz;
                                }
                            }
                        }
                    }
                }
                ++it;
            }
        }
        if (lane == 0) s_acc[warp] = acc;
        __syncthreads();
        if (phase == 2) {
            // the block's dN2 rows are complete in racc: store them, partial sums for the pre-norm
            float2 t = make_float2(0.f, 0.f);
            for (int i = threadIdx.x; i < m.b1 - m.b0; i += blockDim.x) {
                const float v = racc[i];
                d.dN2[m.b0 + i] = v;
                if (d.g_ffn != nullptr) {
                    const float zz = d.r1[m.b0 + i];
                    t.x += v * d.g_ffn[m.b0 + i] * zz;
                    t.y += zz * zz;
                }
            }
            t = block_sum2(t, red);
            if (threadIdx.x == 0) p.pp[p.nblocks + blockIdx.x] = t;
        } else if (threadIdx.x == 0) {
            float2 t = make_float2(0.f, 0.f);
            for (int w = 0; w < kPW; ++w) {
                t.x += s_acc[w].x;
                t.y += s_acc[w].y;
            }
            p.pp[(phase == 1 ? 0 : 2) * p.nblocks + blockIdx.x] = t;
        }
        if (!ok) s_abort = 1;
        __syncthreads();
        if (s_abort) break;
    }
    if (s_abort) {
        // wind down: wait (bounded) for this warp's copies still in flight, then leave
        if (gemv_warp) {
            for (int i = it; i < it + kSlotsPerWarp; ++i)
                if (warp + i * p.ngemv < total)
                    mbar_wait(&mbar[kSlotsPerWarp * warp + (i % kSlotsPerWarp)], (i / kSlotsPerWarp) & 1, p.status, 2u);
        }
        return;
    }
    // ---------------------------------------------------------------- phase 4: attention
    if (!grid_sync(p, 3, base, &s_abort)) return;
    {
        const int G = d.nh / d.nkv, hd = VPL * 32;
        float rinv = 1.f, c = 0.f;
        const bool sub = d.flags & TLB_SUB_NORM;
        if (sub) coef(sum_pp(p.pp + 2 * p.nblocks, p.nblocks, red), d.qd, d.eps, rinv, c);
        if (blockIdx.x == 0)
            for (int i = threadIdx.x; i < d.H; i += blockDim.x) d.d_hidden[i] = __ldcg(d.dR1 + i);
        float *sC = reinterpret_cast<float *>(smem);            // [G][hd]
        float *sR = sC + G * hd;                                // [kPW][G][2][hd]
        __shared__ float sDp[kPW][GM];
        const int nitems = d.nkv * p.achunks;
        for (int it = blockIdx.x; it < nitems; it += p.nblocks) {
            const int kvh = it / p.achunks, chunk = it % p.achunks;
            __syncthreads();
            for (int i = threadIdx.x; i < G * hd; i += blockDim.x) {
                const int q = kvh * G * hd + i;
                const float ds = __ldcg(d.dSub + q);
                sC[i] = sub ? rinv * (ds * d.g_sub_attn[q] - d.ctx[q] * c) : ds;
            }
            __syncthreads();
            const int d0 = lane * VPL;
            float U[GM][VPL], W[GM][VPL], dsum[GM];
#pragma unroll
            for (int gg = 0; gg < GM; ++gg) {
                dsum[gg] = 0.f;
#pragma unroll
                for (int v = 0; v < VPL; ++v) U[gg][v] = W[gg][v] = 0.f;
            }
            constexpr int KPW = kKeysPerItem / kPW;
#pragma unroll
            for (int kk = 0; kk < KPW; ++kk) {
                const int j = chunk * kKeysPerItem + warp * KPW + kk;
                if (j >= d.L) break;
                float kv[VPL], vv[VPL];
                const float *kr = d.k + int64_t(kvh) * d.sh + int64_t(j) * d.sp + d0;
                const float *vr = d.v + int64_t(kvh) * d.sh + int64_t(j) * d.sp + d0;
#pragma unroll
                for (int v = 0; v < VPL; ++v) {
                    kv[v] = kr[v];
                    vv[v] = vr[v];
                }
                const float pl = lane < G ? d.attn[int64_t(kvh * G + lane) * d.L + j] : 0.f;
#pragma unroll
                for (int gg = 0; gg < GM; ++gg) {
                    if (gg >= G) break;
                    float t = 0.f;
#pragma unroll
                    for (int v = 0; v < VPL; ++v) t = fmaf(sC[gg * hd + d0 + v], vv[v], t);
                    const float dA = warp_sum(t);
                    const float P = __shfl_sync(0xffffffffu, pl, gg);
                    const float pd = P * dA;
                    dsum[gg] += pd;
#pragma unroll
                    for (int v = 0; v < VPL; ++v) {
                        U[gg][v] = fmaf(pd, kv[v], U[gg][v]);
                        W[gg][v] = fmaf(P, kv[v], W[gg][v]);
                    }
                }
            }
#pragma unroll
            for (int gg = 0; gg < GM; ++gg) {
                if (gg >= G) break;
#pragma unroll
                for (int v = 0; v < VPL; ++v) {
                    sR[((warp * G + gg) * 2 + 0) * hd + d0 + v] = U[gg][v];
                    sR[((warp * G + gg) * 2 + 1) * hd + d0 + v] = W[gg][v];
                }
                if (lane == 0) sDp[warp][gg] = dsum[gg];
            }
            __syncthreads();
            for (int i = threadIdx.x; i < G * 2 * hd; i += blockDim.x) {
                float t = 0.f;
#pragma unroll
                for (int w = 0; w < kPW; ++w) t += sR[w * G * 2 * hd + i];
                const int gg = i / (2 * hd), which = (i / hd) & 1, dd = i % hd;
                float *dst = which ? d.Wpart : d.Upart;
                dst[(int64_t(chunk) * d.nh + kvh * G + gg) * hd + dd] = t;
            }
            if (threadIdx.x < G) {
                float t = 0.f;
                for (int w = 0; w < kPW; ++w) t += sDp[w][threadIdx.x];
                d.Dpart[int64_t(chunk) * d.nh + kvh * G + threadIdx.x] = t;
            }
            // dV of the current token and its share of gh_v
            if (d.pos / kKeysPerItem == chunk) {
                __shared__ float sv[256];
                __shared__ float rr[16][kPW];
                for (int dd = threadIdx.x; dd < hd; dd += blockDim.x) {
                    float t = 0.f;
                    for (int gg = 0; gg < G; ++gg)
                        t = fmaf(d.attn[int64_t(kvh * G + gg) * d.L + d.pos], sC[gg * hd + dd], t);
                    sv[dd] = t;
                    d.dv[kvh * hd + dd] = t;
                }
                __syncthreads();
                float ar[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) ar[r] = 0.f;
                for (int dd = threadIdx.x; dd < hd; dd += blockDim.x) {
                    const float *br = d.lv.b + int64_t(kvh * hd + dd) * d.rank;
#pragma unroll
                    for (int r = 0; r < 16; ++r)
                        if (r < d.rank) ar[r] = fmaf(sv[dd], br[r], ar[r]);
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    const float t = warp_sum(ar[r]);
                    if (lane == 0) rr[r][warp] = t;
                }
                __syncthreads();
                if (threadIdx.x < d.rank) {
                    float t = 0.f;
                    for (int w = 0; w < kPW; ++w) t += rr[threadIdx.x][w];
                    atomicAdd(d.gh + d.rank + threadIdx.x, d.lora_scaling * t);
                }
            }
        }
    }
    // ---------------------------------------------------------------- phase 5: dQpre, gh_q
    if (!grid_sync(p, 4, base, &s_abort)) return;
    for (int h = blockIdx.x; h < d.nh; h += p.nblocks) {
        const int hd = VPL * 32;
        float *su = reinterpret_cast<float *>(smem);           // [groups][hd] partial U
        float *sw = su + kPT;                                   // [groups][hd] partial W
        float *sq = sw + kPT;                                   // [hd]
        __shared__ float sD;
        __shared__ float red16[16][kPW];
        const int groups = kPT / hd;
        const int grp = threadIdx.x / hd, dd = threadIdx.x % hd;
        __syncthreads();
        if (threadIdx.x < 32) {
            float t = 0.f;
            for (int c = lane; c < p.achunks; c += 32) t += __ldcg(d.Dpart + int64_t(c) * d.nh + h);
            t = warp_sum(t);
            if (lane == 0) sD = t;
        }
        {
            float u = 0.f, w = 0.f;
            for (int c = grp; c < p.achunks; c += groups) {
                const int64_t idx = (int64_t(c) * d.nh + h) * hd + dd;
                u += __ldcg(d.Upart + idx);
                w += __ldcg(d.Wpart + idx);
            }
            su[threadIdx.x] = u;
            sw[threadIdx.x] = w;
        }
        __syncthreads();
        for (int t = threadIdx.x; t < hd; t += blockDim.x) {
            float u = 0.f, w = 0.f;
            for (int q = 0; q < groups; ++q) {
                u += su[q * hd + t];
                w += sw[q * hd + t];
            }
            sq[t] = d.scale * (u - sD * w);
        }
        __syncthreads();
        const int half = hd >> 1;
        for (int t = threadIdx.x; t < half; t += blockDim.x) {
            float y1 = sq[t], y2 = sq[t + half];
            if (d.flags & TLB_ROPE) {
                float cs, sn;
                rope_cos_sin(float(d.pos), p.fr.hi[t], p.fr.lo[t], cs, sn);
                const float t1 = y1 * cs + y2 * sn, t2 = -y1 * sn + y2 * cs;
                y1 = t1;
                y2 = t2;
            }
            d.dqpre[h * hd + t] = y1;
            d.dqpre[h * hd + t + half] = y2;
            sq[t] = y1;
            sq[t + half] = y2;
        }
        __syncthreads();
        float ar[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) ar[r] = 0.f;
        for (int t = threadIdx.x; t < hd; t += blockDim.x) {
            const float *br = d.lq.b + int64_t(h * hd + t) * d.rank;
#pragma unroll
            for (int r = 0; r < 16; ++r)
                if (r < d.rank) ar[r] = fmaf(sq[t], br[r], ar[r]);
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const float t = warp_sum(ar[r]);
            if (lane == 0) red16[r][warp] = t;
        }
        __syncthreads();
        if (threadIdx.x < d.rank) {
            float t = 0.f;
            for (int w = 0; w < kPW; ++w) t += red16[threadIdx.x][w];
            atomicAdd(d.gh + threadIdx.x, d.lora_scaling * t);
        }
    }
    // ---------------------------------------------------------------- phase 6: LoRA + AdamW
    if (!grid_sync(p, 5, base, &s_abort)) return;
    {
        const int64_t nbq = int64_t(d.qd) * d.rank, nbv = int64_t(d.kvd) * d.rank, na = int64_t(d.rank) * d.H;
        const int64_t n = nbq + nbv + 2 * na;
        float sa = 0.f, sb = 0.f;
        for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < n; e += int64_t(p.nblocks) * blockDim.x) {
            if (e < nbq) {
                const int o = int(e / d.rank), r = int(e % d.rank);
                const float gq = d.lora_scaling * __ldcg(d.dqpre + o) * d.hq[r];
                if (d.lq.grad_b) d.lq.grad_b[e] = gq;
                float mm = d.lq.m_b[e], vv = d.lq.v_b[e];
                d.lq.b[e] = adam_elem(d.lq.b[e], gq, mm, vv, d.kb);
                d.lq.m_b[e] = mm;
                d.lq.v_b[e] = vv;
                sb += gq * gq;
            } else if (e < nbq + nbv) {
                const int64_t f = e - nbq;
                const int o = int(f / d.rank), r = int(f % d.rank);
                const float gv = d.lora_scaling * __ldcg(d.dv + o) * d.hv[r];
                if (d.lv.grad_b) d.lv.grad_b[f] = gv;
                float mm = d.lv.m_b[f], vv = d.lv.v_b[f];
                d.lv.b[f] = adam_elem(d.lv.b[f], gv, mm, vv, d.kb);
                d.lv.m_b[f] = mm;
                d.lv.v_b[f] = vv;
                sb += gv * gv;
            } else {
                const int64_t f = e - nbq - nbv;
                const bool isq = f < na;
                const int64_t f2 = isq ? f : f - na;
                const int r = int(f2 / d.H), cidx = int(f2 % d.H);
                const tlb_lora &l = isq ? d.lq : d.lv;
                const float ga = __ldcg(d.gh + (isq ? 0 : d.rank) + r) * d.x[cidx];
                if (l.grad_a) l.grad_a[f2] = ga;
                float mm = l.m_a[f2], vv = l.v_a[f2];
                l.a[f2] = adam_elem(l.a[f2], ga, mm, vv, d.ka);
                l.m_a[f2] = mm;
                l.v_a[f2] = vv;
                sa += ga * ga;
            }
        }
        if (d.sumsq) {
            const float2 s = block_sum2(make_float2(sa, sb), red);
            if (threadIdx.x == 0) {
                atomicAdd(d.sumsq, double(s.x));
                atomicAdd(d.sumsq + 1, double(s.y));
            }
        }
    }
}

// Every block, on every path out of the body (including a wind-down after a bounded wait
// ran out), counts itself done; the last one resets the barrier counter, so that each call
// starts from zero whatever the previous call on this workspace went through.
template <int WT, int VPL>
__global__ void __launch_bounds__(kPT, 1) dec_persistent(PArgs p) {
    persistent_body<WT, VPL>(p);
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(p.gbar + 1, 1ull) == (unsigned long long)(p.nblocks - 1)) {
            atomicExch(p.gbar, 0ull);
            atomicExch(p.gbar + 1, 0ull);
            __threadfence();
        }
    }
}

template <int WT, int VPL>
int launch_p(const PArgs &p, size_t dyn, cudaStream_t st) {
    auto k = dec_persistent<WT, VPL>;
    TLB_CUDA(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, int(dyn)));
    int per_sm = 0;
    TLB_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kPT, dyn));
    TLB_REQUIRE(per_sm >= 1, TLB_EUNSUPPORTED, "decode: persistent kernel does not fit an SM");
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(p.nblocks));
    cfg.blockDim = dim3(kPT);
    cfg.dynamicSmemBytes = dyn;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    TLB_CUDA(cudaLaunchKernelEx(&cfg, k, p));
    TLB_TRY(check_launch("decode persistent"));
    return TLB_OK;
}

template <int WT>
int launch_vpl(const PArgs &p, size_t dyn, cudaStream_t st) {
    switch (p.d.hd) {
        case 32: return launch_p<WT, 1>(p, dyn, st);
        case 64: return launch_p<WT, 2>(p, dyn, st);
        case 128: return launch_p<WT, 4>(p, dyn, st);
        default: return launch_p<WT, 8>(p, dyn, st);
    }
}

struct Geometry {
    int slot_bytes, xbytes, ngemv, rpi, nsplit;
    size_t dyn;
};

bool geometry(const tlb_layer_cfg &c, Geometry &g) {
    const int es = c.wtype == TLB_W_F32 ? 4 : (c.wtype == TLB_W_BF16 ? 2 : 1);
    const int E = 16 / es;
    const int hd = c.head_dim, G = c.n_heads / c.n_kv_heads;
    const int64_t rowH = int64_t(c.dim) * es, rowI = int64_t(c.ffn_dim) * es;
    // phase-2 items: the two weights' rows cut into nsplit column ranges of whole chunks,
    // so that an item stays near 8 KiB
    // phase-2 items: two rows of W_gate and of W_up, one of nsplit column ranges of whole
    // chunks, about 14 KiB in all
    g.nsplit = 1;
    for (int n = 1; n <= 8; ++n) {
        if (c.ffn_dim % (n * E)) continue;
        g.nsplit = n;
        if (4 * rowI / n <= 14336) break;
    }
    g.slot_bytes = int(std::max<int64_t>(4 * rowI / g.nsplit, rowH));
    g.rpi = int(std::min<int64_t>(kMaxRowsPerItem, g.slot_bytes / rowH));
    g.xbytes = int(((std::max<int64_t>(c.dim, 2 * int64_t(c.ffn_dim)) * 4) + 127) / 128 * 128);
    int dev = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return false;
    const int64_t budget = int64_t(optin) - 8 * 1024;     // static shared memory and slack
    g.ngemv = int(std::min<int64_t>(kPW, (budget - g.xbytes) / (kSlotsPerWarp * int64_t(g.slot_bytes))));
    if (g.ngemv < 4) return false;
    const size_t attn = size_t(1 + 2 * kPW) * G * hd * 4;          // dCtx + per-warp U, W
    const size_t fin = size_t(2 * kPT + 256) * 4;                   // per-head finalize
    g.dyn = std::max({size_t(g.xbytes) + size_t(kSlotsPerWarp) * g.ngemv * g.slot_bytes, attn, fin});
    return int64_t(g.dyn) <= budget;
}

}  // namespace

bool persistent_supported(const tlb_layer_cfg &c, int64_t S, int64_t L) {
    const int hd = c.head_dim, G = c.n_heads / c.n_kv_heads;
    const int E = c.wtype == TLB_W_F32 ? 4 : (c.wtype == TLB_W_BF16 ? 8 : 16);
    if (S != 1 || L < 1 || c.rank > 16 || c.n_heads > kPT || (c.flags & TLB_QK_NORM)) return false;
    if (c.wtype == TLB_W_TERNARY_2B) return false;    // packed weights take the multi-kernel chain
    if (!(hd == 32 || hd == 64 || hd == 128 || hd == 256) || G * (hd / 32) > 16) return false;
    if (c.dim % E || c.ffn_dim % E || c.dim % 4 || c.ffn_dim % 4) return false;
    if (ceil_div(c.dim, std::min(num_sms(), kMaxPersistentBlocks)) + 1 > kMaxBlockRows) return false;
    Geometry g;
    return geometry(c, g);
}

int decode_persistent_launch(const DecodeArgs &d, const tlb_layer_cfg &c, int64_t L, void *ws, size_t off_gbar,
                             size_t off_pp, cudaStream_t st) {
    Geometry g;
    TLB_REQUIRE(geometry(c, g), TLB_EUNSUPPORTED, "decode: no persistent geometry");
    PArgs p;
    p.d = d;
    p.skip_block = g_skip_arrival.exchange(-1);
    p.status = ws_at<uint32_t>(ws, 0);
    p.gbar = ws_at<unsigned long long>(ws, off_gbar);
    p.pp = ws_at<float2>(ws, off_pp);
    p.nblocks = std::min(num_sms(), kMaxPersistentBlocks);
    p.ngemv = g.ngemv;
    p.slot_bytes = g.slot_bytes;
    p.xbytes = g.xbytes;
    p.rpi = g.rpi;
    p.nsplit = g.nsplit;
    p.achunks = int(ceil_div(L, kKeysPerItem));
    rope_freqs(p.fr, c.head_dim, c.rope_base);
    switch (c.wtype) {
        case TLB_W_F32: return launch_vpl<TLB_W_F32>(p, g.dyn, st);
        case TLB_W_BF16: return launch_vpl<TLB_W_BF16>(p, g.dyn, st);
        default: return launch_vpl<TLB_W_TERNARY_I8>(p, g.dyn, st);
    }
}

}  // namespace tlb

extern "C" int tlb_debug_skip_barrier_arrival(int32_t block) {
    tlb::g_skip_arrival.store(block < 0 ? -1 : int(block));
    return TLB_OK;
}
