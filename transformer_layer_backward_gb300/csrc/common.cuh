// Shared helpers of the sm_103a layer-backward library: error reporting, vector
// loads, warp / block reductions, weight-element decoding, workspace carving.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include "tlb.h"

namespace tlb {

// ------------------------------------------------------------------ host side

void set_error(const char *fmt, ...);
void clear_error();

#define TLB_REQUIRE(cond, code, ...)            \
    do {                                        \
        if (!(cond)) {                          \
            ::tlb::set_error(__VA_ARGS__);      \
            return (code);                      \
        }                                       \
    } while (0)

#define TLB_CUDA(call)                                                          \
    do {                                                                        \
        cudaError_t e_ = (call);                                                \
        if (e_ != cudaSuccess) {                                                \
            ::tlb::set_error("%s failed: %s", #call, cudaGetErrorString(e_));   \
            return TLB_ECUDA;                                                   \
        }                                                                       \
    } while (0)

#define TLB_TRY(expr)                  \
    do {                               \
        int rc_ = (expr);              \
        if (rc_ != TLB_OK) return rc_; \
    } while (0)

// Error of the last launch on this thread (a launch error never enqueues work).
int check_launch(const char *what);

// Profiling of one layer call (tlb_profile_events): while a ProfileScope lives, event 0
// is recorded at its start and event k after the k-th kernel launched through
// check_launch, on the scope's stream, and the kernels' names are kept.
struct ProfileScope {
    explicit ProfileScope(cudaStream_t st);
    ~ProfileScope();
};

inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Number of SMs of the current device (queried once per process).
int num_sms();

// Blocks for a grid-stride loop over `work` items: enough to fill the GPU, no more.
unsigned stream_grid(int64_t work, int block);

// Workspace carving: every region 256-byte aligned.  The first region is the
// device status block (kStatusBytes).
constexpr size_t kStatusBytes = 256;
struct WsPlan {
    size_t off = kStatusBytes;
    size_t take(size_t bytes) {
        size_t o = off;
        off += (bytes + 255) & ~size_t(255);
        return o;
    }
};
template <typename T>
inline T *ws_at(void *ws, size_t off) {
    return reinterpret_cast<T *>(reinterpret_cast<char *>(ws) + off);
}

// Device status block (uint32 words at the start of a workspace).
// kStatusGate: with TLB_CHECK_FINITE, 1 if a non-finite gradient was seen by the checks
// ordered before the AdamW kernels that read it (written after each layer's last check).
enum StatusWord { kStatusCode = 0, kStatusWhere = 1, kStatusGate = 2 };
enum DeviceError { kDevOk = 0, kDevTimeout = 1, kDevNonFinite = 2 };

// ------------------------------------------------------------------ device side

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float2 warp_sum2(float2 v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
        v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
    }
    return v;
}

// Sum over all threads of the block; `red` holds >= 32 floats of shared memory.
// Every thread gets the result.  Must be called by all threads of the block.
__device__ __forceinline__ float block_sum(float v, float *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = (blockDim.x + 31) >> 5;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = (lane < nwarps) ? red[lane] : 0.f;
    return warp_sum(t);
}

__device__ __forceinline__ float2 block_sum2(float2 v, float2 *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = (blockDim.x + 31) >> 5;
    v = warp_sum2(v);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float2 t = (lane < nwarps) ? red[lane] : make_float2(0.f, 0.f);
    return warp_sum2(t);
}

// Streaming (read-once) 128-bit loads: no L1 allocation.
__device__ __forceinline__ float4 ld_stream(const float4 *p) {
    float4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w) : "l"(p));
    return r;
}
__device__ __forceinline__ uint4 ld_stream_u4(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

// Programmatic dependent launch: let the next kernel of the stream be scheduled
// (trigger), and wait until the previous kernel has finished and its writes are
// visible (wait; a no-op when the kernel was launched without the attribute).
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Fire-and-forget prefetch of [p, p + bytes) into L2 (p and bytes multiples of 16).
__device__ __forceinline__ void l2_prefetch(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ float dot4(float4 a, float4 b) {
    return a.x * b.x + a.y * b.y + a.z * b.z + a.w * b.w;
}

// Four signed bytes of `w` as exact floats.  Each byte is biased to [0, 255] and
// placed in the mantissa of 2^23 (a float whose ulp is 1); subtracting 2^23 + 128
// then gives the byte's value.  Both steps are exact.
__device__ __forceinline__ void i8x4_to_f32(uint32_t w, float &a, float &b, float &c, float &d) {
    const uint32_t u = w ^ 0x80808080u;
    const float bias = 8388736.0f;   // 2^23 + 128
    a = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7650)) - bias;
    b = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7651)) - bias;
    c = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7652)) - bias;
    d = __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7653)) - bias;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Element idx of a weight matrix of storage type WT, as float (scale not applied).
template <int WT>
__device__ __forceinline__ float weight_at(const void *w, int64_t idx) {
    if constexpr (WT == TLB_W_F32) {
        return __ldg(reinterpret_cast<const float *>(w) + idx);
    } else if constexpr (WT == TLB_W_BF16) {
        unsigned short b = __ldg(reinterpret_cast<const unsigned short *>(w) + idx);
        return __uint_as_float(uint32_t(b) << 16);
    } else if constexpr (WT == TLB_W_TERNARY_I8) {
        return float(__ldg(reinterpret_cast<const signed char *>(w) + idx));
    } else {
        const uint32_t b = __ldg(reinterpret_cast<const unsigned char *>(w) + (idx >> 2));
        return float((b >> (2 * uint32_t(idx & 3))) & 3u) - 1.f;     // code q = w + 1
    }
}

// sum_i q_i x_i over the four 2-bit codes q_i of byte b (lowest bits first) and the four
// floats of x.  Each code becomes an exact float by OR-ing it into the mantissa of 2^23
// and subtracting 2^23; the ternary dot product is this minus the sum of x (w = q - 1),
// which the caller forms once for all the rows that share x.
__device__ __forceinline__ float t2_qdot4(uint32_t b, float4 x) {
    const float q0 = __uint_as_float(0x4B000000u | (b & 3u)) - 8388608.f;
    const float q1 = __uint_as_float(0x4B000000u | ((b >> 2) & 3u)) - 8388608.f;
    const float q2 = __uint_as_float(0x4B000000u | ((b >> 4) & 3u)) - 8388608.f;
    const float q3 = __uint_as_float(0x4B000000u | ((b >> 6) & 3u)) - 8388608.f;
    return fmaf(q3, x.w, fmaf(q2, x.z, fmaf(q1, x.y, q0 * x.x)));
}

// cos and sin of theta = pos * f with f = f_hi + f_lo (a float pair carrying the
// frequency computed in double).  pos * f_hi is formed as a rounded product plus
// its exact rounding error (FMA), the multiple of 2*pi is removed in three parts
// (Cody and Waite's additive range reduction), and only the reduced angle, within
// [-pi, pi], goes to sincosf.  The angle error stays near 2e-7 rad for pos < 2^16.
__device__ __forceinline__ void rope_cos_sin(float pos, float f_hi, float f_lo, float &c, float &s) {
    const float p = pos * f_hi;
    const float e = fmaf(pos, f_hi, -p);
    const float t_lo = fmaf(pos, f_lo, e);
    const float k = rintf(p * 0.15915494309189535f);
    // 2*pi = C1 + C2 + C3 (+ 3e-19): C1 has 8 significant bits, so k * C1 is exact.
    const float C1 = 6.28125f;
    const float C2 = __uint_as_float(0x3afdaa22u);   // 1.9353071693331003e-03
    const float C3 = __uint_as_float(0x2d34611au);   // 1.0253376273028358e-11
    float r = fmaf(-k, C1, p);
    r = fmaf(-k, C2, r);
    r = r + t_lo;
    r = fmaf(-k, C3, r);
    sincosf(r, &s, &c);
}

// Frequencies f_d = base^(-2d/head_dim), d < head_dim/2, as float pairs (filled on
// the host in double).  Passed by value as a kernel parameter.
struct RopeFreqs {
    float hi[128];
    float lo[128];
};
void rope_freqs(RopeFreqs &f, int head_dim, float base);

// Gated-activation backward of one element ([FFN] "ReLU^2 x Mul Backward"; [RS] SwiGLU):
// hidden = act(g) * u, dh = dL/dhidden -> dg = dL/dg, du = dL/du.  With CACHE, s = silu(g)
// comes from the forward's cache.
template <int ACT, bool CACHE>
__device__ __forceinline__ void act_bwd_elem(float g, float u, float s, float dh, float &dg, float &du) {
    if constexpr (ACT == TLB_ACT_RELU2_MUL) {
        const float r = fmaxf(g, 0.f);
        dg = dh * u * 2.f * r;
        du = dh * r * r;
    } else {
        const float sig = 1.f / (1.f + expf(-g));
        const float y = g * sig;
        dg = dh * u * (sig * (1.f + g - y));
        du = dh * (CACHE ? s : y);
    }
}

// The same for results rounded to bf16 (the tensor-core W_down^T epilogue): the exponential
// and the reciprocal are the fast hardware approximations, whose relative error (~1e-6) is
// far below the 2^-9 of the bf16 rounding that follows.
template <int ACT>
__device__ __forceinline__ void act_bwd_elem_bf16(float g, float u, float dh, float &dg, float &du) {
    if constexpr (ACT == TLB_ACT_RELU2_MUL) {
        const float r = fmaxf(g, 0.f);
        dg = dh * u * 2.f * r;
        du = dh * r * r;
    } else {
        const float sig = __fdividef(1.f, 1.f + __expf(-g));
        const float y = g * sig;
        dg = dh * u * (sig * (1.f + g - y));
        du = dh * y;
    }
}

// bf16 outputs (the A operands of the [W_gate | W_up]^T tensor-core GEMM)
__device__ __forceinline__ uint2 pack_bf16x4(float a, float b, float c, float d) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
    return make_uint2(*reinterpret_cast<const uint32_t *>(&lo), *reinterpret_cast<const uint32_t *>(&hi));
}

// AdamW constants of one parameter tensor ([RS] cpu_adamw).  1 - beta and the bias
// corrections are formed in double on the host and rounded once.
struct AdamCoef {
    float lr, beta1, beta2, omb1, omb2, eps, wd, bc1, bc2;
};
AdamCoef adam_coef(const tlb_adamw_cfg &c, float lr_mult);

__device__ __forceinline__ float adam_elem(float p, float g, float &m, float &v, const AdamCoef &k) {
    m = k.beta1 * m + k.omb1 * g;
    v = k.beta2 * v + k.omb2 * g * g;
    const float mh = m * k.bc1, vh = v * k.bc2;
    return p - k.lr * (mh / (sqrtf(vh) + k.eps) + k.wd * p);
}

}  // namespace tlb
