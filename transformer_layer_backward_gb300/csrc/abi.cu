// extern "C" entry points of the standalone steps, error reporting and the small
// host-side helpers shared by all translation units.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "common.cuh"
#include "kernels.cuh"

namespace tlb {

static thread_local char g_err[512] = "";
static unsigned long long g_launches = 0;
static void *const *g_prof_events = nullptr;
static int g_prof_n = 0;
// the layer call being profiled: its stream, kernels so far and their names
static bool g_prof_on = false;
static cudaStream_t g_prof_stream = nullptr;
static int g_prof_k = 0;
static const char *g_prof_names[256];
// names of the most recent launches, indexed by launch number modulo kLaunchLog
constexpr unsigned long long kLaunchLog = 4096;
static const char *g_launch_names[kLaunchLog];

static void prof_record(int i, cudaStream_t st) {
    // external record: inside a stream capture this becomes an event node whose
    // timestamps remain readable with cudaEventElapsedTime after the graph runs
    if (g_prof_events != nullptr && i >= 0 && i < g_prof_n)
        cudaEventRecordWithFlags(reinterpret_cast<cudaEvent_t>(g_prof_events[i]), st, cudaEventRecordExternal);
}

ProfileScope::ProfileScope(cudaStream_t st) {
    if (g_prof_events == nullptr) return;
    g_prof_on = true;
    g_prof_stream = st;
    g_prof_k = 0;
    prof_record(0, st);
}

ProfileScope::~ProfileScope() { g_prof_on = false; }

void set_error(const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
}

void clear_error() { g_err[0] = '\0'; }

int check_launch(const char *what) {
    const unsigned long long n = __atomic_fetch_add(&g_launches, 1ull, __ATOMIC_RELAXED);
    g_launch_names[n % kLaunchLog] = what;
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        set_error("%s: kernel launch failed: %s", what, cudaGetErrorString(e));
        return TLB_ECUDA;
    }
    if (g_prof_on) {
        if (g_prof_k < 256) g_prof_names[g_prof_k] = what;
        ++g_prof_k;
        prof_record(g_prof_k, g_prof_stream);
    }
    return TLB_OK;
}

int num_sms() {
    static int n = 0;
    if (n == 0) {
        int dev = 0, v = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
            n = v;
        else
            return 148;
    }
    return n;
}

unsigned stream_grid(int64_t work, int block) {
    const int64_t want = ceil_div(work, block);
    const int64_t cap = int64_t(num_sms()) * 8;
    return (unsigned)(want < 1 ? 1 : (want < cap ? want : cap));
}

void rope_freqs(RopeFreqs &f, int head_dim, float base) {
    for (int d = 0; d < 128; ++d) {
        double v = 0.0;
        if (d < head_dim / 2) v = std::pow(double(base), -2.0 * double(d) / double(head_dim));
        f.hi[d] = float(v);
        f.lo[d] = float(v - double(f.hi[d]));
    }
}

AdamCoef adam_coef(const tlb_adamw_cfg &c, float lr_mult) {
    AdamCoef k;
    k.lr = float(c.lr * double(lr_mult));
    k.beta1 = float(c.beta1);
    k.beta2 = float(c.beta2);
    k.omb1 = float(1.0 - c.beta1);
    k.omb2 = float(1.0 - c.beta2);
    k.eps = float(c.eps);
    k.wd = float(c.weight_decay);
    k.bc1 = float(1.0 / (1.0 - std::pow(double(c.beta1), double(c.step))));
    k.bc2 = float(1.0 / (1.0 - std::pow(double(c.beta2), double(c.step))));
    return k;
}

}  // namespace tlb

using namespace tlb;

extern "C" {

const char *tlb_last_error(void) { return g_err; }

const char *tlb_build_info(void) {
    static char info[128];
    snprintf(info, sizeof(info), "tlb sm_103a build, CUDA %d.%d", CUDART_VERSION / 1000,
             (CUDART_VERSION % 1000) / 10);
    return info;
}

uint64_t tlb_launch_count(void) { return __atomic_load_n(&g_launches, __ATOMIC_RELAXED); }

void tlb_profile_events(void *const *events, int32_t n) {
    g_prof_events = events;
    g_prof_n = events != nullptr && n > 0 ? n : 0;
    g_prof_on = false;
}

const char *tlb_launch_name(uint64_t i) {
    const unsigned long long n = __atomic_load_n(&g_launches, __ATOMIC_RELAXED);
    return (i < n && n - i <= kLaunchLog) ? g_launch_names[i % kLaunchLog] : nullptr;
}

const char *tlb_profile_kernel_name(int32_t k) {
    return (k >= 0 && k < g_prof_k && k < 256) ? g_prof_names[k] : nullptr;
}

size_t tlb_linear_workspace_bytes(int32_t wtype, int64_t S, int64_t out_dim, int64_t in_dim) {
    if (S < 0 || out_dim < 0 || in_dim < 0) return 0;
    return linear_ws_bytes(wtype, S, out_dim, in_dim);
}

int tlb_linear_backward(int32_t wtype, const void *W, float scale, const float *dY, int64_t S,
                        int64_t out_dim, int64_t in_dim, float *dX, int32_t accumulate, void *ws,
                        size_t ws_bytes, void *stream) {
    clear_error();
    TLB_REQUIRE(wtype == TLB_W_F32 || wtype == TLB_W_BF16 || wtype == TLB_W_TERNARY_I8 || wtype == TLB_W_TERNARY_2B,
                TLB_EINVAL, "linear_backward: unknown weight type %d", wtype);
    TLB_REQUIRE(wtype != TLB_W_TERNARY_2B || out_dim % 4 == 0, TLB_EINVAL,
                "linear_backward: packed ternary rows need out_dim %% 4 == 0");
    TLB_REQUIRE(S >= 0 && out_dim >= 0 && in_dim >= 0, TLB_EINVAL, "linear_backward: negative size");
    if (S == 0 || in_dim == 0) return TLB_OK;
    TLB_REQUIRE(W && dX && (dY || out_dim == 0), TLB_EINVAL, "linear_backward: null pointer");
    const size_t need = linear_ws_bytes(wtype, S, out_dim, in_dim);
    TLB_REQUIRE(ws != nullptr && ws_bytes >= need, TLB_EINVAL,
                "linear_backward: workspace of %zu bytes is smaller than the %zu bytes needed", ws_bytes, need);
    return linear_t_launch(wtype, W, scale, dY, S, out_dim, in_dim, dX, accumulate != 0, as_stream(stream), ws,
                           ws_bytes);
}

int tlb_softmax_backward(const float *attn, const float *dattn, float *dscores, int64_t rows,
                         int64_t len, void *stream) {
    clear_error();
    TLB_REQUIRE(rows >= 0 && len >= 0, TLB_EINVAL, "softmax_backward: negative size");
    if (rows == 0 || len == 0) return TLB_OK;
    TLB_REQUIRE(attn && dattn && dscores, TLB_EINVAL, "softmax_backward: null pointer");
    return softmax_backward_launch(attn, dattn, dscores, rows, len, as_stream(stream));
}

int tlb_act_backward(int32_t act, const float *gate, const float *up, const float *silu_gate,
                     const float *dh, float *dgate, float *dup, int64_t n, void *stream) {
    clear_error();
    TLB_REQUIRE(act == TLB_ACT_RELU2_MUL || act == TLB_ACT_SILU_MUL, TLB_EINVAL,
                "act_backward: unknown activation %d", act);
    TLB_REQUIRE(n >= 0, TLB_EINVAL, "act_backward: negative size");
    if (n == 0) return TLB_OK;
    TLB_REQUIRE(gate && up && dh && dgate && dup, TLB_EINVAL, "act_backward: null pointer");
    return act_backward_launch(act, gate, up, silu_gate, dh, dgate, dup, n, as_stream(stream));
}

int tlb_rmsnorm_backward(const float *x, const float *gamma, const float *dy, float *dx, int64_t rows,
                         int64_t n, float eps, int32_t accumulate, void *stream) {
    clear_error();
    TLB_REQUIRE(rows >= 0 && n >= 0, TLB_EINVAL, "rmsnorm_backward: negative size");
    if (rows == 0 || n == 0) return TLB_OK;
    TLB_REQUIRE(x && gamma && dy && dx, TLB_EINVAL, "rmsnorm_backward: null pointer");
    TLB_REQUIRE(!(accumulate && dx == dy), TLB_EINVAL,
                "rmsnorm_backward: dx may alias dy only when accumulate = 0");
    return rmsnorm_backward_launch(x, gamma, dy, dx, rows, n, eps, accumulate ? 1 : 0,
                                   as_stream(stream));
}

int tlb_rope_backward(const float *dy, float *dx, int64_t rows, int32_t n_heads, int32_t head_dim,
                      int64_t pos0, float base, void *stream) {
    clear_error();
    TLB_REQUIRE(rows >= 0 && n_heads >= 0 && pos0 >= 0, TLB_EINVAL, "rope_backward: negative size");
    TLB_REQUIRE(head_dim > 0 && head_dim % 2 == 0, TLB_EINVAL, "rope_backward: head_dim must be even");
    TLB_REQUIRE(head_dim <= 256, TLB_EUNSUPPORTED, "rope_backward: head_dim > 256");
    TLB_REQUIRE(pos0 + rows <= (int64_t(1) << 24), TLB_EUNSUPPORTED,
                "rope_backward: positions >= 2^24");
    if (rows == 0 || n_heads == 0) return TLB_OK;
    TLB_REQUIRE(dy && dx, TLB_EINVAL, "rope_backward: null pointer");
    return rope_backward_launch(dy, dx, rows, n_heads, head_dim, pos0, base, as_stream(stream));
}

int tlb_adamw(float *p, const float *g, float *m, float *v, int64_t n, const tlb_adamw_cfg *cfg,
              float lr_mult, double *sumsq, void *stream) {
    clear_error();
    TLB_REQUIRE(cfg != nullptr, TLB_EINVAL, "adamw: null cfg");
    TLB_REQUIRE(cfg->step >= 1, TLB_EINVAL, "adamw: step must be >= 1");
    TLB_REQUIRE(n >= 0, TLB_EINVAL, "adamw: negative size");
    if (n == 0) return TLB_OK;
    TLB_REQUIRE(p && g && m && v, TLB_EINVAL, "adamw: null pointer");
    return adamw_launch(p, g, m, v, n, *cfg, lr_mult, sumsq, as_stream(stream));
}

int tlb_workspace_status(void *ws, size_t ws_bytes, void *stream) {
    clear_error();
    TLB_REQUIRE(ws != nullptr && ws_bytes >= kStatusBytes, TLB_EINVAL,
                "workspace_status: workspace too small");
    uint32_t words[2] = {0, 0};
    cudaStream_t st = as_stream(stream);
    TLB_CUDA(cudaMemcpyAsync(words, ws, sizeof(words), cudaMemcpyDeviceToHost, st));
    TLB_CUDA(cudaStreamSynchronize(st));
    if (words[kStatusCode] == kDevOk) return TLB_OK;
    TLB_CUDA(cudaMemsetAsync(ws, 0, sizeof(words), st));
    TLB_CUDA(cudaStreamSynchronize(st));
    if (words[kStatusCode] == kDevNonFinite) {
        set_error("device status: non-finite gradient (%s); the adapters were not stepped",
                  words[kStatusWhere] == 1 ? "the dOut entering a layer" : "a layer's dR1");
        return TLB_ENONFINITE;
    }
    set_error("device status: a bounded wait ran out (code %u, site %u)", words[kStatusCode],
              words[kStatusWhere]);
    return TLB_ETIMEOUT;
}

}  // extern "C"
