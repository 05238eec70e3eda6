// LoRA gradient + AdamW step for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: code that runs under
// an allocator it does not own (a framework's caching allocator that is locked,
// or a memory pool already fully committed to model state), plugins loaded into a
// host process that forbids device allocations after start-up, and code running
// inside a region where a cudaMalloc would synchronise the device and stall other
// work.  tlb_lora_grad_adamw_noalloc serves them: it computes what
// tlb_lora_grad_adamw computes (the same sums, reduced per element over S instead
// of in tiles, so equal up to float rounding), but its only scratch buffer (the
// [S, rank] rows gh = s G B_old) lives in a fixed array inside this library instead
// of in a caller workspace.
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace tlb {

// Largest S * rank the array holds: 65536 floats (256 KiB), e.g. S = 4096 rows at
// rank 16.  Every GPU that loads the library keeps this array until the process exits.
constexpr int64_t kNoAllocGhFloats = 65536;

static __device__ __align__(256) float g_noalloc_gh[kNoAllocGhFloats];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float *g_gh_ptr[kMaxDevices] = {nullptr};

// Device address of g_noalloc_gh on the current device.  In host code the array's
// name is only a host-side stand-in, so the address is asked of the runtime, with the
// device current.  Outside a stream capture it is asked on every call, so that a device
// reset (which loads the module again, possibly elsewhere) never leaves a stale address;
// inside a capture the address of the last call outside one is used.
int gh_address(cudaStream_t st, float **out) {
    int dev = 0;
    TLB_CUDA(cudaGetDevice(&dev));
    TLB_REQUIRE(dev >= 0 && dev < kMaxDevices, TLB_EUNSUPPORTED, "lora_grad_adamw_noalloc: device %d", dev);
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    TLB_CUDA(cudaStreamIsCapturing(st, &cs));
    std::lock_guard<std::mutex> lock(g_mu);
    if (cs == cudaStreamCaptureStatusNone || g_gh_ptr[dev] == nullptr) {
        void *p = nullptr;
        TLB_CUDA(cudaGetSymbolAddress(&p, g_noalloc_gh));
        g_gh_ptr[dev] = static_cast<float *>(p);
    }
    *out = g_gh_ptr[dev];
    return TLB_OK;
}

}  // namespace
}  // namespace tlb

using namespace tlb;

extern "C" int tlb_lora_grad_adamw_noalloc(int64_t S, int32_t out_dim, int32_t in_dim, int32_t rank, float alpha,
                                           const float *G, const float *h, const float *x, const tlb_lora *lora,
                                           const tlb_adamw_cfg *adam, double *sumsq, void *stream) {
    clear_error();
    TLB_REQUIRE(S >= 0 && out_dim > 0 && in_dim > 0, TLB_EINVAL, "lora_grad_adamw_noalloc: bad sizes");
    TLB_REQUIRE(rank >= 1 && rank <= 64, TLB_EINVAL, "lora_grad_adamw_noalloc: rank must be in 1..64");
    TLB_REQUIRE(S * int64_t(rank) <= kNoAllocGhFloats, TLB_EINVAL,
                "lora_grad_adamw_noalloc: S * rank = %lld exceeds the built-in scratch of %lld floats",
                (long long)(S * rank), (long long)kNoAllocGhFloats);
    TLB_REQUIRE(lora && lora->a && lora->b && lora->m_a && lora->v_a && lora->m_b && lora->v_b, TLB_EINVAL,
                "lora_grad_adamw_noalloc: NULL adapter pointer");
    TLB_REQUIRE(adam != nullptr && adam->step >= 1, TLB_EINVAL, "lora_grad_adamw_noalloc: bad adamw cfg");
    TLB_REQUIRE(S == 0 || (G && h && x), TLB_EINVAL, "lora_grad_adamw_noalloc: NULL input");
    if (S == 0) return TLB_OK;
    float *gh = nullptr;
    TLB_TRY(gh_address(as_stream(stream), &gh));
    // gh is written in full by the first kernel before anything reads it, so the
    // array needs no clearing between calls.
    return lora_launch(S, out_dim, in_dim, rank, alpha, G, h, x, *lora, *adam, sumsq, gh, as_stream(stream));
}
