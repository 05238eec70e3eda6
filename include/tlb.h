/*
 * tlb.h - C ABI of the GB300 (sm_103a) LoRA transformer layer backward.
 *
 * One call computes one step (or one whole layer) of the backward pass of a
 * transformer layer fine-tuned with LoRA adapters on Q and V, and applies the
 * AdamW step with the LoRA+ learning rate to the adapters.
 *
 * Sources of the operations (page and section):
 *   [FFN] Hesper API, Hesper/Training/FFNBackward ("FFN Backward GPU Kernels"):
 *         the FFN backward chain, ReLU^2 x Mul backward, executeFFNBackward.
 *   [ATT] Hesper API, Hesper/Training/AttentionBackward ("Attention Backward GPU
 *         Kernels"): gradient flow, softmax / score / apply / RoPE / RMSNorm
 *         backward kernels and their execute* wrappers.
 *   [RS]  entrenar train/transformer_trainer/wgpu_backward.rs (aprender-train
 *         0.34.0): cpu_adamw, LayerActivations, backward_through_layers.
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers owned by the caller unless stated otherwise;
 *     tensors are dense, row-major float32 unless stated otherwise.
 *   - Weights are stored [in, out] (the layout the Rust trainer calls
 *     "pre-transposed"), so each input gradient is dX = scale * dY @ W^T.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Calls only enqueue work: they never allocate, free or synchronise (except
 *     tlb_workspace_status), so a sequence of calls can be captured into a CUDA
 *     graph.  Scratch memory comes from the caller's workspace `ws` of `ws_bytes`
 *     bytes (256-byte aligned), sized by tlb_workspace_bytes().  A workspace must be
 *     zero-filled before its first use (it holds a device status block and grid-barrier
 *     counters that every call leaves as it found them); calls sharing a workspace must
 *     not overlap on the GPU.
 *   - Return value: TLB_OK or a negative TLB_E* code; tlb_last_error() gives a
 *     message (thread-local) for the last failing call of this thread.  Argument
 *     errors are detected on the host before anything is enqueued.  Errors found
 *     on the device (a bounded wait that ran out) are recorded in the workspace's
 *     status word and returned by tlb_workspace_status().
 *   - Outputs must not alias inputs unless a function says so.
 */
#ifndef TLB_H_
#define TLB_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TLB_OK 0
#define TLB_EINVAL (-1)        /* bad argument: shape, null pointer, alignment */
#define TLB_EUNSUPPORTED (-2)  /* valid but not implemented (e.g. head_dim > 256) */
#define TLB_ENONFINITE (-3)    /* a non-finite gradient was found (TLB_CHECK_FINITE) */
#define TLB_ETIMEOUT (-4)      /* a device-side bounded wait ran out */
#define TLB_ECUDA (-5)         /* a CUDA runtime call failed */

/* gated activation of the FFN */
#define TLB_ACT_RELU2_MUL 0    /* hidden = max(0, gate)^2 * up            [FFN] */
#define TLB_ACT_SILU_MUL 1     /* hidden = silu(gate) * up (SwiGLU)       [RS]  */

/* weight storage types (all weights of one layer share the type) */
#define TLB_W_F32 0            /* float32 */
#define TLB_W_BF16 1           /* bfloat16 (tensor-core path for S > 1) */
#define TLB_W_TERNARY_I8 2     /* int8 in {-1, 0, +1}; the per-tensor float scale multiplies */
#define TLB_W_TERNARY_2B 3     /* ternary packed four to a byte ([FFN] BitLinear weights): a row of
                                  `out` weights is out / 4 bytes; weight 4k + i of the row sits in
                                  bits 2i, 2i + 1 of byte k as code q = w + 1 (0: -1, 1: 0, 2: +1;
                                  3 is not a valid code).  out must be a multiple of 4; the
                                  per-tensor float scale multiplies.  S = 1 runs the streaming
                                  GEMVs (row lengths multiples of 64 weights), S > 1 the CUDA-core
                                  GEMM */

/* composition flags of a layer */
#define TLB_SUB_NORM 1         /* RMSNorm on the attention context and on the FFN hidden */
#define TLB_PRE_NORM 2         /* RMSNorm before the FFN; its backward adds into dResidual */
#define TLB_RESIDUAL 4         /* r1 = x + attn and out = r1 + ffn */
#define TLB_ROPE 8             /* NeoX split-half rotary embedding on q and k */
#define TLB_USE_SILU_CACHE 16  /* SwiGLU: silu_gate holds silu(gate) and may be read instead of
                                  recomputing it (the fused tensor-core W_down^T epilogue, bound
                                  by its loads, recomputes it all the same) */
#define TLB_CAUSAL 32          /* query row i sees keys j <= L - S + i only; attn is 0 elsewhere */
#define TLB_PERSISTENT 64      /* single-token layers: one persistent cooperative kernel (TMA-streamed
                                  weights, grid barriers) instead of the multi-kernel schedule */
#define TLB_QK_NORM 128        /* q (and k) pass a per-head RMSNorm over head_dim before RoPE ([RS]
                                  LayerActivations caches them after a QK-norm and RoPE): dQ is
                                  taken back through it, which needs q_raw and gamma_q.  Not with
                                  TLB_PERSISTENT (such layers take the multi-kernel schedule) */
#define TLB_CHECK_FINITE 256   /* [RS] backward_through_layers contract C-WGPU-TRAIN-007 (grad_hidden
                                  finite): the dOut entering a layer (or the top of a stack) and each
                                  layer's dR1 (the gradient it hands down) are checked before any
                                  adapter gradient is formed from them.  A non-finite value is
                                  recorded in the workspace status block (tlb_workspace_status then
                                  returns TLB_ENONFINITE) and every later AdamW step of the call
                                  leaves its adapter and moments unchanged; gradient outputs and
                                  sumsq are still written.  Not with TLB_PERSISTENT (such layers take
                                  the multi-kernel schedule) */
#define TLB_EXACT_DIN 512      /* d_hidden returns the exact gradient of the layer input x_in instead of
                                  dR1.  The pages stop the backward at the Q / V projection outputs
                                  ([ATT] "Gradient Flow"; [RS] backward_through_layers); this is the
                                  plain derivative of the same forward with n1 = [RMSNorm(x_in;
                                  gamma_attn)] feeding the Q, K and V projections ([RS] LayerActivations
                                  caches q and k) and both LoRA A products:
                                    dK = scale sum_group dS^T q on the S new cache rows, then RoPE
                                         backward and, with TLB_QK_NORM, the k-side per-head RMSNorm
                                         backward (gamma_k, k_raw);
                                    dn1 = s_q dQpre W_Q^T + s_k dK W_K^T + s_v dV W_V^T
                                          + s (dQpre B_q) A_q + s (dV B_v) A_v   (A, B before AdamW);
                                    d_in = [RESIDUAL: dR1 +] [PRE_NORM: RMSNorm_bwd(x_in, gamma_attn,
                                           dn1), else dn1].
                                  Needs w_q, w_k, w_v and acts->q; with PRE_NORM x_in and gamma_attn;
                                  with TLB_QK_NORM k_raw and gamma_k.  Not with TLB_PERSISTENT, and a
                                  single-token stack runs its layers one after another */
#define TLB_RECOMPUTE_P 1024   /* the attention weights are not read from acts->attn (which may be NULL)
                                  but recomputed where they are used from the queries and the
                                  logsumexp of each query row: attn[h,i,j] = exp(attn_scale <q[i,h],
                                  k[j,kvh]> - lse[h,i]) on the visible keys (flash-style, so that the
                                  [n_heads, S, L] weights need not be cached; [RS] LayerActivations
                                  attn_weights is that cache).  Needs acts->q and acts->lse.  Runs the
                                  CUDA-core attention kernels (fp32) for every S, also with bf16
                                  weights */

/* Shapes and constants of one layer. q_dim = n_heads*head_dim, kv_dim = n_kv_heads*head_dim. */
typedef struct {
    int32_t dim;          /* hidden size H */
    int32_t ffn_dim;      /* intermediate size I */
    int32_t n_heads;
    int32_t n_kv_heads;   /* divides n_heads; KV head of head h is h / (n_heads / n_kv_heads) */
    int32_t head_dim;     /* even, <= 256 */
    int32_t rank;         /* LoRA rank r, 1..64 */
    float lora_alpha;     /* LoRA scaling s = lora_alpha / rank */
    float rope_base;      /* theta_d = pos * rope_base^(-2d/head_dim) */
    float norm_eps;       /* RMSNorm eps: rms = sqrt(mean(x^2) + eps) */
    float attn_scale;     /* softmax logit scale, normally 1/sqrt(head_dim) */
    int32_t act;          /* TLB_ACT_* */
    int32_t wtype;        /* TLB_W_* */
    int32_t flags;        /* TLB_* flags above */
} tlb_layer_cfg;

/* One weight matrix stored [in, out] row-major in cfg.wtype, times `scale`. */
typedef struct {
    const void *w;
    float scale;          /* 1 for plain float weights; the BitLinear scale for ternary */
} tlb_weight;

typedef struct {
    tlb_weight w_down;              /* [ffn_dim, dim] */
    tlb_weight w_gate;              /* [dim, ffn_dim] */
    tlb_weight w_up;                /* [dim, ffn_dim] */
    tlb_weight w_o;                 /* [q_dim, dim]   */
    const float *gamma_sub_ffn;     /* [ffn_dim], TLB_SUB_NORM */
    const float *gamma_ffn;         /* [dim],     TLB_PRE_NORM */
    const float *gamma_sub_attn;    /* [q_dim],   TLB_SUB_NORM */
    const float *gamma_q;           /* [head_dim], TLB_QK_NORM: the per-head norm's gain (all heads) */
    /* TLB_EXACT_DIN only (NULL otherwise): */
    tlb_weight w_q;                 /* [dim, q_dim]  */
    tlb_weight w_k;                 /* [dim, kv_dim] */
    tlb_weight w_v;                 /* [dim, kv_dim] */
    const float *gamma_attn;        /* [dim], with TLB_PRE_NORM: the attention pre-norm's gain */
    const float *gamma_k;           /* [head_dim], with TLB_QK_NORM: the k-side per-head norm's gain */
} tlb_layer_weights;

/* Cached forward activations of one layer ([RS] LayerActivations, [FFN]
 * executeFFNBackward saved buffers).  S query rows sit at positions
 * L - S .. L - 1 of a cache of L keys. */
typedef struct {
    const float *x;          /* attention input (normalised) [S, dim]: LoRA input */
    const float *gate;       /* [S, ffn_dim] */
    const float *up;         /* [S, ffn_dim] */
    const float *silu_gate;  /* [S, ffn_dim] = silu(gate), may be read if TLB_USE_SILU_CACHE */
    const float *hidden;     /* FFN hidden before the sub-norm [S, ffn_dim], TLB_SUB_NORM */
    const float *r1;         /* residual stream before the FFN norm [S, dim], TLB_PRE_NORM */
    const float *ctx;        /* attention context before the sub-norm [S, q_dim], TLB_SUB_NORM */
    const float *k;          /* K cache (after RoPE): element (kvh, j, d) at        */
    const float *v;          /*   k[kvh*kv_stride_head + j*kv_stride_pos + d]; V alike */
    int64_t kv_stride_head;  /* [L, kv_dim] layout: head_dim; [n_kv, L, hd]: L*head_dim */
    int64_t kv_stride_pos;   /* [L, kv_dim] layout: kv_dim;   [n_kv, L, hd]: head_dim   */
    const float *attn;       /* softmax weights [n_heads, S, L] */
    const float *lora_q_h;   /* x @ A_q^T [S, rank] */
    const float *lora_v_h;   /* x @ A_v^T [S, rank] */
    const float *q_raw;      /* Q projection output before the per-head norm [S, q_dim], TLB_QK_NORM */
    /* TLB_EXACT_DIN only (NULL otherwise): */
    const float *x_in;       /* layer input before the attention pre-norm [S, dim], with TLB_PRE_NORM */
    const float *q;          /* queries after RoPE (and the QK-norm) [S, q_dim] */
    const float *k_raw;      /* K projection output of the S new rows before the norm [S, kv_dim], with TLB_QK_NORM */
    /* TLB_RECOMPUTE_P only (NULL otherwise; q above is needed too): */
    const float *lse;        /* [n_heads, S] logsumexp over the visible keys of attn_scale <q[i,h], k[j,kvh]> */
} tlb_layer_acts;

/* A LoRA adapter (A [rank, in], B [out, rank]) and its AdamW moments, updated in place.
 * grad_a / grad_b: optional outputs of the gradients (NULL = not written). */
typedef struct {
    float *a, *b;
    float *m_a, *v_a, *m_b, *v_b;
    float *grad_a, *grad_b;
} tlb_lora;

/* [RS] cpu_adamw hyperparameters; B of each adapter uses lr * lr_b_mult (LoRA+, 16 on the page).
 * Held in double so that 1 - beta and the bias corrections are exact before the kernels
 * round them to float once (0.999f alone is 1.3e-5 away from 0.999 in 1 - beta2). */
typedef struct {
    double lr, beta1, beta2, eps, weight_decay, lr_b_mult;
    int32_t step;            /* >= 1; bias corrections 1/(1 - beta^step) */
} tlb_adamw_cfg;

/* ---------------------------------------------------------------- library */

/* Message of the last failing call on this thread ("" if none). Owned by the library. */
const char *tlb_last_error(void);
/* Build description (compute capability compiled for, version). Owned by the library. */
const char *tlb_build_info(void);
/* Number of kernels this process has enqueued through the library so far (all threads). */
uint64_t tlb_launch_count(void);
/* Name of launch number i (0 = the first launch counted by tlb_launch_count), kept for
 * the last 4096 launches; NULL for an index not yet reached or no longer kept.  Lets a
 * caller see which kernels a call ran: the launches numbered from tlb_launch_count()
 * before the call to tlb_launch_count() after it.  Owned by the library; while other
 * threads call the library an entry may already be overwritten. */
const char *tlb_launch_name(uint64_t i);
/* Benchmarking aid.  With events != NULL, each later tlb_layer_backward call records
 * (cudaEventRecordExternal, so it also works inside stream capture) events[0] on its
 * stream before its first kernel and events[k + 1] right after its k-th kernel, for
 * indices < n, so a caller can time the kernels of a layer one by one; NULL turns it off.
 * Events are cudaEvent_t passed as void*.  Process-wide setting: do not use while other
 * threads call the library. */
void tlb_profile_events(void *const *events, int32_t n);
/* Test hook of the device-side timeout path: the next single-token layer call with
 * TLB_PERSISTENT has block `block` (of its one cooperative kernel) skip its arrival at
 * the kernel's third global-memory grid barrier, a point where no block has a bulk copy
 * in flight.  Every block's bounded wait there runs out (about a second), each records
 * TLB_ETIMEOUT in the workspace status block and leaves; the context stays usable.  The
 * hook then clears itself; block < 0 clears it.  Process-wide: for tests only. */
int tlb_debug_skip_barrier_arrival(int32_t block);
/* Name of the k-th kernel (from 0) of the last layer call profiled with
 * tlb_profile_events, or NULL past its last kernel.  Owned by the library. */
const char *tlb_profile_kernel_name(int32_t k);

/* ---------------------------------------------------------------- standalone steps */

/* [ATT] softmaxBackwardKernel / executeSoftmaxBackward:
 *   dscores[r, j] = attn[r, j] * (dattn[r, j] - sum_j' attn[r, j'] dattn[r, j'])
 * rows x len, row-major.  rows >= 0, len >= 0 (empty is a no-op). */
int tlb_softmax_backward(const float *attn, const float *dattn, float *dscores,
                         int64_t rows, int64_t len, void *stream);

/* [FFN] reluSqrMulBackwardKernel / executeReluSqrMulBackward (act = TLB_ACT_RELU2_MUL):
 *   dgate = dh * up * 2 max(0, gate),  dup = dh * max(0, gate)^2
 * [RS] SiLU backward (act = TLB_ACT_SILU_MUL), sig = 1/(1+e^-g):
 *   dgate = dh * up * sig (1 + g - g sig),  dup = dh * (silu_gate ? silu_gate : g sig)
 * n elements; silu_gate may be NULL. */
int tlb_act_backward(int32_t act, const float *gate, const float *up, const float *silu_gate,
                     const float *dh, float *dgate, float *dup, int64_t n, void *stream);

/* [ATT] rmsNormBackwardKernel / executeRmsNormBackward, one row of n per row:
 *   rms = sqrt(mean(x^2) + eps),  dx = (1/rms) (dy*gamma - x dot(dy*gamma, x) / (n rms^2))
 * accumulate = 0 stores dx, 1 adds it into dx ([FFN] "dResidual +=").  dx may alias dy
 * when accumulate = 0. */
int tlb_rmsnorm_backward(const float *x, const float *gamma, const float *dy, float *dx,
                         int64_t rows, int64_t n, float eps, int32_t accumulate, void *stream);

/* [ATT] ropeBackwardKernel / executeRopeBackward: inverse NeoX rotation R(-theta) of
 * dy [rows, n_heads, head_dim]; row r is at position pos0 + r, theta_d = pos *
 * base^(-2d/head_dim), d < head_dim/2.  dx may alias dy.  head_dim even, <= 256. */
int tlb_rope_backward(const float *dy, float *dx, int64_t rows, int32_t n_heads,
                      int32_t head_dim, int64_t pos0, float base, void *stream);

/* [ATT] O projection backward ("BitLinear transpose"); [FFN] W_down^T, W_gate^T, W_up^T
 * products; [RS] gemm_backward_a (C = A B^T with the weight stored pre-transposed):
 *   dX[S, in_dim] (+)= scale * dY[S, out_dim] . W[in_dim, out_dim]^T
 * W in storage type wtype (TLB_W_*); accumulate = 1 adds into dX.  S = 1 runs a GEMV;
 * S > 1 a GEMM: for bf16 weights on the tcgen05 tensor cores (dY rounded to bf16, fp32
 * accumulation), otherwise on CUDA cores in fp32.  The tensor-core GEMM needs out_dim % 8
 * == 0, in_dim % 4 == 0, dY, W and dX 16-byte aligned and ws_bytes >=
 * tlb_linear_workspace_bytes(); a bf16 call that misses one of these runs the CUDA-core
 * GEMM instead (same result within bf16 rounding; tlb_launch_name shows which ran).
 * ws: zero-filled workspace of at least tlb_linear_workspace_bytes() bytes (bf16 copy of
 * dY and split-K partials). */
size_t tlb_linear_workspace_bytes(int32_t wtype, int64_t S, int64_t out_dim, int64_t in_dim);
int tlb_linear_backward(int32_t wtype, const void *W, float scale, const float *dY, int64_t S,
                        int64_t out_dim, int64_t in_dim, float *dX, int32_t accumulate, void *ws,
                        size_t ws_bytes, void *stream);

/* [RS] cpu_adamw on n parameters with learning rate cfg->lr * lr_mult.
 * If sumsq != NULL (device double), sum(g^2) is added to *sumsq. */
int tlb_adamw(float *p, const float *g, float *m, float *v, int64_t n,
              const tlb_adamw_cfg *cfg, float lr_mult, double *sumsq, void *stream);

/* ---------------------------------------------------------------- layer pieces */

/* Workspace bytes needed by tlb_ffn_backward / tlb_attn_backward /
 * tlb_lora_grad_adamw / tlb_layer_backward for this layer and S, L. */
size_t tlb_workspace_bytes(const tlb_layer_cfg *cfg, int64_t S, int64_t L);

/* Device status recorded in a workspace by earlier calls on `stream`: synchronises
 * the stream, returns TLB_OK or the first device error (TLB_ETIMEOUT or, with
 * TLB_CHECK_FINITE, TLB_ENONFINITE), and clears it.  After TLB_ETIMEOUT the outputs of
 * the call that timed out are undefined; the workspace needs nothing more than this call
 * to be used again (grid-barrier counters are reset by the kernel that used them, on
 * every path out of it). */
int tlb_workspace_status(void *ws, size_t ws_bytes, void *stream);

/* [FFN] executeFFNBackward (sequence form: [RS] backward_through_layers, FFN part).
 *   dF  = dOut W_down^T;  dh = SUB_NORM ? RMSNorm_bwd(hidden, gamma_sub_ffn, dF) : dF
 *   dG, dU = activation backward;  dN2 = dG W_gate^T + dU W_up^T
 *   d_residual = (RESIDUAL ? d_out : 0) + (PRE_NORM ? RMSNorm_bwd(r1, gamma_ffn, dN2) : dN2)
 * d_out [S, dim]; d_residual [S, dim] output, which may alias d_out (the result is
 * then dR1, written over dOut). */
int tlb_ffn_backward(const tlb_layer_cfg *cfg, int64_t S, const float *d_out,
                     const tlb_layer_weights *w, const tlb_layer_acts *acts,
                     float *d_residual, void *ws, size_t ws_bytes, void *stream);

/* [ATT] gradient flow from the O projection down to dQpre; [RS] attention block.
 *   dSub = dR1 W_O^T;  dCtx = SUB_NORM ? RMSNorm_bwd(ctx, gamma_sub_attn, dSub) : dSub
 *   per head h, kvh = h / (n_heads/n_kv_heads):
 *     dAttn = dCtx_h V_kvh^T;  dS = attn_h (dAttn - rowsum(attn_h dAttn));  dQ_h = scale dS K_kvh
 *     dV_kvh += attn_h^T dCtx_h
 *   d_qpre [S, q_dim] = ROPE ? R(-theta) dQ : dQ   (row i at position L - S + i)
 *   d_v    [S, kv_dim] = dV rows of the S newest cache positions L - S .. L - 1
 * d_attn_out = dR1 [S, dim]. */
int tlb_attn_backward(const tlb_layer_cfg *cfg, int64_t S, int64_t L, const float *d_attn_out,
                      const tlb_layer_weights *w, const tlb_layer_acts *acts,
                      float *d_qpre, float *d_v, void *ws, size_t ws_bytes, void *stream);

/* [RS] "LoRA Q backward" / "LoRA V backward" and cpu_adamw, s = alpha / rank:
 *   dB = s G^T h [out, r];  gh = s G B_old [S, r];  dA = gh^T x [r, in]
 *   then AdamW on A (lr) and B (lr * lr_b_mult); B is read before it is updated.
 * G [S, out_dim], h [S, rank], x [S, in_dim].  sumsq (device double[2], may be NULL)
 * += {sum dA^2, sum dB^2}.  S = 0 is a no-op (no gradient, no step).  ws: at least
 * tlb_workspace_bytes of a layer with this rank, dim >= in_dim and q_dim >= out_dim,
 * 256-byte aligned; it holds partial sums over 64-token tiles. */
int tlb_lora_grad_adamw(int64_t S, int32_t out_dim, int32_t in_dim, int32_t rank, float alpha,
                        const float *G, const float *h, const float *x, const tlb_lora *lora,
                        const tlb_adamw_cfg *adam, double *sumsq, void *ws, size_t ws_bytes,
                        void *stream);

/* Same result as tlb_lora_grad_adamw (up to float rounding: its sums over S run per
 * element rather than in tiles), for callers that cannot allocate device memory
 * and so have no workspace to pass (for example code running under an allocator it
 * does not control, or where a cudaMalloc would synchronise the device).  The pages
 * have no counterpart: it exists only for such callers.  Its one scratch buffer, the
 * [S, rank] rows gh, is a fixed 65536-float (256 KiB) array inside the library that
 * every GPU loading the library keeps until the process exits.
 *   - S * rank must not exceed 65536; larger calls fail with TLB_EINVAL.
 *   - It allocates and frees nothing.  Each call outside a stream capture looks up the
 *     array's device address with its device current (so a device reset, which loads
 *     the library's device code again, leaves no stale address); a call inside a capture
 *     uses the address of the last call outside one.  So make one call on each device
 *     before any stream capture, and again after a device reset.
 *   - All calls share the one array and it keeps the last call's contents (every call
 *     overwrites the rows it uses before reading them): calls that overlap on the GPU,
 *     on different streams, race and give wrong results.  Serialise them. */
int tlb_lora_grad_adamw_noalloc(int64_t S, int32_t out_dim, int32_t in_dim, int32_t rank, float alpha,
                                const float *G, const float *h, const float *x, const tlb_lora *lora,
                                const tlb_adamw_cfg *adam, double *sumsq, void *stream);

/* One whole layer: FFN backward, attention backward, LoRA Q/V gradients and AdamW.
 * d_hidden [S, dim] in/out: dOut on entry, the gradient for the layer below on return
 * ([RS] grad_hidden): dR1, or with TLB_EXACT_DIN the exact gradient of the layer input.
 * sumsq (device double[2]) += {sum dA^2, sum dB^2} over both adapters; the page's
 * gradient norm over a stack is sqrt(sumsq[0]).  lora_q: A [r, dim], B [q_dim, r];
 * lora_v: A [r, dim], B [kv_dim, r]. */
int tlb_layer_backward(const tlb_layer_cfg *cfg, int64_t S, int64_t L,
                       const tlb_layer_weights *w, const tlb_layer_acts *acts,
                       const tlb_lora *lora_q, const tlb_lora *lora_v,
                       const tlb_adamw_cfg *adam, float *d_hidden, double *sumsq,
                       void *ws, size_t ws_bytes, void *stream);

/* [RS] backward_through_layers: a stack of n_layers layers of one configuration, run
 * from the top (layer n_layers - 1) down to layer 0.  Layer l's d_in becomes layer
 * l - 1's dOut, its adapters take their AdamW step, and sumsq accumulates over all of
 * them: the result is that of tlb_layer_backward called for l = n_layers - 1 .. 0 in
 * turn on the same d_hidden, up to the order of float atomic additions.
 *   w, acts, lora_q, lora_v: host arrays of n_layers structs, entry l for layer l.
 *   d_hidden [S, dim] in/out: the top layer's dOut on entry, layer 0's d_in on return.
 *   ws: tlb_stack_workspace_bytes(cfg, S, L) bytes, 256-byte aligned, zero-filled once
 *   (four layer workspaces for S = 1, one for S > 1).
 * Single-token layers (S = 1 on the single-token path) overlap: layer l's attention,
 * LoRA and AdamW kernels run on a second, lower-priority stream of the library beside
 * layer l - 1's FFN and O-projection kernels, and `stream` joins that stream before the
 * call's work ends.  The second stream and its events are created on the first such call
 * on each device, which must therefore not be made inside a stream capture; later calls
 * may be captured.  Calls that share that device's second stream are serialised on the
 * host.  Other layers run one after another on `stream`; with bf16 weights and S > 1 each
 * layer's first product reads the bf16 copy of d_in that the layer above left in the
 * workspace instead of converting d_hidden again.  Errors as tlb_layer_backward;
 * n_layers = 0 or S = 0 is a no-op. */
size_t tlb_stack_workspace_bytes(const tlb_layer_cfg *cfg, int64_t S, int64_t L);
int tlb_stack_backward(const tlb_layer_cfg *cfg, int64_t S, int64_t L, int32_t n_layers,
                       const tlb_layer_weights *w, const tlb_layer_acts *acts,
                       const tlb_lora *lora_q, const tlb_lora *lora_v,
                       const tlb_adamw_cfg *adam, float *d_hidden, double *sumsq,
                       void *ws, size_t ws_bytes, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* TLB_H_ */
