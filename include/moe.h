/*
 * libmoe: a single-GPU DeepSeek-V3-style Mixture-of-Experts layer for GB300
 * (sm_103a).  C ABI: plain pointers and sizes, no framework types.
 *
 * The layer (Mixture-of-Kittens blog post, section "Overlapping computation
 * and communication in MoE"; "Mixture-of-Kittens: MoE Megakernel for NVL72s",
 * section 2.1), per token t with x_t in R^d:
 *
 *   logits_t = W_router x_t (+ router_bias)                 router projection
 *   (e_t0..e_t,k-1) = top-k of logits_t, descending, ties to the lower index
 *   g_tj = softmax of the selected logits (= full softmax renormalized on them)
 *   FFN_e(v) = W_down[e] (SiLU(W_gate[e] v) * (W_up[e] v))   SwiGLU expert
 *   y_t = FFN_shared(x_t) + sum_j g_tj FFN_{e_tj}(x_t)       shared weight is 1
 *
 * Routes are grouped by expert with the two-pass counting schedule of the
 * blog's "Scheduling" section (count, prefix offsets, stable write in
 * (token, slot) order).  Floating-point work happens in a fixed order, so every
 * output is bitwise reproducible run to run ("Determinism" section).  The
 * backward returns the router-weight gradient <h, W_down^T dy> ("Router weight
 * gradient computation" section) and propagates it through the softmax into
 * W_router and x.
 *
 * Conventions for every entry point
 *   - Matrices are row-major and contiguous; "bf16" is IEEE bfloat16.
 *   - All pointers are DEVICE pointers unless stated otherwise, 16-byte
 *     aligned.  The caller owns every buffer; the library never allocates,
 *     frees or keeps a pointer after returning.
 *   - `stream` is a cudaStream_t passed as void*; all work is enqueued on it
 *     and nothing synchronizes the host (except moe_read_device_status).
 *     Buffers must stay valid until the stream has executed the work.
 *   - Argument and shape checks run before anything is enqueued: on any
 *     error return nothing has been launched.
 *   - Supported shapes: 1 <= E <= 512, 1 <= top_k <= min(E, 32),
 *     d, I, I_shared multiples of 64, d >= 64, T*top_k + E*127 < 2^31.
 *     T == 0 is valid and does nothing.  Other shapes give MOE_ERR_UNSUPPORTED.
 *   - Device-side problems (a bounded wait that ran out) are recorded in a
 *     status word at the start of the workspace; see moe_read_device_status.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,    /* null/misaligned pointer, negative size */
  MOE_ERR_UNSUPPORTED = 2,    /* shape or precision outside the supported set */
  MOE_ERR_WORKSPACE = 3,      /* workspace pointer missing */
  MOE_ERR_CUDA = 4,           /* a CUDA runtime call or launch failed */
  MOE_ERR_DEVICE = 5,         /* a kernel saw an invalid value */
  MOE_ERR_DEVICE_TIMEOUT = 6  /* a kernel's bounded wait ran out */
} moe_status;

typedef enum { MOE_BF16 = 0, MOE_MXFP8 = 1 } moe_precision;

/* moe_config.flags.
 * MOE_FLAG_REPLAY: the saved state holds the routing and the shared expert's
 *   a and b only; moe_backward first recomputes the routed experts' forward
 *   up to the SwiGLU activation (the expert-grouped x rows, a and b) into its
 *   workspace ("forward activation replay", Mixture-of-Kittens blog post,
 *   section "Reversed ring to minimize forward replay during backward").  The
 *   saved buffer shrinks by Rp*(2d + 4I) bytes in bf16 mode (Rp: routes padded
 *   per expert), the backward workspace grows by as much, and the backward
 *   does the dispatch and the routed gate/up GEMM again.  Results are bitwise
 *   identical to those without the flag. */
#define MOE_FLAG_REPLAY 1u
/* MOE_FLAG_WGRAD_FP32: moe_backward writes dW_gate, dW_up, dW_down and dWs_*
 *   as fp32 (same shapes) instead of bf16: the same fp32 accumulators without
 *   the final rounding, for callers that accumulate gradients in fp32.  bf16 mode only (with MOE_MXFP8 it gives
 *   MOE_ERR_UNSUPPORTED).  dW_router is fp32 either way. */
#define MOE_FLAG_WGRAD_FP32 2u

typedef struct {
  int64_t T;        /* tokens */
  int64_t d;        /* model dimension */
  int64_t I;        /* routed expert intermediate dimension */
  int64_t E;        /* routed experts */
  int64_t top_k;    /* experts per token */
  int64_t n_shared; /* shared experts: 0 or 1 */
  int64_t I_shared; /* shared expert intermediate dimension (ignored if n_shared == 0) */
  int32_t precision;/* moe_precision */
  uint32_t flags;   /* MOE_FLAG_* bits; any other bit gives MOE_ERR_UNSUPPORTED */
} moe_config;

typedef struct {
  const void* W_router;     /* [E, d] bf16 */
  const float* router_bias; /* [E] fp32, or NULL; a constant (no gradient) */
  const void* W_gate;       /* [E, I, d] bf16 */
  const void* W_up;         /* [E, I, d] bf16 */
  const void* W_down;       /* [E, d, I] bf16 */
  const void* Ws_gate;      /* [I_s, d] bf16 (n_shared == 1) */
  const void* Ws_up;        /* [I_s, d] bf16 */
  const void* Ws_down;      /* [d, I_s] bf16 */
  const void* mxfp8;        /* MOE_MXFP8: the buffer moe_quantize_weights_mxfp8 filled from
                               W_gate, W_up and W_down (NULL in bf16 mode) */
} moe_weights;

typedef struct {
  float* dW_router; /* [E, d] fp32 */
  void* dW_gate;    /* [E, I, d] bf16 (fp32 with MOE_FLAG_WGRAD_FP32) */
  void* dW_up;      /* [E, I, d] bf16 (likewise) */
  void* dW_down;    /* [E, d, I] bf16 (likewise) */
  void* dWs_gate;   /* [I_s, d] bf16 (n_shared == 1; likewise) */
  void* dWs_up;     /* [I_s, d] bf16 (likewise) */
  void* dWs_down;   /* [d, I_s] bf16 (likewise) */
  float* d_topk_w;  /* [T, top_k] fp32 router-weight gradient dL/dg, or NULL */
  void* dx_ready;   /* cudaEvent_t or NULL: when given, moe_backward records it on the stream
                       as soon as dx is complete, before the weight gradients are computed,
                       so that a caller can start using dx (e.g. copy it out) early */
} moe_grads;

/* Byte sizes of the caller-allocated buffers for a configuration:
 *   fwd_ws  scratch for moe_forward and moe_route_topk
 *   saved   state moe_forward leaves for moe_backward (routing; the shared
 *           expert's a and b; the routed x rows, a and b unless
 *           MOE_FLAG_REPLAY)
 *   bwd_ws  scratch for moe_backward
 * Each buffer must be 256-byte aligned (moe_route_topk, moe_forward and
 * moe_backward return MOE_ERR_INVALID_ARG otherwise); its first 256 bytes hold
 * the device status word and must be zero before the buffer's first use. */
moe_status moe_workspace_size(const moe_config* cfg, size_t* fwd_ws, size_t* saved, size_t* bwd_ws);

/* MXFP8 mode (precision = MOE_MXFP8, d and I multiples of 128; blog section
 * "MXFP8 support"): the routed experts' GEMMs run on E4M3 operands with one
 * E8M0 scale per 32 elements along each GEMM's reduction axis
 * (X = 2^(floor(log2 amax) - 8), elements rounded to nearest even and
 * saturated at 448); router and shared expert stay bf16.
 * moe_mxfp8_weights_size gives the bytes of the buffer that holds the
 * pre-quantized weights; moe_quantize_weights_mxfp8 fills it from the bf16
 * weights (once per weight update).  The buffer holds, in order, each
 * 256-byte aligned: W_gate and W_up as [E*I, d] along d, W_down as [E*d, I]
 * along I, W_down^T per expert as [E*I, d] along d, and [W_gate; W_up]^T per
 * expert as [E*d, 2I] along 2I, each followed by its scales: for R rows and
 * K columns, R/128 x K/128 blocks of 512 bytes (block (q, g) at offset
 * (g * R/128 + q) * 512; inside it row r, 32-column block j at
 * 16*(r%32) + 4*(r/32) + j) and one spare 512-byte block.  moe_forward and
 * moe_backward read it through moe_weights.mxfp8 (the bf16 W_gate, W_up and
 * W_down must still be given: the shared expert and the router stay bf16,
 * and the saved state is laid out as in bf16 mode). */
moe_status moe_mxfp8_weights_size(const moe_config* cfg, size_t* bytes);
moe_status moe_quantize_weights_mxfp8(const moe_config* cfg, const moe_weights* w, void* mx, void* stream);

/* Router projection, softmax + top-k and the expert schedule (blog sections
 * "Overlapping computation and communication in MoE" and "Scheduling").
 *   x [T, d] bf16; W_router [E, d] bf16; router_bias [E] fp32 or NULL.
 *   logits_in  [T, E] fp32 or NULL: when given, route these logits instead of
 *              computing them (x and W_router may then be NULL).
 *   logits_out [T, E] fp32 or NULL: receives the computed logits.
 *   topk_idx [T, k] int32, topk_w [T, k] fp32: slots in descending-logit order.
 *   counts [E] int32: routes per expert.  offsets [E+1] int32: exclusive
 *   prefix sum of counts.  perm_token [T*k] int32: row r of the expert-grouped
 *   order -> token.  route_row [T, k] int32: (token, slot) -> row.
 *   Rows of one expert are in ascending (token, slot) order.
 *   ws: forward workspace. */
moe_status moe_route_topk(const moe_config* cfg, const void* x, const void* W_router,
                          const float* router_bias, const float* logits_in, float* logits_out,
                          int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
                          int32_t* perm_token, int32_t* route_row, void* ws, void* stream);

/* Routing for callers that cannot allocate device memory.  (The method's pages
 * have no counterpart to this entry point: it exists for the library's users.)
 * Some callers cannot hand the library a workspace: their device memory is
 * owned by a pool fixed when the process starts, or they must not create
 * allocations while they run because an allocation can block, fail or
 * fragment memory that another component manages.  This call computes exactly
 * what moe_route_topk computes, with the same arguments (minus `ws`) and the
 * same results, but keeps its intermediate arrays in one static device array
 * owned by the library (9 MiB, resident on every GPU that loads the library
 * until the process exits) instead of in `ws`.  It allocates nothing.
 *   - It takes BF16 configurations with flags == 0 only; other precisions and
 *     flags return MOE_ERR_UNSUPPORTED (the routing results do not depend on
 *     them).  The rest of the configuration is checked as moe_route_topk
 *     checks it.
 *   - logits_out is required when logits_in is NULL (the computed logits are
 *     not kept in the static array).
 *   - The intermediates take about 12*T*k + 8*E*ceil(T/64) + 504*E bytes plus
 *     2 KB: up to T = 65536 tokens fit at top-8 with 256 experts.  Larger
 *     shapes return MOE_ERR_UNSUPPORTED before anything is enqueued.
 *   - The first call on a device looks up the device address of the static
 *     array (cudaGetSymbolAddress) with that device current.
 *   - All calls on a device share the array.  Calls whose GPU work overlaps
 *     (different streams without ordering between them) race on it and give
 *     wrong results; calls ordered on one stream are safe.
 *   - Device-side problems are not reported: NaN logits, and a bounded wait
 *     of the router projection that ran out (its results are then invalid).
 *     Use moe_route_topk and moe_read_device_status when that matters. */
moe_status moe_route_topk_noalloc(const moe_config* cfg, const void* x, const void* W_router,
                                  const float* router_bias, const float* logits_in, float* logits_out,
                                  int32_t* topk_idx, float* topk_w, int32_t* counts, int32_t* offsets,
                                  int32_t* perm_token, int32_t* route_row, void* stream);

/* Forward of the whole layer: y [T, d] bf16 from x [T, d] bf16.
 * saved: buffer of moe_workspace_size's `saved` bytes that moe_backward will
 * read, or NULL for inference.  ws: forward workspace. */
moe_status moe_forward(const moe_config* cfg, const void* x, const moe_weights* w, void* y,
                       void* saved, void* ws, void* stream);

/* Backward of the layer for L = sum(dy * y), given the `saved` buffer of the
 * matching moe_forward call.  dy [T, d] bf16 -> dx [T, d] bf16 and every
 * weight gradient in `g` (all of them required, d_topk_w optional).  Gradients
 * are written, not accumulated.  ws: backward workspace. */
moe_status moe_backward(const moe_config* cfg, const void* x, const moe_weights* w, const void* dy,
                        const void* saved, void* dx, const moe_grads* g, void* ws, void* stream);

/* Synchronizes `stream`, reads the status word of workspace `ws` (device
 * pointer), resets it to zero and returns it (MOE_OK when no kernel recorded a
 * problem). */
moe_status moe_read_device_status(void* ws, void* stream);

/* Diagnostics, not part of the layer's computation.  While profiling is
 * enabled (process-wide), every launch step of this library is bracketed by
 * two CUDA events recorded on the launching stream, which costs a few
 * microseconds per step.  moe_profile_report waits for the recorded events,
 * writes one line per step name, "<name> <calls> <kernels> <total_ms>\n"
 * (calls: timed calls; kernels: kernels they launched, more than calls where
 * one step runs as several kernels, e.g. a grouped GEMM's 2-SM pass and its
 * pass over leftover tiles), into buf (host memory, NUL-terminated, truncated
 * to buflen bytes) and clears the records.  Returns MOE_ERR_CUDA if an event
 * could not be read. */
moe_status moe_profile_enable(int enable);
moe_status moe_profile_report(char* buf, size_t buflen);

/* Static English description of a status code. */
const char* moe_status_string(moe_status s);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
