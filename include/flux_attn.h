/*
 * flux_attn.h -- C ABI of the B300 (sm_103a) joint text/image attention library.
 *
 * One operation: the attention forward pass of a FLUX-style diffusion
 * transformer block, where the text tokens, the noisy target-image tokens and
 * (for image-to-image) the reference-image tokens are concatenated into one
 * sequence and attend jointly ("Speed up image generation with FLUX 3 Image
 * Klein on NVIDIA Blackwell GPUs", section "FLUX 3 inference with TensorRT LLM
 * VisualGen").  Q and K first get per-head RMSNorm and multi-axis rotary
 * position embedding, the normalisation and RoPE that the same page's section
 * "GEMM kernel optimisation" fuses into the QKV projection.  An FP8 (E4M3)
 * variant with per-(batch, head) scales follows the same page's section
 * "Quantized and sparse attention" (qk_dtype fp8, v_dtype fp8).
 *
 * Math, per batch b and head h, with d = head_dim = 128:
 *   q'_n = RoPE(RMSNorm(q_n) * w_q, pos_n),  k'_n = RoPE(RMSNorm(k_n) * w_k, pos_n)
 *   RMSNorm(x)_i = x_i / sqrt(mean_j x_j^2 + eps)
 *   RoPE: the head dimension is cut into consecutive blocks of axes_dim[0..2]
 *         dims; in block a the adjacent pair (2j, 2j+1) is rotated by
 *         pos_n[a] * theta^(-2j / axes_dim[a]).
 *   out_n = sum_m softmax_m(q'_n . k'_m / sqrt(d)) v_m   (no mask, non-causal)
 *
 * Conventions shared by every call:
 *   - Tensors q, k, v, out are bf16, layout [B, N, H, 128], contiguous
 *     (token-major, heads interleaved, the layout a QKV projection writes).
 *   - N = txt_len + img_h * img_w + ref_h * ref_w, token order
 *     [text | image row-major | reference row-major].
 *   - Every pointer is a DEVICE pointer unless stated otherwise, 16-byte
 *     aligned, owned by the caller, and must stay valid until the work
 *     enqueued on `stream` has completed.  The library owns its workspace.
 *   - Calls enqueue work on `stream` and return without synchronising.  One
 *     handle serves one stream at a time (its workspace is shared).
 *   - The attention kernel (and the QKV GEMM) is launched with programmatic
 *     stream serialisation: it may be scheduled while the kernel before it
 *     in the stream is finishing, and it waits for that kernel to complete
 *     before it reads any memory, so stream order holds as usual.
 *   - Every call returns a flux_attn_status.  On a nonzero status nothing was
 *     enqueued, except FLUX_ATTN_ERR_CUDA from a failed launch.  Errors found
 *     on the device (a bounded wait that ran out) are reported later by
 *     flux_attn_sync_status.  flux_attn_last_error() describes the last
 *     failure of the calling thread.
 */
#ifndef FLUX_ATTN_H
#define FLUX_ATTN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define FLUX_ATTN_API __attribute__((visibility("default")))
#else
#define FLUX_ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FLUX_ATTN_OK = 0,
  FLUX_ATTN_ERR_INVALID_ARG = 1,    /* bad pointer, size, alignment or geometry */
  FLUX_ATTN_ERR_UNSUPPORTED = 2,    /* device is not compute capability 10.3, or head_dim != 128 */
  FLUX_ATTN_ERR_OOM = 3,            /* workspace allocation failed in create */
  FLUX_ATTN_ERR_CUDA = 4,           /* a CUDA runtime or driver call failed */
  FLUX_ATTN_ERR_DEVICE_TIMEOUT = 5  /* a kernel's bounded wait ran out; its output is invalid */
} flux_attn_status;

typedef enum {
  FLUX_ATTN_BF16 = 0,      /* bf16 Q'/K'/V/P operands, fp32 accumulation */
  FLUX_ATTN_FP8_E4M3 = 1   /* E4M3 Q'/K'/V operands with per-(b, h) scales, E4M3 P */
} flux_attn_precision;

/* debug_flags bits */
#define FLUX_ATTN_DEBUG_FORCE_TIMEOUT 1  /* the attention kernel waits on a barrier nothing
                                            signals; every CTA gives up after its bounded
                                            wait and sync_status reports DEVICE_TIMEOUT */

typedef struct {
  int batch;          /* B >= 1 */
  int num_heads;      /* 1 <= H <= 192 */
  int head_dim;       /* must be 128 */
  int max_tokens;     /* upper bound on N for every later call (sizes the workspace) */
  int axes_dim[3];    /* RoPE axis block sizes, even, summing to head_dim; FLUX uses 16, 56, 56 */
  float rope_theta;   /* RoPE base, FLUX uses 10000 */
  float rms_eps;      /* RMSNorm epsilon, FLUX uses 1e-6 */
  int precision;      /* flux_attn_precision */
  int debug_flags;    /* FLUX_ATTN_DEBUG_* bits, 0 in production */
  float vc_repair_budget;  /* VC-Attention repair budget rho in [0, 1] (FP8 handles only; 0 = plain
                              FP8).  Per (b, h) the R = ceil(rho N) key tokens with the largest
                              quantisation error |k' - deq(k')|^2 + |v - deq(v)|^2 attend with their
                              exact K', V ("Quantized and sparse attention": vc_attention,
                              vc_repair_budget 0.005; the worst-quantised share of the tokens has
                              its quantisation residual corrected).  Equal errors: the lower
                              token index is repaired first. */
  float sol_tau;      /* Sol-Attention threshold tau >= 0 (BF16 handles only; 0 = no block-sparse
                         calls).  Per (b, h), 128-token query block i keeps 128-key block j when the
                         pooled mass mu_ij = c_j exp(q_bar_i . k_bar_j / sqrt(128)) / sum_j' (...)
                         (means of the normalised, rotated rows; c_j = keys in block j) is at least
                         tau / nb, and always keeps its block of largest mass ("Quantized and sparse
                         attention": algorithm sol_attn, tau 1.0). */
  float sol_disabled_until_timestep;  /* flux_attn_forward_sol runs dense while timestep > this
                                         value (the page's configuration: 0.96 on a schedule
                                         that falls from 1 to 0) */
} flux_attn_config;

typedef struct flux_attn* flux_attn_t;

/* Create a handle on the current CUDA device: checks the device, allocates
 * the workspace for cfg->max_tokens (BF16: normalised Q'/K', a V buffer and
 * the RoPE table of the QKV projection; FP8: codes and scales; both: the
 * device error word).  *out receives the handle (NULL on failure). */
FLUX_ATTN_API int flux_attn_create(const flux_attn_config* cfg, flux_attn_t* out);

/* Destroy a handle and free its workspace.  The caller must have completed
 * (synchronised) every stream that used it.  NULL is accepted. */
FLUX_ATTN_API int flux_attn_destroy(flux_attn_t h);

/* The whole hot path: QK-RMSNorm + RoPE prologue (and, in FP8 mode, the amax
 * and quantisation passes) followed by the joint attention kernel.
 *   q, k, v       bf16 [B, N, H, 128]
 *   geometry      txt_len, img_h, img_w, ref_h, ref_w >= 0; N = txt + img_h*img_w + ref_h*ref_w,
 *                 1 <= N <= max_tokens (N == 0 is accepted and does nothing)
 *   pos_ids       int32 [N, 3] position ids, or NULL: then text tokens get (0,0,0), image token
 *                 (r, c) gets (0, r, c) and reference token (r, c) gets (1, r, c)
 *   q_norm_w, k_norm_w  fp32 [128] RMSNorm weights (shared by all heads)
 *   out           bf16 [B, N, H, 128]; must not alias q, k or v */
FLUX_ATTN_API int flux_attn_forward(flux_attn_t h, const void* q, const void* k, const void* v,
                      int txt_len, int img_h, int img_w, int ref_h, int ref_w,
                      const int32_t* pos_ids, const float* q_norm_w, const float* k_norm_w,
                      void* out, cudaStream_t stream);

/* Prologue step alone (BF16 handles): writes the normalised, rotated Q' and K'
 * in head-major layout, bf16 [B, H, N, 128], into the caller's qn and kn.
 * Same argument rules as flux_attn_forward. */
FLUX_ATTN_API int flux_attn_prologue(flux_attn_t h, const void* q, const void* k,
                       int txt_len, int img_h, int img_w, int ref_h, int ref_w,
                       const int32_t* pos_ids, const float* q_norm_w, const float* k_norm_w,
                       void* qn, void* kn, cudaStream_t stream);

/* Attention step alone (BF16 handles): out = softmax(qn kn^T / sqrt(128)) v for
 *   qn, kn  bf16 [B, H, N, 128] (as written by flux_attn_prologue)
 *   v       bf16 [B, N, H, 128]
 *   out     bf16 [B, N, H, 128]
 * with 1 <= n_tokens <= max_tokens (0 does nothing). */
FLUX_ATTN_API int flux_attn_attend(flux_attn_t h, const void* qn, const void* kn, const void* v, int n_tokens,
                     void* out, cudaStream_t stream);

/* Prologue step alone (FP8 handles): per (b, h), amax of Q', K' and V, then
 * E4M3 codes (round to nearest even, saturating at 448) of x / scale with
 * scale = amax / 448 (1 when amax == 0).  V's codes are those of the exact
 * quotient, ties included; Q', K' are computed in fp32, so a value within fp32
 * rounding of a midpoint between two codes may take the neighbouring code.
 *   q8, k8  uint8 [B, H, N, 128];  v8t  uint8 [B, H, 128, Npad] (V transposed,
 *   Npad = N rounded up to a multiple of 16, padding columns zero; within
 *   every 8 columns, 8g .. 8g+7, the tokens 8g + 0, 2, 4, 6, 1, 3, 5, 7: the
 *   key order of flux_attn_attend_fp8's P.V MMA)
 *   scales  fp32 [B, H, 3] = (scale_q, scale_k, scale_v) */
FLUX_ATTN_API int flux_attn_prologue_fp8(flux_attn_t h, const void* q, const void* k, const void* v,
                           int txt_len, int img_h, int img_w, int ref_h, int ref_w,
                           const int32_t* pos_ids, const float* q_norm_w, const float* k_norm_w,
                           void* q8, void* k8, void* v8t, float* scales, cudaStream_t stream);

/* Attention step alone (FP8 handles) on the outputs of flux_attn_prologue_fp8;
 * out bf16 [B, N, H, 128]. */
FLUX_ATTN_API int flux_attn_attend_fp8(flux_attn_t h, const void* q8, const void* k8, const void* v8t,
                         const float* scales, int n_tokens, void* out, cudaStream_t stream);

/* VC-Attention FP8 ("Speed up image generation with FLUX 3 Image Klein on
 * NVIDIA Blackwell GPUs", section "Quantized and sparse attention":
 * vc_attention with a repair budget), step by step, for handles whose
 * vc_repair_budget gives R = ceil(rho N) > 0 repaired tokens
 * (flux_attn_forward runs both steps on such a handle; the plain FP8 steps
 * reject it).  R for n_tokens: flux_attn_vc_repair_count.
 *
 * flux_attn_prologue_fp8_vc: the FP8 prologue (codes and scales as for
 * flux_attn_prologue_fp8), then per (b, h) the R tokens of largest
 * |k' - deq(k')|^2 + |v - deq(v)|^2 (computed in fp32 from the kernel's own
 * K' and codes; equal errors: lower index first):
 *   repair_idx  int32 [B, H, R]: the repaired tokens, ascending
 *   k8, v8t     the codes of the N - R other tokens sit in positions
 *               0 .. N-R-1 (v8t in the 8-column order of
 *               flux_attn_prologue_fp8, by position)
 *               (a repaired token's position below N - R receives,
 *               in order, the codes of a non-repaired token from the last R
 *               positions); positions N-R .. N-1 are not read afterwards
 *   k_rep, v_rep  bf16 [B, H, R, 128]: k' / s_k and v / s_v of the repaired
 *               tokens, in repair_idx order (the units of the codes)
 * flux_attn_attend_fp8_vc: the attention over the outputs of the above:
 * every query attends to the R repaired keys with their exact values and to
 * the N - R others through their codes; out bf16 [B, N, H, 128]. */
FLUX_ATTN_API int flux_attn_prologue_fp8_vc(flux_attn_t h, const void* q, const void* k, const void* v,
                              int txt_len, int img_h, int img_w, int ref_h, int ref_w,
                              const int32_t* pos_ids, const float* q_norm_w, const float* k_norm_w,
                              void* q8, void* k8, void* v8t, float* scales, int32_t* repair_idx,
                              void* k_rep, void* v_rep, cudaStream_t stream);

FLUX_ATTN_API int flux_attn_attend_fp8_vc(flux_attn_t h, const void* q8, const void* k8, const void* v8t,
                            const float* scales, const void* k_rep, const void* v_rep, int n_tokens,
                            void* out, cudaStream_t stream);

/* R = ceil(vc_repair_budget * n_tokens) of the handle (0 for BF16 handles or a zero budget). */
FLUX_ATTN_API int flux_attn_vc_repair_count(flux_attn_t h, int n_tokens);

/* Sol-Attention ("Speed up image generation with FLUX 3 Image Klein on NVIDIA
 * Blackwell GPUs", section "Quantized and sparse attention": block-sparse
 * attention, algorithm sol_attn with tau and disabled_until_timestep), BF16
 * handles with sol_tau > 0 and max_tokens <= 262144.  nb = ceil(N / 128).
 *
 * flux_attn_forward_sol: as flux_attn_forward (same arguments, plus the
 * denoising timestep), dense when timestep > sol_disabled_until_timestep,
 * otherwise every query attends only to the keys of the blocks its query
 * block keeps (the mask of sol_tau, computed on the device from this call's
 * Q', K' in fp32).
 * flux_attn_sol_mask: the mask alone, for Q', K' bf16 [B, H, N, 128] as
 * written by flux_attn_prologue:  keep  uint8 [B, H, nb, nb], 1 = query block
 * i keeps key block j.
 * flux_attn_attend_sol: the block-sparse attention for Q', K' (as above), v
 * bf16 [B, N, H, 128] and any mask keep [B, H, nb, nb] in which every query
 * block keeps at least one block; out bf16 [B, N, H, 128]. */
FLUX_ATTN_API int flux_attn_forward_sol(flux_attn_t h, const void* q, const void* k, const void* v,
                          int txt_len, int img_h, int img_w, int ref_h, int ref_w,
                          const int32_t* pos_ids, const float* q_norm_w, const float* k_norm_w,
                          float timestep, void* out, cudaStream_t stream);

FLUX_ATTN_API int flux_attn_sol_mask(flux_attn_t h, const void* qn, const void* kn, int n_tokens,
                       uint8_t* keep, cudaStream_t stream);

FLUX_ATTN_API int flux_attn_attend_sol(flux_attn_t h, const void* qn, const void* kn, const void* v,
                         const uint8_t* keep, int n_tokens, void* out, cudaStream_t stream);

/* QKV projection with the query/key normalisation and RoPE fused into the
 * GEMM epilogue ("Speed up image generation with FLUX 3 Image Klein on
 * NVIDIA Blackwell GPUs", section "GEMM kernel optimisation"), BF16 handles:
 *   y = x W^T (+ b),  y = [Q | K | V] with head h of each part owning features
 *   h*128 .. h*128+127;  qn = RoPE(RMSNorm(Q) w_q), kn = RoPE(RMSNorm(K) w_k)
 *   x       bf16 [B, N, d_model], token-major (row b*N + n)
 *   w_qkv   bf16 [3 H 128, d_model] (a linear layer's [out, in] layout)
 *   b_qkv   fp32 [3 H 128], or NULL for no bias
 *   d_model a multiple of 64 in [64, 65536]
 *   geometry, pos_ids, q_norm_w, k_norm_w: as for flux_attn_forward
 *   qn, kn  bf16 [B, H, N, 128] (the layout flux_attn_attend reads)
 *   v       bf16 [B, N, H, 128]
 * Outputs must not overlap each other or x.  FLUX_ATTN_ERR_UNSUPPORTED on FP8
 * handles (they take flux_attn_qkv_fp8) and for other d_model. */
FLUX_ATTN_API int flux_attn_qkv(flux_attn_t h, const void* x, const void* w_qkv, const float* b_qkv, int d_model,
                  int txt_len, int img_h, int img_w, int ref_h, int ref_w, const int32_t* pos_ids,
                  const float* q_norm_w, const float* k_norm_w, void* qn, void* kn, void* v, cudaStream_t stream);

/* QKV projection for FP8 handles (same section): the GEMM and its epilogue
 * as in flux_attn_qkv, written as bf16 to the handle's workspace while the
 * epilogue reduces the per-(b, h) |max| of the Q', K', V values it writes;
 * then one pass writes their E4M3 codes with scale = amax / 448, in the
 * layouts flux_attn_attend_fp8 reads:
 *   q8, k8  uint8 [B, H, N, 128];  v8t  uint8 [B, H, 128, pad16(N)] (columns in
 *   the order flux_attn_prologue_fp8 gives them);  scales  fp32 [B, H, 3]
 * The codes are those of the bf16 values (rounded once more than the codes of
 * flux_attn_prologue_fp8, which quantises its fp32 Q', K').  Other arguments
 * as for flux_attn_qkv; UNSUPPORTED for handles with vc_repair_budget > 0. */
FLUX_ATTN_API int flux_attn_qkv_fp8(flux_attn_t h, const void* x, const void* w_qkv, const float* b_qkv,
                      int d_model, int txt_len, int img_h, int img_w, int ref_h, int ref_w,
                      const int32_t* pos_ids, const float* q_norm_w, const float* k_norm_w, void* q8, void* k8,
                      void* v8t, float* scales, cudaStream_t stream);

/* The front half of a FLUX-style block in one call: the QKV projection with
 * its fused QK-norm + RoPE epilogue (flux_attn_qkv; FP8 handles:
 * flux_attn_qkv_fp8), written to the handle's workspace, then the joint
 * attention over it (BF16 or FP8 as the handle's precision; not for handles
 * with vc_repair_budget > 0).
 *   x, w_qkv, b_qkv, d_model, geometry, pos_ids, norm weights: as for flux_attn_qkv
 *   out     bf16 [B, N, H, 128]; must not alias x */
FLUX_ATTN_API int flux_attn_forward_hidden(flux_attn_t h, const void* x, const void* w_qkv, const float* b_qkv,
                             int d_model, int txt_len, int img_h, int img_w, int ref_h, int ref_w,
                             const int32_t* pos_ids, const float* q_norm_w, const float* k_norm_w, void* out,
                             cudaStream_t stream);

/* Allocation-free forward (BF16).  The pages this library follows have no
 * counterpart to this call; it exists for callers that must not allocate
 * device memory while they run: engines that reserve and plan all device
 * memory once at start-up and forbid any later cudaMalloc, plugin hosts that
 * hand a plugin only the buffers it declared, and latency-critical callers
 * that cannot take the implicit device-wide synchronisation cudaMalloc and
 * cudaFree may cause.
 *
 * It computes exactly what flux_attn_forward computes, with the same kernels,
 * but needs no handle and allocates nothing: its Q'/K' scratch and its
 * device error word live in one file-scope device array of 16 MiB + 256 B
 * that the library's CUDA module holds on every device that loads it, until
 * the process exits.
 *   cfg           as for flux_attn_create; precision must be FLUX_ATTN_BF16
 *   q, k, v, out, geometry, pos_ids, norm weights, stream: as for flux_attn_forward
 *   device_error  optional device uint32: after the kernels it receives the
 *                 call's device error word (0 when every bounded wait was
 *                 satisfied, nonzero when one ran out); NULL to skip.
 * Limits: batch * num_heads * N <= 32768 (FLUX_ATTN_ERR_INVALID_ARG beyond).
 * Every call shares the one scratch array and the error word is cleared at
 * the start of each call; calls that overlap on the GPU (other streams,
 * other host threads) race on it, so serialise them per device.  The first
 * call on a device does a one-time set-up (it looks up the array's device
 * address and sets the attention kernel's shared-memory limit); make that
 * first call before any stream capture. */
FLUX_ATTN_API int flux_attn_forward_noalloc(const flux_attn_config* cfg, const void* q, const void* k,
                                            const void* v, int txt_len, int img_h, int img_w, int ref_h,
                                            int ref_w, const int32_t* pos_ids, const float* q_norm_w,
                                            const float* k_norm_w, void* out, uint32_t* device_error,
                                            cudaStream_t stream);

/* Synchronise `stream`, then read and clear the handle's device error word.
 * Returns FLUX_ATTN_OK, FLUX_ATTN_ERR_DEVICE_TIMEOUT or FLUX_ATTN_ERR_CUDA. */
FLUX_ATTN_API int flux_attn_sync_status(flux_attn_t h, cudaStream_t stream);

/* Bytes of device workspace the handle holds. */
FLUX_ATTN_API size_t flux_attn_workspace_bytes(flux_attn_t h);

/* Kernel launches one flux_attn_forward call makes for n_tokens tokens. */
FLUX_ATTN_API int flux_attn_launches_per_forward(flux_attn_t h, int n_tokens);

/* Static description of a status code. */
FLUX_ATTN_API const char* flux_attn_status_string(int status);

/* Description of the last failure in the calling thread ("" if none). */
FLUX_ATTN_API const char* flux_attn_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FLUX_ATTN_H */
