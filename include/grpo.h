/*
 * grpo.h - C ABI of the GB300 (sm_103a) memory-efficient GRPO loss library.
 *
 * The library computes the "linear" GRPO loss of the Unsloth GRPO blog
 * (zjt100.com translation, "Unsloth 高效 GRPO 算法" and "GRPO 的数学和发现的问题"):
 * the lm_head projection, the log-softmax and the GRPO objective fused over
 * the flattened (generations x completion length) token axis, without ever
 * forming the [N, V] logits. The backward pass recomputes the logit tiles
 * (Unsloth "grpo-long-context" page, offloaded log-softmax section) and
 * walks the token axis in chunks (same page, flattened sequence chunking,
 * Equation 3).
 *
 * Notation. B = num_seqs sequences of seq_len = T tokens; row n = b*T + t
 * (the G generations of a prompt are contiguous sequences). N = B*T rows, d
 * = hidden size, V = vocab. H_pol / H_ref are the policy / frozen reference
 * hidden states [N, d]; W is the lm_head weight [V, d] (logits = H W^T);
 * ids[n] is the token scored at row n (the caller has already shifted);
 * mask[n] in {0,1}; cnt_b = sum_t mask[b*T+t];
 * w_n = mask[n] / (B * max(cnt_b, 1)).
 * q_n = log softmax(H_pol[n] W^T)[ids[n]], p_n likewise from H_ref,
 * x_n = p_n - q_n, KL_n = exp(x_n) - x_n - 1 (reverse-KL estimator).
 * loss = sum_n w_n * (-(A_b - beta * KL_n)), the value of
 * exp(q - q.detach()) * A being 1.
 *
 * Conventions shared by every call:
 *  - Every tensor argument is a DEVICE pointer owned by the caller,
 *    row-major and contiguous, 16-byte aligned. The library never
 *    allocates device memory; scratch space is the caller's workspace.
 *  - Calls are asynchronous on `stream`; nothing synchronises except
 *    grpo_get_device_status and grpo_profile_collect. A workspace must not
 *    be shared by calls that may run concurrently.
 *  - The return value reports host-detectable errors, found before any
 *    launch (bad sizes, null pointers, short workspace). Errors found on the
 *    device (a valid token with an id outside [0, V), a pipeline wait that
 *    timed out) are recorded in the workspace's error word and read by
 *    grpo_get_device_status; the outputs of that call are then unspecified.
 *  - Outputs are overwritten, never accumulated.
 */
#ifndef GRPO_H
#define GRPO_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same definition as the CUDA runtime's stream handle. */
typedef struct CUstream_st *cudaStream_t;

typedef enum grpo_status {
  GRPO_OK = 0,
  GRPO_ERR_INVALID_ARG = 1,  /* null pointer, inconsistent sizes, bad group */
  GRPO_ERR_UNSUPPORTED = 2,  /* a layout the kernels do not handle (d % 8 != 0) */
  GRPO_ERR_WORKSPACE = 3,    /* workspace null, misaligned or too small */
  GRPO_ERR_CUDA = 4,         /* a CUDA runtime call failed */
  GRPO_ERR_TIMEOUT = 5,      /* device: a bounded pipeline wait expired */
  GRPO_ERR_BAD_TOKEN = 6     /* device: a valid token id outside [0, V) */
} grpo_status;

/* Element type of H_pol, H_ref, W and dH. GRPO_F32 inputs are rounded to
 * bf16 for the tensor-core products; accumulation is float32 either way.
 * GRPO_E4M3 problems take FP8 operands with row scales and are run by
 * grpo_loss_fwd_e4m3 / grpo_loss_bwd_e4m3 (their dH is bf16). */
typedef enum grpo_dtype { GRPO_F32 = 0, GRPO_BF16 = 1, GRPO_E4M3 = 2 } grpo_dtype;

typedef struct grpo_problem {
  int64_t N;            /* rows = num_seqs * seq_len */
  int64_t d;            /* hidden size, multiple of 8 (of 16 for GRPO_E4M3) */
  int64_t V;            /* vocab size */
  int32_t num_seqs;     /* B */
  int32_t seq_len;      /* T */
  int32_t group_size;   /* G generations per prompt (divides B) */
  float beta;           /* KL weight, the pages use 0.04 */
  float eps;            /* advantage denominator guard, e.g. 1e-4 */
  int32_t std_unbiased; /* 1: group std with Bessel's correction, 0: without */
  int64_t chunk_rows;   /* backward token chunk; 0 = chosen from a 4 GiB dZ budget */
  int32_t compute_dW;   /* 1: grpo_loss_bwd also writes dW (the lm_head gradient) */
  grpo_dtype dtype;
  /* Optional variants; a zero-initialised field keeps the default. */
  int32_t token_level;  /* 1: loss = sum_n m_n l_n / sum_n m_n (token-level mean)
                           instead of the per-sequence mean averaged over B */
  float logit_multiply; /* logit transforms, applied in this order before the
                           log-softmax (Unsloth "grpo-long-context" page: the
                           chunked selective log-softmax takes logit scale,
                           softcapping and temperature): z *= logit_multiply */
  float logit_divide;   /*   z /= logit_divide                (0 = off)      */
  float softcap;        /*   z = softcap * tanh(z / softcap)  (0 = off)      */
  float temperature;    /*   z /= temperature                 (0 = off)      */
  int32_t ref_logp_given; /* 1: grpo_loss_fwd reads the reference log-probs
                             from logp_ref instead of computing them; H_ref
                             is not used and may be NULL */
  int32_t kl_mode;      /* KL term, after the four experiments of the
                           zjt100.com page ("GRPO 的数学和发现的问题"), whose
                           formulas are lost (x = p - q):
                           0: exp(x) - x - 1 (reference implementation);
                           1: the same value, the advantage term without its
                              detach (exp(q - q) * A: no gradient);
                           2: exp(q) * (exp(x) - x - 1) (the extra Q factor);
                           3: x exp(x) - exp(x) + 1 (forward KL under Q) */
  int32_t cluster_mode; /* GEMM tiling, when the column tile is at least 128
                           wide: 0 one CTA per 128-row tile (default);
                           1 CTA pairs on tcgen05 cta_group::2 (256-row tiles,
                           half of each B tile per CTA). On a power-capped
                           GB300 step mode 1 settled ~16% lower in clock and
                           ran ~8% slower than mode 0. Any other value:
                           GRPO_ERR_UNSUPPORTED if positive, INVALID_ARG if
                           negative. */
} grpo_problem;

/*
 * Workspace bytes needed by grpo_loss_fwd and grpo_loss_bwd for `problem`
 * on the current device (the chunk plan depends on its SM count).
 * Either output pointer may be NULL.
 */
grpo_status grpo_workspace_size(const grpo_problem *problem, size_t *fwd_bytes,
                                size_t *bwd_bytes);

/*
 * The backward's chunk plan over the flattened (sequences x tokens) axis
 * (Unsloth "grpo-long-context" page, flattened sequence chunking, Equations
 * 1-3: only one chunk's logits exist at a time). The pages set the number of
 * chunks by a multiplier; here the size of the bf16 dZ chunk sets it. With
 * chunk_rows = 0 the chunk is the largest number of 128-row blocks whose
 * dZ (blocks * 128 rows * ldv columns * 2 bytes, ldv = V rounded up to a
 * multiple of 8) fits GRPO_DEFAULT_DZ_BUDGET_BYTES, rounded down to a
 * multiple of SMs / gcd(SMs, dH column tiles) blocks when that many fit, so
 * each chunk's dH GEMM fills whole waves of the device's SMs; when fewer fit,
 * the count between 3/4 of that largest one and the largest whose dH tiles
 * fill their last wave best (ties to the larger). Otherwise it is chunk_rows
 * rounded up to a multiple of 128; never more than the problem's blocks.
 *   chunk_rows      rows per chunk (a multiple of 128)
 *   n_chunks        chunks the backward launches (ceil of blocks / chunk)
 *   dz_chunk_bytes  bytes of the dZ chunk buffer in the backward workspace
 * Any output pointer may be NULL. Host-only apart from reading the current
 * device's SM count.
 */
#define GRPO_DEFAULT_DZ_BUDGET_BYTES ((size_t)4 << 30)
grpo_status grpo_chunk_plan(const grpo_problem *problem, int64_t *chunk_rows, int32_t *n_chunks,
                            size_t *dz_chunk_bytes);

/*
 * Group-relative advantages (aibit.im GRPO blog, GRPO section: several
 * answers per prompt are scored and an advantage is derived from the rewards
 * statistically; zjt100.com page, "GRPO 的数学和发现的问题": A is the
 * advantage after all reward functions). For each group of group_size
 * contiguous entries: A_b = (r_b - mean) / (std + eps), std with ddof 1 if
 * std_unbiased else 0; mean and std are formed in float64.
 *   rewards  device float32 [num_seqs], read only
 *   adv      device float32 [num_seqs], written
 * INVALID_ARG if num_seqs < 1, group_size < 1, group_size does not divide
 * num_seqs, or std_unbiased with group_size < 2.
 */
grpo_status grpo_advantages(const float *rewards, int32_t num_seqs, int32_t group_size,
                            float eps, int32_t std_unbiased, float *adv,
                            cudaStream_t stream);

/*
 * Forward pass of the fused loss (zjt100.com page, "Unsloth 高效 GRPO 算法":
 * a linear-cross-entropy style kernel adapted to GRPO; "GRPO 的数学和发现的问题":
 * reverse KL, beta, the exp(q - q.detach()) * A term, the logsumexp trick;
 * Unsloth "grpo-long-context" page: chunk logits kept in float32).
 * Policy and reference rows share each W tile; per row an online
 * max / sum-exp over vocab tiles gives the logsumexp, and the target logit
 * is gathered in the same pass.
 *   H_pol, H_ref  [N, d] dtype   W [V, d] dtype   ids int32 [N]
 *   mask uint8 [N] (0 or non-zero)                adv float32 [B]
 *   logp_pol, logp_ref  float32 [N]  written; 0 at masked rows (with
 *                                    ref_logp_given, logp_ref is read, not
 *                                    written)
 *   lse_pol             float32 [N]  written; the policy logsumexp, needed by
 *                                    grpo_loss_bwd; unspecified at masked rows
 *   loss                float32 [1]  written
 *   kl_mean             float32 [1]  written (sum mask*KL / sum mask, 0 if no
 *                                    valid row); may be NULL
 * Masked rows may carry any id; valid rows need 0 <= id < V (else
 * GRPO_ERR_BAD_TOKEN on the device).
 */
grpo_status grpo_loss_fwd(const grpo_problem *problem, const void *H_pol, const void *H_ref,
                          const void *W, const int32_t *ids, const uint8_t *mask,
                          const float *adv, float *logp_pol, float *logp_ref, float *lse_pol,
                          float *loss, float *kl_mean, void *workspace, size_t workspace_bytes,
                          cudaStream_t stream);

/*
 * Backward pass: gradient of `loss` scaled by grad_loss with respect to
 * H_pol (the reference model is frozen; Unsloth "grpo-long-context" page,
 * offloaded log-softmax: the backward recomputes the chunked log-softmax).
 * With c_n = grad_loss * w_n * (A_b + beta * (exp(x_n) - 1)) the logit
 * gradient is dZ_n = c_n * (softmax(z_n) - onehot(ids_n)) and dH = dZ W.
 * The logits are recomputed tile by tile for chunks of rows; dZ lives only
 * as a bf16 chunk in the workspace. With compute_dW the same chunk also
 * feeds dW = sum over chunks of dZ^T H_pol (a full fine-tune trains the
 * lm_head; LoRA and QLoRA runs freeze it, hence optional).
 *   logp_pol, logp_ref, lse_pol  the outputs of grpo_loss_fwd on the same
 *                                inputs
 *   dH      [N, d] dtype, written; rows of masked tokens are 0
 *   dW      float32 [V, d], written (accumulated in float32 over chunks in a
 *           fixed order), required when compute_dW = 1 and NULL otherwise
 *           (else GRPO_ERR_INVALID_ARG)
 */
grpo_status grpo_loss_bwd(const grpo_problem *problem, const void *H_pol, const void *W,
                          const int32_t *ids, const uint8_t *mask, const float *adv,
                          const float *logp_pol, const float *logp_ref, const float *lse_pol,
                          float grad_loss, void *dH, float *dW, void *workspace,
                          size_t workspace_bytes, cudaStream_t stream);

/*
 * Forward pass without a workspace, for callers that cannot allocate device
 * memory: hosts with no allocator of their own, for which cudaMalloc would
 * synchronise the device, and code running under a memory budget that is
 * fixed once training starts. This entry point has no counterpart in the
 * pages; it computes exactly what grpo_loss_fwd computes, with the same
 * arguments minus the workspace.
 *
 * Scratch lives in a static device array of GRPO_NOALLOC_SCRATCH_BYTES that
 * every GPU loading the library holds until the process exits. Its device
 * address is looked up on the first call on each device (with that device
 * current), so make that first call before any stream capture. The address
 * belongs to that device's context: do not use this entry point across a
 * cudaDeviceReset or any other teardown of the context. The call itself
 * never allocates (no cudaMalloc or cudaFree).
 *
 * Every call on a device shares the one array, and the array keeps the last
 * call's contents: calls that may overlap on the GPU (different streams, or
 * different host threads) race and must not be issued. Returns
 * GRPO_ERR_WORKSPACE, before any launch, when the problem needs more scratch
 * than the array holds. The need is grpo_workspace_size's forward bytes on
 * the device the call runs on: query it there and compare it with
 * GRPO_NOALLOC_SCRATCH_BYTES, since it depends on the device's SM count.
 * For bf16 inputs it is about 8 + 16 * S * h bytes per token with S = 1..8
 * vocab slices and h = 2 when d <= 1024, else 1 (e.g. 72 bytes on the
 * Llama-8B head on a 152-SM GPU, so a few hundred thousand tokens fit);
 * float32 inputs also need bf16 copies of H_pol, H_ref and W.
 * A device-detected error (a valid token id outside [0, V), an expired
 * pipeline wait) makes *loss and *kl_mean NaN, since there is no workspace
 * to query; the per-token outputs are then undefined.
 */
#define GRPO_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
grpo_status grpo_loss_fwd_noalloc(const grpo_problem *problem, const void *H_pol,
                                  const void *H_ref, const void *W, const int32_t *ids,
                                  const uint8_t *mask, const float *adv, float *logp_pol,
                                  float *logp_ref, float *lse_pol, float *loss, float *kl_mean,
                                  cudaStream_t stream);

/*
 * FP8 operands. The pages name Float8 training only as a feature that
 * combines with the long-context loss (Unsloth "grpo-long-context" page, the
 * hint listing the features that combine, item 3) and fix no format, so the
 * format is OCP FP8 E4M3 (the "fn" flavour: no infinities, codes 0x7F and
 * 0xFF are NaN, largest finite value 448) with one float32 scale per row:
 * row r of an operand stands for s[r] * decode(q[r][:]). An e4m3 problem
 * (problem->dtype = GRPO_E4M3) is the loss above evaluated on the
 * dequantized H_pol, H_ref and W; dH and dW are its gradients with respect
 * to the dequantized H_pol and W. The three products H W^T (reference and
 * policy forward, backward recompute) run on e4m3 tensor-core operands with
 * float32 accumulation, the row scales applied to the accumulator; the
 * dH = dZ W and dW = dZ^T H products take bf16 roundings of the dequantized
 * W and H_pol, since dZ keeps bf16.
 *
 * grpo_quantize_e4m3_rows turns float32 or bf16 rows into such operands, per
 * row in float32 arithmetic: amax = max |x|, scale = amax / 448,
 * q = e4m3(x * (448 / amax)) rounded to nearest even and saturated to
 * +-448 (divisions and the product correctly rounded); a row of zeros gets
 * scale 1 and zero codes.
 *   x      device [rows, cols] of x_dtype (GRPO_F32 or GRPO_BF16), read only
 *   q      device uint8 [rows, cols], written
 *   scale  device float32 [rows], written
 * INVALID_ARG for null pointers, rows < 0, cols < 1 or another x_dtype;
 * UNSUPPORTED unless cols % 16 == 0 and x, q, scale are 16-byte aligned.
 * rows = 0 launches nothing. x must be finite: a row holding an infinity or
 * a NaN gets unspecified codes and scale (no error is reported).
 */
grpo_status grpo_quantize_e4m3_rows(const void *x, grpo_dtype x_dtype, int64_t rows,
                                    int64_t cols, uint8_t *q, float *scale,
                                    cudaStream_t stream);

/*
 * grpo_loss_fwd for an e4m3 problem (problem->dtype = GRPO_E4M3, d % 16 == 0):
 *   H_pol, H_ref  uint8 e4m3 [N, d] with s_pol, s_ref float32 [N]
 *   W             uint8 e4m3 [V, d] with s_W float32 [V]
 * every other argument and output as in grpo_loss_fwd (with ref_logp_given,
 * H_ref and s_ref are not read and may be NULL). The scales must be finite
 * (they are used as given; the NaN codes 0x7F and 0xFF propagate as NaN).
 * s_W must be 16-byte aligned (UNSUPPORTED otherwise). The workspace is sized by
 * grpo_workspace_size on the same problem. grpo_loss_fwd and grpo_loss_bwd
 * reject e4m3 problems (INVALID_ARG), and these two reject the others.
 */
grpo_status grpo_loss_fwd_e4m3(const grpo_problem *problem, const uint8_t *H_pol,
                               const float *s_pol, const uint8_t *H_ref, const float *s_ref,
                               const uint8_t *W, const float *s_W, const int32_t *ids,
                               const uint8_t *mask, const float *adv, float *logp_pol,
                               float *logp_ref, float *lse_pol, float *loss, float *kl_mean,
                               void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * grpo_loss_bwd for an e4m3 problem: the operands as in grpo_loss_fwd_e4m3,
 * dH bf16 [N, d] (the gradient with respect to the dequantized H_pol; rows
 * of masked tokens are 0), dW float32 [V, d] or NULL as in grpo_loss_bwd.
 */
grpo_status grpo_loss_bwd_e4m3(const grpo_problem *problem, const uint8_t *H_pol,
                               const float *s_pol, const uint8_t *W, const float *s_W,
                               const int32_t *ids, const uint8_t *mask, const float *adv,
                               const float *logp_pol, const float *logp_ref,
                               const float *lse_pol, float grad_loss, void *dH, float *dW,
                               void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Synchronises `stream`, reads and clears the error word of a workspace
 * used by grpo_loss_fwd or grpo_loss_bwd, and returns GRPO_OK,
 * GRPO_ERR_TIMEOUT or GRPO_ERR_BAD_TOKEN (timeout wins if both occurred).
 */
grpo_status grpo_get_device_status(void *workspace, cudaStream_t stream);

/* Human-readable name of a status code (static string). */
const char *grpo_status_string(grpo_status status);

/*
 * Kernel timing, for benchmarks. While enabled, every kernel the library
 * launches is bracketed by CUDA events recorded on its launching stream.
 * grpo_profile_collect synchronises on those events and returns, for each
 * kernel kind k < n_kinds, the summed milliseconds and the launch count
 * since the last collect (then clears them). Kinds are numbered 0 ..
 * grpo_profile_kind_count()-1 and named by grpo_profile_kind_name.
 * Not thread-safe; at most 65536 launches between collects.
 */
grpo_status grpo_profile_enable(int32_t on);
grpo_status grpo_profile_collect(double *ms, int64_t *launches, int32_t n_kinds);
int32_t grpo_profile_kind_count(void);
const char *grpo_profile_kind_name(int32_t kind);

/*
 * Testing hook for the device-side failure path. With on = 1, the next
 * forward GEMM launches withhold the first shared-memory stage of CTA 0, so
 * that CTA's MMA wait expires: the kernel records GRPO_ERR_TIMEOUT in the
 * workspace's error word, drains its copies, frees tensor memory and
 * returns, and the context stays usable. wait_ms sets the pipeline wait
 * limit of every kernel launched afterwards (0 restores the default of 4 s).
 * Call with on = 0, wait_ms = 0 to restore normal operation. Not thread-safe.
 */
grpo_status grpo_test_pipeline_stall(int32_t on, uint32_t wait_ms);

#ifdef __cplusplus
}
#endif

#endif /* GRPO_H */
