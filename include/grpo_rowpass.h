/*
 * grpo_rowpass.h -- C ABI of the GB300 (sm_103a) row pass over LM-head logits.
 *
 * One row r = one token (b, l) of a [B, L, V] logits tensor, r = b*L + l.  With
 * z_j = x_j / T (T the sampling temperature):
 *
 *   lse_r   = log sum_j exp(z_j)
 *   logp_r  = z_idx - lse_r                  (selective log-softmax)
 *   H_r     = sum_j p_j (lse_r - z_j)        (entropy, p_j = exp(z_j - lse_r))
 *   ratio_r = exp(logp_r - old_logp_r)
 *   pg_r    = -min(ratio_r * A_b, clip(ratio_r, 1 - eps_low, 1 + eps_high) * A_b)
 *   kl_r    = beta * (exp(d_r) - d_r - 1),   d_r = ref_logp_r - logp_r
 *   loss_r  = (pg_r + kl_r) on unmasked tokens, +0.0 on masked ones
 *
 * and the backward  dlogits_rj = g_r * (1[j == idx_r] - p_j)  with one scalar g_r
 * per row.  A row whose g_r is exactly zero is stored as +0.0 and its logits are
 * never read.
 *
 * Sources (web pages the method is described on):
 *   [Liger-bwd]  "LinkedIn Liger-Kernel GRPO Loss Backward optimisation" (write-up of
 *                Liger-Kernel PR #1550), sections "Code analysis" and "Why it's good".
 *   [axolotl]    "Axolotl: entropy and selective log-softmax with Triton kernels"
 *                (write-up of axolotl PR #3510), sections "1. benchmarks/bench_entropy.py",
 *                "2. benchmarks/bench_selective_logsoftmax.py", "Why it's good".
 *   [Liger-TRL]  "Liger GRPO meets TRL", sections 2 and 4.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every pointer argument is a DEVICE pointer (cudaMalloc'd, or any memory the GPU
 *   can address) owned by the caller.  The library allocates nothing, keeps no state
 *   between calls, and launches its kernels asynchronously on `stream` (NULL = the
 *   legacy default stream).  Results are visible once the stream is synchronised.
 * - Per-row arrays ([B*L]) are contiguous, indexed by r = b*L + l.  Per-sequence
 *   arrays ([B]) are contiguous.  float arrays need 4-byte, int64 arrays 8-byte
 *   alignment.
 * - The logits are described by grpo_rows: element (b, l, j) lives at
 *   ptr + b*stride_b + l*stride_l + j (strides in ELEMENTS, vocab stride 1), so a
 *   non-contiguous view such as logits[:, :-1, :] of a [B, L+1, V] tensor is read in
 *   place, with no copy.  Rows may start at any element boundary; rows whose start is
 *   16-byte aligned take the fastest path.
 * - Return value: GRPO_OK, or an error found on the host BEFORE any launch
 *   (GRPO_ERR_INVALID_ARG / GRPO_ERR_UNSUPPORTED; nothing is written), or
 *   GRPO_ERR_CUDA when the launch itself failed (cudaGetLastError after the launch).
 *   B*L == 0 is valid and launches nothing; the data pointers (including the
 *   descriptors' ptr fields, but not the descriptors themselves) may then be NULL.
 * - `dev_err` (nullable) is a device int32 word the kernels OR error bits into
 *   (GRPO_DEVERR_*).  The library never clears it and never traps: a row with an
 *   out-of-range idx gets NaN in its idx-dependent outputs and the bit is set.
 * - NaN / Inf logits propagate to that row's outputs the way the definitions above
 *   propagate them; nothing faults.  Finite logits are supported up to |x / T| < 2^30;
 *   beyond that the fp32 exponent offset can overflow and a row may read Inf/NaN.
 *   The saved lse is fp32, so the backward's bf16 outputs are within 1 ulp of the
 *   exact result while |lse| < 2^15.
 */
#ifndef GRPO_ROWPASS_H_
#define GRPO_ROWPASS_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared without the CUDA headers. */
struct CUstream_st;
typedef struct CUstream_st* grpo_stream_t;

typedef enum {
  GRPO_OK = 0,
  GRPO_ERR_INVALID_ARG = 1, /* a null/misaligned pointer, bad size, stride, scalar or aliasing */
  GRPO_ERR_UNSUPPORTED = 2, /* valid arguments the library does not handle (e.g. B*L >= 2^31) */
  GRPO_ERR_CUDA = 3         /* the kernel launch failed */
} grpo_status;

typedef enum { GRPO_FP32 = 0, GRPO_BF16 = 1 } grpo_dtype;

/* Bits OR-ed into *dev_err by the kernels. */
#define GRPO_DEVERR_IDX_OUT_OF_RANGE 1
/* A kernel gave up waiting for its own asynchronous copies (about 2 s): a tensor-core GEMM of
 * grpo_fused_linear(_noalloc) (copies or MMAs), or a row of grpo_loss_fused (the bulk copy of
 * the part of the row kept in shared memory).  Those outputs are not valid.  The kernel
 * returns without trapping (the GEMM with its TMEM freed). */
#define GRPO_DEVERR_TIMEOUT 2

/* A [B, L, V] logits (or dlogits) tensor: ptr + b*stride_b + l*stride_l + j. */
typedef struct {
  void* ptr;         /* device pointer, aligned to the element size */
  int32_t dtype;     /* grpo_dtype */
  int32_t reserved;  /* must be 0 */
  int64_t B, L, V;   /* sequences, tokens per sequence, vocabulary (V >= 1) */
  int64_t stride_b;  /* elements between (b, l, 0) and (b+1, l, 0); >= 0 */
  int64_t stride_l;  /* elements between (b, l, 0) and (b, l+1, 0); >= 0 */
} grpo_rows;

/*
 * grpo_loss_fwd -- forward of the GRPO per-token loss, one pass over each unmasked row.
 *
 * Defined by: the clipped-ratio objective whose zero-gradient ("PPO-clipped") tokens
 * [Liger-bwd] "Why it's good" names, the k3 KL term whose gradient
 * beta*(1 - exp(ref_logp - logp)) [Liger-bwd] "Code analysis" prints, and the
 * temperature division of the same section; the entropy is the definition in
 * [axolotl] "1. benchmarks/bench_entropy.py".
 *
 *   logits      [B, L, V] bf16 or fp32 (read only)
 *   idx         [B*L] int64 sampled token per row; read only on unmasked rows
 *   old_logp    [B*L] fp32, or NULL meaning old_logp == logp (ratio 1)
 *   ref_logp    [B*L] fp32; may be NULL only when beta == 0 (then never read)
 *   adv         [B]   fp32 advantage per sequence
 *   mask        [B*L] uint8 completion mask (0 = padding), or NULL = every token counts
 *   T > 0 finite; beta >= 0 finite; 0 <= eps_low <= 1; eps_high >= 0 finite
 *   loss, logp, lse   [B*L] fp32 outputs (required); lse is what grpo_loss_bwd needs
 *   kl, entropy       [B*L] fp32 outputs, or NULL to skip
 *   is_clipped        [B*L] uint8 output (1 where the clipped branch is strictly the
 *                     smaller one, so the policy-gradient term has zero gradient), or NULL
 *   dev_err           nullable device int32 error word
 *
 * Masked rows write +0.0 to every output (0 to is_clipped) and read no logits.  With
 * beta == 0 the KL term is never evaluated (kl = +0.0).  An unmasked row whose idx is
 * outside [0, V) writes NaN to loss, logp and kl (lse and entropy stay valid) and sets
 * GRPO_DEVERR_IDX_OUT_OF_RANGE.
 */
grpo_status grpo_loss_fwd(const grpo_rows* logits, const int64_t* idx, const float* old_logp,
                          const float* ref_logp, const float* adv, const uint8_t* mask, float T,
                          float beta, float eps_low, float eps_high, float* loss, float* logp,
                          float* lse, float* kl, uint8_t* is_clipped, float* entropy, int32_t* dev_err,
                          grpo_stream_t stream);

/*
 * grpo_loss_bwd -- backward of sum_r dloss_r * loss_r with respect to the logits.
 *
 * Defined by [Liger-bwd] "Code analysis" (_grpo_loss_bwd_kernel): per row,
 * dlogp = dpg/dlogp + beta*(1 - exp(ref_logp - logp)), scaled by dloss and divided by
 * the temperature, then spread over the row as g * (1[j == idx] - p_j); when that
 * scaled dlogp is exactly 0.0 the row is filled with 0.0 and nothing else is done.
 * dpg/dlogp = -A * ratio where ratio*A <= clip(ratio)*A, else 0 (clipping binds).
 *
 *   logits, idx, old_logp, ref_logp, adv, mask, T, beta, eps_low, eps_high: as in
 *               grpo_loss_fwd (same values)
 *   dloss       [B*L] fp32 upstream gradient of each token's loss
 *   logp, lse   [B*L] fp32 as written by grpo_loss_fwd for the same inputs
 *   dlogits     [B, L, V] output, same dtype and B, L, V as logits, its own strides
 *               (rows must not overlap).  It may alias logits exactly (same ptr and
 *               strides) for an in-place backward; any other overlap is rejected.
 *
 * Rows where g == 0.0 (masked tokens; zero advantage or binding clip with beta == 0;
 * dloss == 0) are written as +0.0 without reading logits, idx or lse.  Other rows are
 * read once and written once; bf16 outputs are rounded to nearest even.  An idx
 * outside [0, V) on a row with g != 0 fills that row with NaN and sets the error bit.
 */
grpo_status grpo_loss_bwd(const grpo_rows* logits, const int64_t* idx, const float* old_logp,
                          const float* ref_logp, const float* adv, const uint8_t* mask,
                          const float* dloss, const float* logp, const float* lse, float T,
                          float beta, float eps_low, float eps_high, const grpo_rows* dlogits,
                          int32_t* dev_err, grpo_stream_t stream);

/*
 * grpo_loss_fused -- grpo_loss_fwd and grpo_loss_bwd in one kernel, for per-token loss
 * weights dloss that are known before the forward (a fixed normalisation such as
 * mask / (B * completion length)).
 *
 * Defined by "Liger GRPO meets TRL", section 4 ([Liger-TRL]: the loss computes the
 * gradients during its forward so the logits are not kept for a later backward), with the
 * forward and backward definitions of grpo_loss_fwd / grpo_loss_bwd above.  Each row is
 * read once for its statistic; the row factor g is decided from the row's own logp (the
 * value written to logp); a row with g == 0.0 is filled with +0.0, any other row is swept
 * again (the same CTA re-reads what it just read, mostly from L2) to write dlogits.
 *
 * Arguments: those of grpo_loss_fwd, plus dloss [B*L] fp32 and dlogits as in
 * grpo_loss_bwd (same dtype/B/L/V as logits; may alias logits exactly).  The outputs equal
 * those of grpo_loss_fwd followed by grpo_loss_bwd on the same inputs (dlogits to within
 * the rounding of the summation order of the idx element).
 */
grpo_status grpo_loss_fused(const grpo_rows* logits, const int64_t* idx, const float* old_logp,
                            const float* ref_logp, const float* adv, const uint8_t* mask, const float* dloss,
                            float T, float beta, float eps_low, float eps_high, float* loss, float* logp,
                            float* lse, float* kl, uint8_t* is_clipped, float* entropy,
                            const grpo_rows* dlogits, int32_t* dev_err, grpo_stream_t stream);

/*
 * entropy_from_logits -- H_r = sum_j p_j (lse_r - z_j) per row, one fused pass.
 *
 * Defined by [axolotl] "1. benchmarks/bench_entropy.py": the original takes
 * log_softmax of each row and sums -exp(logps)*logps; the fused kernel the same page
 * describes reads strided logits in place.  T = 1 reproduces the page's definition.
 *
 *   logits   [B, L, V] bf16 or fp32;  T > 0 finite;  entropy [B*L] fp32 output
 *   lse      [B*L] fp32 output, or NULL (needed by entropy_from_logits_bwd)
 * A logit of -inf has p = 0 and adds 0 (the limit of p log p).
 */
grpo_status entropy_from_logits(const grpo_rows* logits, float T, float* entropy, float* lse,
                                grpo_stream_t stream);

/*
 * entropy_from_logits_bwd -- gradient of sum_r dentropy_r * H_r with respect to the logits:
 *   dlogits_rj = -(dentropy_r / T) p_j (log p_j + H_r).
 *
 * The derivative of the entropy definition of [axolotl] "1. benchmarks/bench_entropy.py"
 * (the pages print no entropy backward).  A row whose dentropy_r / T is exactly 0.0 is
 * written as +0.0 without reading its logits (as in the other backward passes).
 *
 *   logits [B, L, V];  dentropy [B*L] fp32 upstream gradient of H
 *   lse, entropy [B*L] fp32 as written by entropy_from_logits (or grpo_loss_fwd) for the
 *   same logits and T;  dlogits as in grpo_loss_bwd (may alias logits exactly)
 */
grpo_status entropy_from_logits_bwd(const grpo_rows* logits, const float* dentropy, const float* lse,
                                    const float* entropy, float T, const grpo_rows* dlogits,
                                    grpo_stream_t stream);

/*
 * selective_log_softmax_fwd -- logp_r = log_softmax(x_r / T)[idx_r], and lse_r.
 *
 * Defined by [axolotl] "2. benchmarks/bench_selective_logsoftmax.py" (the log-softmax
 * evaluated only at the given index of each row).
 *
 *   logits [B, L, V];  idx [B*L] int64;  T > 0 finite
 *   logp, lse [B*L] fp32 outputs (lse feeds selective_log_softmax_bwd)
 * An idx outside [0, V) writes NaN to logp (lse stays valid) and sets the error bit.
 */
grpo_status selective_log_softmax_fwd(const grpo_rows* logits, const int64_t* idx, float T,
                                      float* logp, float* lse, int32_t* dev_err,
                                      grpo_stream_t stream);

/*
 * selective_log_softmax_bwd -- dlogits_rj = (dlogp_r / T) * (1[j == idx_r] - p_j).
 *
 * Defined by [axolotl] "2. benchmarks/bench_selective_logsoftmax.py" (the backward
 * kernel of the selective log-softmax), with the zero-row early-out of [Liger-bwd]
 * "Code analysis": a row whose dlogp_r / T is exactly 0.0 is written as +0.0 without
 * reading its logits.
 *
 *   logits [B, L, V];  idx [B*L] int64;  dlogp [B*L] fp32 upstream gradient of logp
 *   lse [B*L] fp32 from selective_log_softmax_fwd;  T as in the forward
 *   dlogits: as in grpo_loss_bwd (same dtype/B/L/V, may alias logits exactly)
 */
grpo_status selective_log_softmax_bwd(const grpo_rows* logits, const int64_t* idx,
                                      const float* dlogp, const float* lse, float T,
                                      const grpo_rows* dlogits, int32_t* dev_err,
                                      grpo_stream_t stream);

/*
 * grpo_seq_terms -- sequence-level GRPO: per-sequence importance ratio and objective, and
 * the per-token dlogp that selective_log_softmax_bwd turns into dlogits.
 *
 * [Liger-bwd] "Code analysis" shows a sequence-level backward kernel
 * (_grpo_loss_bwd_kernel_seq) whose token KL gradient beta*(1 - exp(ref_logp - logp)) is
 * weighted by the token's dloss while the policy-gradient part arrives computed per
 * sequence; its ratio is not printed.  The ratio taken here is the length-normalised
 * sequence ratio: for sequence b with n_b unmasked tokens,
 *   s_b = exp(sum_t m_t (logp_t - old_t) / n_b),   pg_b = -min(s_b A_b, clip(s_b) A_b),
 *   loss_t = pg_b + kl_t  (unmasked tokens; +0.0 on masked ones),
 *   dlogp_t = W_b * dpg_b/dlogp_t + beta (1 - exp(ref_t - logp_t)) * dloss_t,
 *   W_b = sum_t dloss_t,  dpg_b/dlogp_t = -A_b s_b / n_b, or 0 where clipping binds,
 * i.e. dlogp_t = dJ/dlogp_t for J = sum_t dloss_t loss_t.  The full pass is:
 *   selective_log_softmax_fwd (logp, lse) -> grpo_seq_terms -> selective_log_softmax_bwd
 *   (dlogits = (dlogp/T)(onehot - p), +0.0 rows where dlogp == 0 without reading logits).
 *
 *   B, L         sequences and tokens per sequence (per-row arrays are [B*L], r = b*L + l)
 *   logp         [B*L] fp32 (from selective_log_softmax_fwd);  old_logp: [B*L] or NULL (= logp)
 *   ref_logp     [B*L], may be NULL when beta == 0;  adv [B];  mask [B*L] or NULL
 *   dloss        [B*L] fp32 per-token loss weights
 *   loss, dlogp  [B*L] fp32 outputs;  kl [B*L] or NULL;  seq_ratio [B] fp32 or NULL;
 *   seq_is_clipped [B] uint8 or NULL.  A sequence with no unmasked token has ratio 1.
 */
grpo_status grpo_seq_terms(int64_t B, int64_t L, const float* logp, const float* old_logp,
                           const float* ref_logp, const float* adv, const uint8_t* mask, const float* dloss,
                           float beta, float eps_low, float eps_high, float* loss, float* kl, float* dlogp,
                           float* seq_ratio, uint8_t* seq_is_clipped, grpo_stream_t stream);

/*
 * Vocabulary-parallel form.  When the LM head is split over ranks by vocabulary (rank k
 * holds the columns [vocab_start_k, vocab_start_{k+1}) of every row), the row pass runs
 * per shard; the only exchange is one all-gather of a 4-float statistic per row:
 *
 *   1. grpo_vocab_shard_stats on each rank's shard         -> stats_k [B*L][4]
 *   2. all-gather of stats_k over the ranks (the caller's collective, rank order)
 *                                                          -> stats_all [world][B*L][4]
 *   3. grpo_vocab_combine on every rank (same result on each): lse, logp, entropy and
 *      the GRPO terms of the full rows, and p_rest for the backward
 *   4. grpo_loss_bwd_vocab_shard (or selective_log_softmax_bwd_vocab_shard) on each
 *      rank's shard -> that shard's columns of dlogits.  entropy_from_logits_bwd needs no
 *      variant: given the full rows' lse and H it is already column-local.
 *
 * The definitions are those of the unsplit entry points above (the pages shard nothing;
 * the split is exact algebra of the log-sum-exp).  A shard's statistic is, with
 * c = log2(e) / T and its own offset a (its maximum logit times c, rounded to fp32):
 *   a,  s = sum_j 2^(x_j c - a),  u = sum_j 2^(x_j c - a) (x_j c - a),
 *   x_sel = the raw logit at idx if idx falls in the shard, else 0.
 * Merged over the shards (largest offset A first): lse = ln2 A + ln S,
 * H = ln S - ln2 U / S, logp = ln2 (x_sel c - A) - ln S, as in the unsplit forward.
 */

/*
 * grpo_vocab_shard_stats -- the per-row statistic of one vocabulary shard.
 *
 *   logits_shard  [B, L, V_k] bf16 or fp32: columns [vocab_start, vocab_start + V_k)
 *                 of the full rows, any row strides (a column slice of the full tensor
 *                 is a valid view)
 *   vocab_start   >= 0, the shard's first column in the full vocabulary
 *   idx           [B*L] int64 sampled tokens (full-vocabulary indices), or NULL
 *   mask          [B*L] uint8 or NULL; masked rows are not read and get (0, 0, 0, 0)
 *   T             > 0 finite
 *   stats         [B*L][4] fp32 output (a, s, u, x_sel), 16-byte aligned
 */
grpo_status grpo_vocab_shard_stats(const grpo_rows* logits_shard, int64_t vocab_start, const int64_t* idx,
                                   const uint8_t* mask, float T, float* stats, grpo_stream_t stream);

/*
 * grpo_vocab_combine -- merge the gathered shard statistics into the full rows' forward
 * outputs.
 *
 *   world         1 <= world <= GRPO_VOCAB_MAX_WORLD shards
 *   stats_all     [world][B*L][4] fp32: shard k's grpo_vocab_shard_stats output at k
 *   vocab_starts  HOST array of world + 1 increasing int64: shard k holds columns
 *                 [vocab_starts[k], vocab_starts[k+1]); vocab_starts[0] = 0 and
 *                 vocab_starts[world] = V, the full vocabulary
 *   B, L          rows are r = b*L + l
 *   idx           [B*L] int64 or NULL.  NULL: entropy / lse only (logp, loss, p_rest NULL)
 *   lse           [B*L] fp32 output (required);  entropy: [B*L] fp32 output or NULL
 *   logp          [B*L] fp32 output (required when idx is given)
 *   p_rest        [B*L] fp32 output or NULL: the probability mass of the row outside the
 *                 shard that holds idx; the backward of that shard needs it
 *   loss          NULL: selective log-softmax only.  Otherwise the GRPO terms as in
 *                 grpo_loss_fwd, with old_logp, ref_logp, adv, mask, beta, eps_low,
 *                 eps_high, kl, is_clipped meaning what they mean there
 *   dev_err       nullable device int32 error word
 *
 * Masked rows (mask given and 0) write +0.0 to every output.  An idx outside [0, V) on
 * an unmasked row writes NaN to logp, loss, kl and p_rest and sets
 * GRPO_DEVERR_IDX_OUT_OF_RANGE.  The result is the same on every rank for the same
 * stats_all.
 */
#define GRPO_VOCAB_MAX_WORLD 64
grpo_status grpo_vocab_combine(int32_t world, const float* stats_all, const int64_t* vocab_starts, int64_t B,
                               int64_t L, const int64_t* idx, const float* old_logp, const float* ref_logp,
                               const float* adv, const uint8_t* mask, float T, float beta, float eps_low,
                               float eps_high, float* loss, float* logp, float* lse, float* kl,
                               uint8_t* is_clipped, float* entropy, float* p_rest, int32_t* dev_err,
                               grpo_stream_t stream);

/*
 * grpo_loss_bwd_vocab_shard -- grpo_loss_bwd on one vocabulary shard: the shard's
 * columns of dlogits_rj = g_r (1[j == idx_r] - p_j), with the same row factor g_r and the
 * same zero-row early-out.  The idx element, on the shard that holds it, is
 * g_r (1 - p_idx) = sign(g_r) |g_r| (sum of the shard's other p_j + p_rest_r).
 *
 *   logits_shard, vocab_start   as in grpo_vocab_shard_stats
 *   vocab_total                 V, the full vocabulary (idx must lie in [0, V))
 *   idx, old_logp, ref_logp, adv, mask, dloss, T, beta, eps_low, eps_high: as in
 *   grpo_loss_bwd;  logp, lse, p_rest [B*L] fp32 from grpo_vocab_combine
 *   dlogits_shard               [B, L, V_k] output, same dtype and shape as logits_shard
 *                               (may alias it exactly)
 */
grpo_status grpo_loss_bwd_vocab_shard(const grpo_rows* logits_shard, int64_t vocab_start, int64_t vocab_total,
                                      const int64_t* idx, const float* old_logp, const float* ref_logp,
                                      const float* adv, const uint8_t* mask, const float* dloss,
                                      const float* logp, const float* lse, const float* p_rest, float T,
                                      float beta, float eps_low, float eps_high, const grpo_rows* dlogits_shard,
                                      int32_t* dev_err, grpo_stream_t stream);

/*
 * selective_log_softmax_bwd_vocab_shard -- selective_log_softmax_bwd on one vocabulary
 * shard (g_r = dlogp_r / T), with lse and p_rest from grpo_vocab_combine; arguments as in
 * grpo_loss_bwd_vocab_shard.
 */
grpo_status selective_log_softmax_bwd_vocab_shard(const grpo_rows* logits_shard, int64_t vocab_start,
                                                  int64_t vocab_total, const int64_t* idx, const float* dlogp,
                                                  const float* lse, const float* p_rest, float T,
                                                  const grpo_rows* dlogits_shard, int32_t* dev_err,
                                                  grpo_stream_t stream);

/*
 * grpo_fused_linear -- the GRPO loss on top of the LM head, with the gradients of the
 * hidden states and of the head weight, in chunks of rows.
 *
 * Defined by [Liger-TRL] sections 3 and 4: the logits are the head applied to the hidden
 * states, x = h W^T; the loss of each chunk of rows computes, during its forward, the
 * gradient of its input chunk and of the head weight, the weight gradient accumulated over
 * the chunks, so the logits of the whole batch never exist at once.  Per chunk:
 *   x_c = h_c W^T (fp32, tensor-core GEMM)  ->  the row pass of grpo_loss_fused on x_c
 *   (forward outputs, dlogits in bf16)  ->  grad_hidden_c = dlogits_c W,
 *   grad_weight += dlogits_c^T h_c  (tensor-core GEMMs, fp32 accumulation).
 * All of it runs in this library's kernels: the GEMMs are tcgen05 kernels with TMA-staged
 * bf16 operands and fp32 accumulators in tensor memory.  The logits GEMM forms each row's
 * softmax statistic per 128 columns from its fp32 results, and stores, instead of the logits,
 * their exponentials relative to each 128-column maximum, e_j = exp((x_j - max) / T), in fp16
 * (scaled by 2^15, so that every e_j above 2^-29 keeps 11 significant bits); the row pass
 * scales them into bf16 dlogits in place.  dlogits thus carry an fp16 rounding of e_j before
 * their bf16 rounding; x[idx] is formed apart in fp32 from the row's hidden state and row
 * idx of the head weight.
 * grad_hidden's GEMM is split along the vocabulary and its splits are summed in a fixed
 * order, and each element of grad_weight receives one add per chunk, so the results do not
 * depend on timing.
 *
 * Masked rows (mask[r] == 0) are left out of the chunks: their outputs and their grad_hidden
 * rows are zero, and they add nothing to grad_weight, so their logits are never formed.  The
 * chunks hold the unmasked rows in batch order, chunk_rows of them each; the packing is done
 * on the device, so the call does not synchronise with the host.  (The zero-gradient
 * early-out of [Liger-bwd], taken for whole masked rows before their logits exist.)  The
 * chunk a row falls in, and so the fp32 summation order of grad_weight, depends on the mask.
 *
 *   hidden        [B*L, H] bf16, row-major, 16-byte aligned;  H a multiple of 8
 *   weight        [V, H] bf16, row-major, 16-byte aligned
 *   idx, old_logp, ref_logp, adv, mask, dloss, T, beta, eps_low, eps_high, loss, logp,
 *   lse, kl, is_clipped, entropy, dev_err: as in grpo_loss_fused (per-row arrays [B*L])
 *   chunk_rows    rows per chunk, >= 1 (the last chunk may be shorter)
 *   workspace     device scratch of at least grpo_fused_linear_workspace_size() bytes,
 *                 256-byte aligned; its contents are not kept between calls.  The size is
 *                 one chunk's 16-bit exponentials / dlogits, statistics, gathered hidden rows
 *                 and row list (2 V8 + 32 ceil(V / 256) + 2 H + 4 bytes a row, V8 = V
 *                 rounded up to a multiple of 8, each part rounded up to 256 bytes, plus
 *                 256) and max(128 MiB, chunk_rows * H * 4) for the K splits of
 *                 grad_hidden (as many splits of chunk_rows * H * 4 bytes as fit, at most 32)
 *   grad_hidden   [B*L, H] fp32 output (overwritten), or NULL
 *   grad_weight   [V, H] fp32, ACCUMULATED into (+=), or NULL; 16-byte aligned
 *
 * The logits are formed in fp32; the statistics (lse, entropy) and x[idx] come from fp32
 * values; dlogits are bf16 (the weight's type) for the two backward GEMMs.  Calls on the same stream run in order.  A GEMM whose own copies or
 * MMAs stall for about 2 s gives up, sets GRPO_DEVERR_TIMEOUT in *dev_err and returns.
 */
grpo_status grpo_fused_linear_workspace_size(int64_t H, int64_t V, int64_t chunk_rows, uint64_t* bytes);
grpo_status grpo_fused_linear(const void* hidden, const void* weight, int64_t B, int64_t L, int64_t H, int64_t V,
                              const int64_t* idx, const float* old_logp, const float* ref_logp, const float* adv,
                              const uint8_t* mask, const float* dloss, float T, float beta, float eps_low,
                              float eps_high, int64_t chunk_rows, void* workspace, uint64_t workspace_bytes,
                              float* loss, float* logp, float* lse, float* kl, uint8_t* is_clipped, float* entropy,
                              float* grad_hidden, float* grad_weight, int32_t* dev_err, grpo_stream_t stream);

/*
 * grpo_fused_linear_noalloc -- grpo_fused_linear without a workspace argument: it allocates
 * no device memory, for callers that cannot call cudaMalloc at the point where the loss
 * runs (a runtime without a device allocator, a process whose device memory is all
 * handed to a pool it does not control, or a step that must not stall on an allocation).
 * The pages have no counterpart; this is a convenience of this library.
 *
 * Its scratch (one chunk's 16-bit exponentials / dlogits, per-128-column statistics, gathered
 * hidden rows and row list, and the K splits of grad_hidden) is a fixed 32 MiB device array
 * inside the library, which every device context that loads the library holds until the
 * process exits.  Limit: the chunk buffers, chunk_rows * (2 V8 + 32 ceil(V / 256) + 2 H + 4)
 * bytes in four parts each rounded up to 256 bytes, plus 256 bytes, plus one split of
 * grad_hidden, chunk_rows * H * 4 bytes, must fit in 32 MiB (V8 = V rounded up to a multiple
 * of 8); a larger chunk returns GRPO_ERR_UNSUPPORTED before any launch.  For V = 151936 and
 * H = 1024 that is at most 101 rows per chunk.
 *
 * The first call on a device (and the first after a cudaDeviceReset) does the set-up: it
 * looks up the array's device address in the current context.  Make that first call
 * before any stream capture.  Every call uses the whole array, so calls that overlap on the
 * GPU race on it: run them on one stream, or one after the other.  The array keeps the last
 * call's contents; nothing in it has to start at zero.
 *
 * Arguments: those of grpo_fused_linear without workspace / workspace_bytes; the results
 * equal grpo_fused_linear's at the same chunk_rows, to within the fp32 summation order of
 * grad_hidden's K splits (fewer splits may fit here).
 */
grpo_status grpo_fused_linear_noalloc(const void* hidden, const void* weight, int64_t B, int64_t L, int64_t H,
                                      int64_t V, const int64_t* idx, const float* old_logp, const float* ref_logp,
                                      const float* adv, const uint8_t* mask, const float* dloss, float T, float beta,
                                      float eps_low, float eps_high, int64_t chunk_rows, float* loss, float* logp,
                                      float* lse, float* kl, uint8_t* is_clipped, float* entropy, float* grad_hidden,
                                      float* grad_weight, int32_t* dev_err, grpo_stream_t stream);

/* A static, human-readable name for a status code (never NULL). */
const char* grpo_status_string(grpo_status status);

#ifdef __cplusplus
}
#endif

#endif /* GRPO_ROWPASS_H_ */
