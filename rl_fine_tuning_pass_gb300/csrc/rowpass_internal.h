// Internal interface between the C-ABI layer (capi.cu) and the kernel launchers.
// Host-validated parameter blocks: every pointer here has been checked for null-ness,
// alignment and aliasing by capi.cu before a launcher sees it.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

namespace grpo {

// Every kernel of the library is launched with programmatic stream serialization, and
// each one waits (griddepcontrol.wait) for the grids before it in the stream to complete
// before it touches memory.  The launch and the CTAs' set-up then overlap the previous
// kernel's drain instead of following it; the ordering the stream guarantees is kept.
template <class... KArgs, class... Args>
inline cudaError_t launch_after_previous(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t stream,
                                         Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
// The same with dynamic shared memory.
template <class... KArgs, class... Args>
inline cudaError_t launch_after_previous_smem(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                              cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Error bit OR-ed into the caller's device error word (GRPO_DEVERR_IDX_OUT_OF_RANGE).
constexpr int GRPO_DEVERR_IDX_OUT_OF_RANGE_BIT = 1;
// A bounded wait on the kernel's own asynchronous copies ran out (GRPO_DEVERR_TIMEOUT).
constexpr int GRPO_DEVERR_TIMEOUT_BIT = 2;

// 16-byte loads in flight per thread: single-warp CTAs keep more of them so that a
// warp streaming a whole row still covers the memory latency.
constexpr int kUnroll = 4;
constexpr int kUnrollSmall = 8;

// Threads per CTA (one CTA per row), from measurements on GB300 (L2 flushed):
// forward: when every row can be resident at once, all rows stream concurrently with no
//   CTA-granularity tail: 128 threads with 2 loads in flight each (up to 16 such CTAs
//   per SM; for 2048 rows of 64 KB this beat 64 threads x 4 loads, 26.6 vs 28.6 us),
//   or 64 threads x 4 loads up to 24 CTAs per SM, and for short rows (8 KB or less);
//   otherwise 256-thread CTAs, several per SM.
// backward: 256-thread CTAs (64 for short rows); rows whose factor is zero finish early
//   and the block scheduler refills their slots.
inline int pick_threads_fwd(int V, int esize, long long rows, int sms) {
  const long long bytes = static_cast<long long>(V) * esize;
  if (bytes <= 8192) return 64;
  if (rows <= 16LL * sms) return 128;
  if (rows <= 24LL * sms) return 64;
  return 256;
}
// Fused forward + backward: the second sweep re-reads the row the CTA has just read, so
// the rows in flight should fit in L2.
// - Rows of 128 KB or more: 512-thread CTAs, about 2 per SM, so some 300 rows in flight
//   (16384 rows of 297 KB: 1528 us against 1686 us with 256 threads).
// - At most 16 rows per SM: 128-thread CTAs (2048 rows of 64 KB: 45.1 us against 47.3 us).
// - Otherwise as the backward.
inline int pick_threads_fused(int V, int esize, long long rows, int sms) {
  const long long bytes = static_cast<long long>(V) * esize;
  if (bytes <= 8192) return 64;
  if (bytes >= 131072) return 512;
  return rows <= 16LL * sms ? 128 : 256;
}
inline int pick_threads_bwd(int V, int esize, long long rows, int sms) {
  (void)rows;
  (void)sms;
  const long long bytes = static_cast<long long>(V) * esize;
  return bytes <= 8192 ? 64 : 256;
}

// Strided [B, L, V] view: element (b, l, j) at ptr + b*sb + l*sl + j.
struct RowsView {
  const void* ptr;
  int64_t L;   // tokens per sequence (row r -> b = r / L, l = r % L)
  int64_t sb;  // stride between sequences, elements
  int64_t sl;  // stride between tokens, elements
  int V;       // vocabulary (< 2^31)
};

struct OutView {
  void* ptr;
  int64_t L, sb, sl;
  int V;
};

enum FwdMode : int {
  kFwdSlsm = 0,     // selective log-softmax: logp, lse
  kFwdEntropy = 1,  // entropy only
  kFwdGrpo = 2,     // GRPO loss, logp, lse (+ kl, is_clipped)
  kFwdGrpoH = 3,    // kFwdGrpo plus the entropy output
  kFwdShard = 4,    // one vocabulary shard's statistic (a, s, u, x_sel) per row
};

struct FwdParams {
  RowsView x;
  const int64_t* idx;
  const float* old_logp;  // nullable: ratio 1
  const float* ref_logp;  // read only when beta != 0
  const float* adv;       // [B]
  const uint8_t* mask;    // nullable: all tokens count
  float c;                // log2(e) / T
  float invT;             // 1 / T
  float beta;
  float lo, hi;           // 1 - eps_low, 1 + eps_high
  float* loss;
  float* logp;
  float* lse;
  float* kl;              // nullable
  uint8_t* is_clipped;    // nullable
  float* entropy;         // nullable except in kFwdEntropy / kFwdGrpoH
  int32_t* dev_err;       // nullable
  // kFwdShard: the shard's first column in the full vocabulary; output [rows][4]
  int64_t vocab_start;
  float* stats;
};

struct BwdParams {
  RowsView x;
  OutView dx;
  const int64_t* idx;
  const float* lse;
  // GRPO row factor inputs
  const float* old_logp;
  const float* ref_logp;
  const float* adv;
  const uint8_t* mask;
  const float* dloss;
  const float* logp;
  // selective-log-softmax row factor input
  const float* dlogp_up;
  // entropy backward inputs: upstream gradient of H and the forward's H
  const float* dentropy;
  const float* entropy;
  float c;  // log2(e) / T
  float T;
  float beta;
  float lo, hi;
  int32_t* dev_err;
  // vocabulary shard (the *_vocab_shard entry points): columns [vocab_start,
  // vocab_start + V) of rows of vocab_total columns; p_rest = mass outside the idx shard
  int64_t vocab_start;
  int64_t vocab_total;
  const float* p_rest;
};

// Fused forward + backward: the forward's inputs and outputs, the gradient rows and the
// per-token loss weights, known before the forward.
struct FusedParams {
  FwdParams f;
  OutView dx;
  const float* dloss;
  float T;
};

// Sequence-level GRPO terms over B sequences of L tokens.
struct SeqParams {
  int64_t B, L;
  const float* logp;
  const float* old_logp;  // nullable: ratio 1
  const float* ref_logp;  // read only when beta != 0
  const float* adv;       // [B]
  const uint8_t* mask;    // nullable
  const float* dloss;
  float beta, lo, hi;
  float* loss;
  float* kl;              // nullable
  float* dlogp;
  float* seq_ratio;       // [B], nullable
  uint8_t* seq_is_clipped;  // [B], nullable
};
cudaError_t launch_seq(const SeqParams& p, cudaStream_t stream);

// Merge of gathered vocabulary-shard statistics (one thread per row).
constexpr int kVocabMaxWorld = 64;
struct VocabCombineParams {
  int world;
  int64_t starts[kVocabMaxWorld + 1];  // shard k: columns [starts[k], starts[k+1])
  const float* stats;                  // [world][rows][4]
  int64_t rows;
  FwdParams f;                         // x.L, idx, old/ref, adv, mask, c, beta, lo, hi, outputs
  float* p_rest;                       // nullable
};
cudaError_t launch_vocab_combine(const VocabCombineParams& p, bool grpo, cudaStream_t stream);

// Kernel launchers, one translation unit per element type (compiled in parallel).
cudaError_t launch_fwd_bf16(int mode, const FwdParams& p, int64_t rows, int sms, cudaStream_t stream);
cudaError_t launch_fwd_f32(int mode, const FwdParams& p, int64_t rows, int sms, cudaStream_t stream);
cudaError_t launch_bwd_bf16(bool grpo, bool same_phase, const BwdParams& p, int64_t rows, int sms,
                            cudaStream_t stream);
cudaError_t launch_bwd_f32(bool grpo, bool same_phase, const BwdParams& p, int64_t rows, int sms,
                           cudaStream_t stream);
// The same backward on one vocabulary shard (BwdParams::vocab_start / vocab_total / p_rest).
cudaError_t launch_bwd_shard_bf16(bool grpo, bool same_phase, const BwdParams& p, int64_t rows, int sms,
                                  cudaStream_t stream);
cudaError_t launch_bwd_shard_f32(bool grpo, bool same_phase, const BwdParams& p, int64_t rows, int sms,
                                 cudaStream_t stream);

cudaError_t launch_entgrad_bf16(bool same_phase, const BwdParams& p, int64_t rows, int sms, cudaStream_t stream);
cudaError_t launch_entgrad_f32(bool same_phase, const BwdParams& p, int64_t rows, int sms, cudaStream_t stream);

inline cudaError_t launch_entgrad(int dtype, bool same_phase, const BwdParams& p, int64_t rows, int sms,
                                  cudaStream_t stream) {
  return dtype == 1 ? launch_entgrad_bf16(same_phase, p, rows, sms, stream)
                    : launch_entgrad_f32(same_phase, p, rows, sms, stream);
}

cudaError_t launch_fused_bf16(const FusedParams& q, int64_t rows, bool same_phase, int sms, cudaStream_t stream);
cudaError_t launch_fused_f32(const FusedParams& q, int64_t rows, bool same_phase, int sms, cudaStream_t stream);

inline cudaError_t launch_fused(int dtype, const FusedParams& q, int64_t rows, bool same_phase, int sms,
                                cudaStream_t stream) {
  return dtype == 1 ? launch_fused_bf16(q, rows, same_phase, sms, stream)
                    : launch_fused_f32(q, rows, same_phase, sms, stream);
}

// Launch the forward over `rows` rows.  dtype: 0 fp32, 1 bf16.
inline cudaError_t launch_fwd(int mode, int dtype, const FwdParams& p, int64_t rows, int sms,
                              cudaStream_t stream) {
  return dtype == 1 ? launch_fwd_bf16(mode, p, rows, sms, stream) : launch_fwd_f32(mode, p, rows, sms, stream);
}
// grpo: GRPO row factor (true) or selective-log-softmax row factor (false).
// same_phase: input and output rows have equal start addresses mod 16 for every row.
inline cudaError_t launch_bwd(bool grpo, int dtype, bool same_phase, const BwdParams& p, int64_t rows, int sms,
                              cudaStream_t stream) {
  return dtype == 1 ? launch_bwd_bf16(grpo, same_phase, p, rows, sms, stream)
                    : launch_bwd_f32(grpo, same_phase, p, rows, sms, stream);
}
inline cudaError_t launch_bwd_shard(bool grpo, int dtype, bool same_phase, const BwdParams& p, int64_t rows,
                                    int sms, cudaStream_t stream) {
  return dtype == 1 ? launch_bwd_shard_bf16(grpo, same_phase, p, rows, sms, stream)
                    : launch_bwd_shard_f32(grpo, same_phase, p, rows, sms, stream);
}

}  // namespace grpo
