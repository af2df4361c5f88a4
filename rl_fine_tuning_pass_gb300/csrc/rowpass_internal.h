// Internal interface between the C-ABI layer (capi.cu) and the kernel launchers.
// Host-validated parameter blocks: every pointer here has been checked for null-ness,
// alignment and aliasing by capi.cu before a launcher sees it.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace grpo {

// Error bit OR-ed into the caller's device error word (GRPO_DEVERR_IDX_OUT_OF_RANGE).
constexpr int GRPO_DEVERR_IDX_OUT_OF_RANGE_BIT = 1;

// Threads per CTA for a row of V elements of `esize` bytes: enough 16-byte vectors per
// thread to keep several loads in flight, and a whole row per CTA.
inline int pick_threads(int V, int esize) {
  const long long bytes = static_cast<long long>(V) * esize;
  if (bytes <= 4096) return 128;
  if (bytes <= 32768) return 256;
  if (bytes <= 131072) return 512;
  return 1024;
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
  float c;  // log2(e) / T
  float T;
  float beta;
  float lo, hi;
  int32_t* dev_err;
};

// Launch one CTA per row over `rows` rows.  dtype: 0 fp32, 1 bf16.
cudaError_t launch_fwd(int mode, int dtype, const FwdParams& p, int64_t rows, cudaStream_t stream);
// grpo: GRPO row factor (true) or selective-log-softmax row factor (false).
// same_phase: input and output rows have equal start addresses mod 16 for every row.
cudaError_t launch_bwd(bool grpo, int dtype, bool same_phase, const BwdParams& p, int64_t rows,
                       cudaStream_t stream);

}  // namespace grpo
