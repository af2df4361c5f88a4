// Sequence-level GRPO terms: one CTA per sequence (the sequence's tokens in registers when
// it has at most 1024 of them, else two passes over it).
//
// "LinkedIn Liger-Kernel GRPO Loss Backward optimisation", section "Code analysis", shows
// a sequence-level backward (_grpo_loss_bwd_kernel_seq) in which the per-token KL
// gradient beta (1 - exp(ref - logp)) is weighted by the token's dloss and the
// policy-gradient part arrives computed per sequence.  Per sequence b with n_b unmasked
// tokens (the length-normalised sequence importance ratio):
//
//   s_b = exp(sum_t m_t (logp_t - old_t) / n_b),  pg_b = -min(s_b A_b, clip(s_b) A_b),
//   loss_t = pg_b + kl_t,  dlogp_t = W_b dpg_b/dlogp_t + beta (1 - e^{ref_t - logp_t}) dloss_t,
//   W_b = sum_t dloss_t,   dpg_b/dlogp_t = -A_b s_b / n_b (unclipped) or 0 (clipping binds).
//
// dlogp feeds selective_log_softmax_bwd, which spreads dlogp / T over each row and writes
// +0.0 rows where it is zero without reading their logits.
#include <cmath>

#include "grpo_rowpass.h"
#include "rowpass_common.cuh"

namespace grpo {
namespace {

template <int THREADS>
__device__ __forceinline__ float block_sum_f(float v) { return block_sum_all<THREADS>(v); }

template <int THREADS>
__global__ void __launch_bounds__(THREADS) seq_kernel(const SeqParams p) {
  wait_for_previous_grids();
  const int64_t b = blockIdx.x;
  const int64_t L = p.L;
  const int64_t base = b * L;
  const int tid = threadIdx.x;

  float sum = 0.f, cnt = 0.f, w = 0.f;
  for (int64_t t = tid; t < L; t += THREADS) {
    const int64_t r = base + t;
    if (p.mask != nullptr && p.mask[r] == 0) continue;
    const float lp = p.logp[r];
    sum += p.old_logp ? lp - p.old_logp[r] : 0.f;
    cnt += 1.f;
    w += p.dloss[r];
  }
  sum = block_sum_f<THREADS>(sum);
  __syncthreads();
  cnt = block_sum_f<THREADS>(cnt);
  __syncthreads();
  w = block_sum_f<THREADS>(w);

  // the sequence's ratio, objective and policy-gradient derivative (same in every thread)
  const float A = p.adv[b];
  const float s = cnt > 0.f ? expf(sum / cnt) : 1.f;
  const float clipped = s < p.lo ? p.lo : (s > p.hi ? p.hi : s);
  const float obj = s * A, obj_clipped = clipped * A;
  const bool is_clipped = obj_clipped < obj;
  const float pg = is_clipped ? -obj_clipped : -obj;
  const float wdpg = (obj <= obj_clipped && cnt > 0.f) ? w * (-A * s / cnt) : 0.f;
  if (tid == 0) {
    if (p.seq_ratio) p.seq_ratio[b] = s;
    if (p.seq_is_clipped) p.seq_is_clipped[b] = is_clipped ? 1 : 0;
  }
  for (int64_t t = tid; t < L; t += THREADS) {
    const int64_t r = base + t;
    if (p.mask != nullptr && p.mask[r] == 0) {
      p.loss[r] = 0.f;
      p.dlogp[r] = 0.f;
      if (p.kl) p.kl[r] = 0.f;
      continue;
    }
    float kl = 0.f, dkl = 0.f;
    if (p.beta != 0.f) {
      const float d = p.ref_logp[r] - p.logp[r];
      const float em1 = expm1f(d);
      kl = p.beta * (em1 - d);
      dkl = -p.beta * em1;  // beta (1 - e^d)
    }
    p.loss[r] = pg + kl;
    p.dlogp[r] = fmaf(dkl, p.dloss[r], wdpg);
    if (p.kl) p.kl[r] = kl;
  }
}

// The same terms with the sequence held in registers (L <= THREADS * KT): every load is
// issued at once, without waiting for the mask; one CTA barrier reduces the three sums.
template <int THREADS, int KT>
__global__ void __launch_bounds__(THREADS) seq_kernel_regs(const SeqParams p) {
  wait_for_previous_grids();
  constexpr int kWarps = THREADS / 32;
  const int64_t b = blockIdx.x;
  const int64_t L = p.L;
  const int64_t base = b * L;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool use_ref = p.beta != 0.f;

  float lp[KT], od[KT], dl[KT], rf[KT];
  bool in[KT], live[KT];
#pragma unroll
  for (int k = 0; k < KT; ++k) {
    const int64_t t = tid + static_cast<int64_t>(k) * THREADS;
    in[k] = t < L;
    const int64_t r = base + (in[k] ? t : 0);
    lp[k] = p.logp[r];
    od[k] = p.old_logp ? p.old_logp[r] : 0.f;
    dl[k] = p.dloss[r];
    rf[k] = use_ref ? p.ref_logp[r] : 0.f;
    live[k] = in[k] && (p.mask == nullptr || p.mask[r] != 0);
  }
  float sum = 0.f, cnt = 0.f, w = 0.f;
#pragma unroll
  for (int k = 0; k < KT; ++k) {
    if (!live[k]) continue;
    sum += p.old_logp ? lp[k] - od[k] : 0.f;  // no old_logp: ratio 1
    cnt += 1.f;
    w += dl[k];
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    sum += __shfl_xor_sync(0xFFFFFFFFu, sum, off);
    cnt += __shfl_xor_sync(0xFFFFFFFFu, cnt, off);
    w += __shfl_xor_sync(0xFFFFFFFFu, w, off);
  }
  __shared__ float part[3][kWarps];
  if (lane == 0) {
    part[0][warp] = sum;
    part[1][warp] = cnt;
    part[2][warp] = w;
  }
  __syncthreads();
  sum = cnt = w = 0.f;
#pragma unroll
  for (int i = 0; i < kWarps; ++i) {
    sum += part[0][i];
    cnt += part[1][i];
    w += part[2][i];
  }

  const float A = p.adv[b];
  const float s = cnt > 0.f ? expf(sum / cnt) : 1.f;
  const float clipped = s < p.lo ? p.lo : (s > p.hi ? p.hi : s);
  const float obj = s * A, obj_clipped = clipped * A;
  const bool is_clipped = obj_clipped < obj;
  const float pg = is_clipped ? -obj_clipped : -obj;
  const float wdpg = (obj <= obj_clipped && cnt > 0.f) ? w * (-A * s / cnt) : 0.f;
  if (tid == 0) {
    if (p.seq_ratio) p.seq_ratio[b] = s;
    if (p.seq_is_clipped) p.seq_is_clipped[b] = is_clipped ? 1 : 0;
  }
#pragma unroll
  for (int k = 0; k < KT; ++k) {
    if (!in[k]) continue;
    const int64_t r = base + tid + static_cast<int64_t>(k) * THREADS;
    float loss = 0.f, kl = 0.f, dlogp = 0.f;
    if (live[k]) {
      float dkl = 0.f;
      if (use_ref) {
        const float d = rf[k] - lp[k];
        const float em1 = expm1f(d);
        kl = p.beta * (em1 - d);
        dkl = -p.beta * em1;  // beta (1 - e^d)
      }
      loss = pg + kl;
      dlogp = fmaf(dkl, dl[k], wdpg);
    }
    p.loss[r] = loss;
    p.dlogp[r] = dlogp;
    if (p.kl) p.kl[r] = kl;
  }
}

}  // namespace

cudaError_t launch_seq(const SeqParams& p, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>(p.B));
  if (p.L <= 256) return launch_after_previous(seq_kernel_regs<256, 1>, grid, dim3(256), stream, p);
  if (p.L <= 512) return launch_after_previous(seq_kernel_regs<256, 2>, grid, dim3(256), stream, p);
  if (p.L <= 1024) return launch_after_previous(seq_kernel_regs<256, 4>, grid, dim3(256), stream, p);
  return launch_after_previous(seq_kernel<256>, grid, dim3(256), stream, p);
}

}  // namespace grpo
