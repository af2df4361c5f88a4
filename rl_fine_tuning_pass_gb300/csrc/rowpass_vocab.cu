// Vocabulary-parallel forward: merge of the gathered per-shard row statistics.
//
// A vocabulary shard's statistic (a, s, u, x_sel) is the online-softmax statistic the
// forward kernel keeps for a whole row, restricted to the shard's columns (rowstats_kernel
// in mode kFwdShard).  Merging the shards in their order with the same combine rule as the
// in-row reduction gives the full row's (A, S, U); the outputs then follow from the same
// epilogue as the unsplit forward (lse, logp and entropy as in "Axolotl: entropy and
// selective log-softmax with Triton kernels"; the GRPO terms as in "LinkedIn Liger-Kernel
// GRPO Loss Backward optimisation", "Code analysis").  The merge is a handful of scalars per
// row: one thread per row, the shards' statistics read with 16-byte loads.
#include "rowpass_fwd.cuh"

namespace grpo {
namespace {

template <int MODE>
__global__ void __launch_bounds__(256) vocab_combine_kernel(const VocabCombineParams q) {
  wait_for_previous_grids();
  const FwdParams& p = q.f;
  const float4* stats = reinterpret_cast<const float4*>(q.stats);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; r < q.rows; r += stride) {
    const int64_t b = r / p.x.L;
    if (p.mask != nullptr && p.mask[r] == 0) {  // masked token: every output +0.0
      if (MODE == kFwdGrpo || MODE == kFwdGrpoH) {
        masked_row_outputs(p, r);
      } else {
        p.lse[r] = 0.f;
        if (p.logp) p.logp[r] = 0.f;
        if (p.entropy) p.entropy[r] = 0.f;
      }
      if (q.p_rest) q.p_rest[r] = 0.f;
      continue;
    }
    // the shards in order, with the in-row combine rule (empty shards are the identity)
    Stat st{-INFINITY, 0.f, 0.f};
    for (int k = 0; k < q.world; ++k) {
      const float4 v = stats[k * q.rows + r];
      st = stat_combine(st, Stat{v.x, v.y, v.z});
    }
    // the shard that holds idx, and the mass of all the others
    bool bad = false;
    float x_sel = 0.f;
    if (p.idx != nullptr) {
      const int64_t id = p.idx[r];
      bad = id < 0 || id >= q.starts[q.world];
      int owner = 0;
      while (owner + 1 < q.world && q.starts[owner + 1] <= id) ++owner;
      if (!bad) x_sel = stats[owner * q.rows + r].w;
      if (q.p_rest) {
        float rest = 0.f;
        for (int k = 0; k < q.world; ++k) {
          if (k == owner) continue;
          const float4 v = stats[k * q.rows + r];
          if (v.y != 0.f) rest += v.y * ex2(v.x - st.a);
        }
        q.p_rest[r] = bad ? __int_as_float(0x7FC00000) : rest / st.s;
      }
    }
    if (MODE == kFwdGrpo || MODE == kFwdGrpoH || MODE == kFwdSlsm) {
      row_epilogue<MODE>(p, r, b, st, p.c, x_sel, bad);
      if (MODE == kFwdSlsm && p.entropy) p.entropy[r] = logf(st.s) - kLn2 * st.u / st.s;
    } else {  // no idx: lse and entropy
      const float ln_s = logf(st.s);
      p.lse[r] = fmaf(st.a, kLn2, ln_s);
      if (p.entropy) p.entropy[r] = ln_s - kLn2 * st.u / st.s;
    }
  }
}

}  // namespace

cudaError_t launch_vocab_combine(const VocabCombineParams& q, bool grpo, cudaStream_t s) {
  const int64_t blocks = (q.rows + 255) / 256;
  const dim3 grid(static_cast<unsigned>(blocks < 65535 ? blocks : 65535));
  if (grpo) {
    if (q.f.entropy) return launch_after_previous(vocab_combine_kernel<kFwdGrpoH>, grid, dim3(256), s, q);
    return launch_after_previous(vocab_combine_kernel<kFwdGrpo>, grid, dim3(256), s, q);
  }
  if (q.f.idx) return launch_after_previous(vocab_combine_kernel<kFwdSlsm>, grid, dim3(256), s, q);
  return launch_after_previous(vocab_combine_kernel<kFwdEntropy>, grid, dim3(256), s, q);
}

}  // namespace grpo
