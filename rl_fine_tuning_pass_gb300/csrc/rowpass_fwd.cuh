// Forward row kernels: one pass over each row's logits computes the online softmax
// statistic (running offset, sum of exponentials, entropy accumulator) and, in the
// epilogue, lse, the selective log-prob, the entropy and the GRPO token loss.
//
// Definitions follow "Axolotl: entropy and selective log-softmax with Triton kernels"
// (sections "1. benchmarks/bench_entropy.py" and "2. ...bench_selective_logsoftmax.py")
// and, for the loss, the clipped-ratio objective with the k3 KL term whose gradient
// "LinkedIn Liger-Kernel GRPO Loss Backward optimisation", section "Code analysis",
// prints.  One CTA per row (a single warp per row when few rows are to be processed);
// each thread streams 16-byte vectors, UNROLL of them in flight, and folds each chunk
// into its statistic with one rescale per chunk and packed f32x2 arithmetic.
#pragma once

#include <cmath>

#include "rowpass_common.cuh"

namespace grpo {
namespace {

constexpr float kNegClamp = -1.152921504606847e18f;  // -2^60: stands in for -inf in the entropy sum

// Per-thread state: the maximum m seen so far (raw logits, exact) decides when to move
// the offset a = m * c; the sums are kept as even/odd pairs for the f32x2 instructions.
struct Running {
  float m, a;
  float2 s, u;
};

template <bool kH>
__device__ __forceinline__ void run_rescale(Running& rs, float newm, float c) {
  const float a_new = newm * c;
  if (rs.s.x != 0.f || rs.s.y != 0.f) {
    const float delta = rs.a - a_new;  // <= 0
    const float alpha = ex2(delta);
    const float2 al = make_float2(alpha, alpha);
    if (kH) rs.u = __fmul2_rn(al, __ffma2_rn(make_float2(delta, delta), rs.s, rs.u));
    rs.s = __fmul2_rn(al, rs.s);
  }
  rs.m = newm;
  rs.a = a_new;
}

// Fold one pair of logits into the sums (the running max already covers them).
template <bool kH>
__device__ __forceinline__ void run_pair(Running& rs, float2 x, float2 c2, float2 na2) {
  const float2 t = __ffma2_rn(x, c2, na2);
  const float2 e = make_float2(ex2(t.x), ex2(t.y));
  rs.s = __fadd2_rn(rs.s, e);
  if (kH) rs.u = __ffma2_rn(e, t, rs.u);
}

template <bool kH>
__device__ __forceinline__ void run_scalar(Running& rs, float x, float c) {
  if (x > rs.m) run_rescale<kH>(rs, x, c);
  if (kH && x < kNegClamp) x = kNegClamp;  // entropy: a -inf logit adds 0, not 0 * -inf
  const float t = fmaf(x, c, -rs.a);
  const float e = ex2(t);
  rs.s.x += e;
  if (kH) rs.u.x = fmaf(e, t, rs.u.x);
}

template <class E, bool kH, int N>
__device__ __forceinline__ void run_vectors(Running& rs, uint4 (&v)[N], float c) {
  const float cm = E::template chunk_max<N>(v);
  if (cm > rs.m) run_rescale<kH>(rs, cm, c);
  const float2 c2 = make_float2(c, c), na2 = make_float2(-rs.a, -rs.a);
#pragma unroll
  for (int k = 0; k < N; ++k) {
    if (kH) E::clamp_low(v[k]);
#pragma unroll
    for (int i = 0; i < E::kPairs; ++i) run_pair<kH>(rs, E::pair(v[k], i), c2, na2);
  }
}

// L2 priority of a row's logits in the forward.
enum FwdL2 : int { kL2Default = 0, kL2First = 1, kL2Last = 2 };

// The row body: 16-byte vectors [0, nvec), UNROLL in flight per thread, loaded with the
// L2 priority POL.
template <class E, int THREADS, int UNROLL, bool kH, int POL>
__device__ __forceinline__ void stream_vectors(Running& rs, const uint4* vb, int nvec, float c) {
  auto load = [](const uint4* q) {
    if constexpr (POL == kL2First) return ld_nc_v4_evict_first(q);
    else if constexpr (POL == kL2Last) return ld_nc_v4_evict_last(q);
    else return ld_nc_v4(q);
  };
  int i = threadIdx.x;
  for (; i + (UNROLL - 1) * THREADS < nvec; i += UNROLL * THREADS) {
    uint4 v[UNROLL];
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) v[k] = load(vb + i + k * THREADS);
    run_vectors<E, kH>(rs, v, c);
  }
  for (; i < nvec; i += THREADS) {
    uint4 v[1];
    v[0] = load(vb + i);
    run_vectors<E, kH>(rs, v, c);
  }
}

// A row's old_logp, ref_logp (0 when beta == 0) and advantage, loaded in advance.
struct RowScalars {
  float old, ref, A;
};

// Outputs of one row from its merged statistic (thread 0); returns logp and lse through
// the optional pointers.  `pre` (optional): the row's scalars, already loaded.
template <int MODE>
__device__ __forceinline__ void row_epilogue(const FwdParams& p, int64_t r, int64_t b, const Stat& st, float c,
                                             float x_idx, bool bad_idx, float* logp_out = nullptr,
                                             float* lse_out = nullptr, const RowScalars* pre = nullptr) {
  constexpr bool kH = MODE == kFwdEntropy || MODE == kFwdGrpoH;
  constexpr bool kGrpo = MODE == kFwdGrpo || MODE == kFwdGrpoH;
  const float ln_s = logf(st.s);
  const float lse = fmaf(st.a, kLn2, ln_s);  // ln2 * a + ln s
  float H = 0.f;
  if (kH) H = ln_s - kLn2 * st.u / st.s;
  if (MODE == kFwdEntropy) {
    p.entropy[r] = H;
    if (p.lse) p.lse[r] = lse;
    return;
  }
  // z_idx - lse = ln2 * (x_idx * c - a) - ln s, with the same offset a as the stream
  const float logp = bad_idx ? __int_as_float(0x7FC00000) : fmaf(kLn2, fmaf(x_idx, c, -st.a), -ln_s);
  if (bad_idx && p.dev_err) atomicOr(p.dev_err, GRPO_DEVERR_IDX_OUT_OF_RANGE_BIT);
  p.logp[r] = logp;
  p.lse[r] = lse;
  if (logp_out) *logp_out = logp;
  if (lse_out) *lse_out = lse;
  if (!kGrpo) return;

  const float ratio = p.old_logp ? expf(logp - (pre ? pre->old : p.old_logp[r])) : 1.f;
  const float A = pre ? pre->A : p.adv[b];
  // clip(ratio, lo, hi) written with comparisons so that a NaN ratio stays NaN
  const float clipped = ratio < p.lo ? p.lo : (ratio > p.hi ? p.hi : ratio);
  const float obj = ratio * A, obj_clipped = clipped * A;
  const bool is_clipped = obj_clipped < obj;
  const float pg = is_clipped ? -obj_clipped : -obj;
  float kl = 0.f;
  if (p.beta != 0.f) {
    const float d = (pre ? pre->ref : p.ref_logp[r]) - logp;
    kl = p.beta * (expm1f(d) - d);  // beta (e^d - d - 1), no cancellation for small d
  }
  if (bad_idx) kl = __int_as_float(0x7FC00000);
  p.loss[r] = pg + kl;
  if (p.kl) p.kl[r] = kl;
  if (p.is_clipped) p.is_clipped[r] = is_clipped ? 1 : 0;
  if (kH) p.entropy[r] = H;
}

__device__ __forceinline__ void masked_row_outputs(const FwdParams& p, int64_t r) {
  p.loss[r] = 0.f;
  p.logp[r] = 0.f;
  p.lse[r] = 0.f;
  if (p.kl) p.kl[r] = 0.f;
  if (p.is_clipped) p.is_clipped[r] = 0;
  if (p.entropy) p.entropy[r] = 0.f;
}

template <class E, int THREADS, int UNROLL, int MODE>
__global__ void __launch_bounds__(THREADS) rowstats_kernel(const FwdParams p) {
  wait_for_previous_grids();
  constexpr bool kShard = MODE == kFwdShard;
  constexpr bool kIdx = MODE != kFwdEntropy;  // kFwdShard: only when p.idx is given
  constexpr bool kH = MODE == kFwdEntropy || MODE == kFwdGrpoH || kShard;
  constexpr bool kGrpo = MODE == kFwdGrpo || MODE == kFwdGrpoH;
  constexpr int VEC = E::kVec;
  using S = typename E::storage;

  const int64_t r = blockIdx.x;
  const int64_t b = r / p.x.L;
  const int64_t l = r - b * p.x.L;
  const int tid = threadIdx.x;

  // with beta == 0, a zero advantage makes the row's gradient zero: the backward will not
  // read this row again (loaded together with the mask: one round trip); every other GRPO
  // row is kept in L2 for the backward
  const float A_pre = (kGrpo && p.beta == 0.f) ? p.adv[b] : 1.f;
  if ((kGrpo || kShard) && p.mask != nullptr && p.mask[r] == 0) {
    // masked token: not part of the objective; every output is +0.0, no logits read
    if (tid == 0) {
      if constexpr (kShard) reinterpret_cast<float4*>(p.stats)[r] = make_float4(0.f, 0.f, 0.f, 0.f);
      else masked_row_outputs(p, r);
    }
    return;
  }

  const S* row = static_cast<const S*>(p.x.ptr) + b * p.x.sb + l * p.x.sl;
  const int V = p.x.V;
  const float c = p.c;

  // idx is loaded now; the selected logit x[idx] only after the stream, so that no
  // dependent load delays the first logits loads of this warp
  int64_t id = 0;
  if (kIdx && tid == 0 && (!kShard || p.idx != nullptr)) id = p.idx[r];

  Running rs{-INFINITY, 0.f, make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  const RowSplit sp = split_row<E>(row, V);
  if (tid < sp.head) run_scalar<kH>(rs, E::load_scalar(row + tid), c);
  if (tid < sp.tail) run_scalar<kH>(rs, E::load_scalar(row + sp.head + sp.nvec * VEC + tid), c);

  const uint4* vb = reinterpret_cast<const uint4*>(row + sp.head);
  if (!kGrpo) stream_vectors<E, THREADS, UNROLL, kH, kL2Default>(rs, vb, sp.nvec, c);
  else if (A_pre == 0.f) stream_vectors<E, THREADS, UNROLL, kH, kL2First>(rs, vb, sp.nvec, c);
  else stream_vectors<E, THREADS, UNROLL, kH, kL2Last>(rs, vb, sp.nvec, c);

  bool bad_idx = false;
  float x_idx = 0.f;
  if (kIdx && tid == 0) {
    if constexpr (kShard) {  // the selected logit, if idx falls in this shard
      const int64_t loc = id - p.vocab_start;
      if (p.idx != nullptr && loc >= 0 && loc < V) x_idx = E::load_scalar(row + static_cast<int>(loc));
    } else {
      bad_idx = id < 0 || id >= V;
      x_idx = E::load_scalar(row + (bad_idx ? 0 : static_cast<int>(id)));
    }
  }
  Stat mine;
  mine.a = rs.a;
  mine.s = rs.s.x + rs.s.y;
  mine.u = rs.u.x + rs.u.y;
  const Stat st = stat_block_reduce<THREADS>(mine);
  if (tid != 0) return;
  if constexpr (kShard) reinterpret_cast<float4*>(p.stats)[r] = make_float4(st.a, st.s, st.u, x_idx);
  else row_epilogue<MODE>(p, r, b, st, c, x_idx, bad_idx);
}

template <class E, int THREADS, int U>
cudaError_t launch_mode(int mode, const FwdParams& p, int64_t rows, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>(rows));
  switch (mode) {
    case kFwdSlsm: return launch_after_previous(rowstats_kernel<E, THREADS, U, kFwdSlsm>, grid, dim3(THREADS), s, p);
    case kFwdEntropy:
      return launch_after_previous(rowstats_kernel<E, THREADS, U, kFwdEntropy>, grid, dim3(THREADS), s, p);
    case kFwdGrpo: return launch_after_previous(rowstats_kernel<E, THREADS, U, kFwdGrpo>, grid, dim3(THREADS), s, p);
    case kFwdGrpoH:
      return launch_after_previous(rowstats_kernel<E, THREADS, U, kFwdGrpoH>, grid, dim3(THREADS), s, p);
    case kFwdShard:
      return launch_after_previous(rowstats_kernel<E, THREADS, U, kFwdShard>, grid, dim3(THREADS), s, p);
    default: return cudaErrorInvalidValue;
  }
}

template <class E>
cudaError_t launch_dtype(int mode, const FwdParams& p, int64_t rows, int sms, cudaStream_t s) {
  switch (pick_threads_fwd(p.x.V, sizeof(typename E::storage), rows, sms)) {
    case 32: return launch_mode<E, 32, kUnrollSmall>(mode, p, rows, s);
    case 64: return launch_mode<E, 64, kUnroll>(mode, p, rows, s);
    case 128: return launch_mode<E, 128, 2>(mode, p, rows, s);
    default: return launch_mode<E, 256, kUnroll>(mode, p, rows, s);
  }
}

}  // namespace
}  // namespace grpo
