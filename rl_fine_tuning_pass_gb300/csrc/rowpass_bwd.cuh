// Backward row kernels: dlogits_j = g * (1[j == idx] - p_j) with one scalar g per row.
//
// g is decided before any logits address is formed ("LinkedIn Liger-Kernel GRPO Loss
// Backward optimisation", section "Code analysis": dlogp from the policy-gradient and
// KL terms, times dloss, divided by the temperature; when it is exactly 0.0 the row is
// filled with 0.0 and the kernel returns).  Rows with g != 0 are read once and written
// once:
//
//   |g| * p_j = 2^(x_j * c - K),   K = lse * log2(e) - log2|g|,   c = log2(e) / T
//
// so each element costs half a packed f32x2 FMA and one ex2; the sign of -g is applied
// in the conversion to the output format.  The idx element needs g * (1 - p_idx);
// 1 - p_idx is formed as the sum of the other columns' p_j (accumulated on the way,
// reduced over the CTA at the end), which keeps full relative accuracy when p_idx is
// close to 1.
#pragma once

#include <cmath>

#include "rowpass_common.cuh"

namespace grpo {
namespace {

// Per-row factor g of the GRPO loss of an unmasked token from its scalars (fp32, same
// operation order as the definition): d(pg + kl)/dlogp * dloss / T.  This is the one body
// of the formula; the backward, fused and LM-head kernels all call it.
__device__ __forceinline__ float grpo_factor_of(float logp, float old, bool has_old, float ref, float A,
                                                float dloss, float beta, float lo, float hi, float T) {
  const float ratio = has_old ? expf(logp - old) : 1.f;
  const float clipped = ratio < lo ? lo : (ratio > hi ? hi : ratio);
  // unclipped branch is the minimum (ties included): d(-ratio*A)/dlogp; else constant
  const float dpg = (ratio * A <= clipped * A) ? -A * ratio : 0.f;
  float dkl = 0.f;
  if (beta != 0.f) dkl = -beta * expm1f(ref - logp);  // beta (1 - e^(ref - logp))
  return (dpg + dkl) * dloss / T;
}

// The same factor with old/ref read from their arrays (NULL old: ratio 1; ref is read
// only when beta != 0).
__device__ __forceinline__ float grpo_factor(float logp, const float* old_logp, const float* ref_logp, float A,
                                             float dloss, float beta, float lo, float hi, float T, int64_t r) {
  const float old = old_logp ? old_logp[r] : logp;
  const float ref = beta != 0.f ? ref_logp[r] : 0.f;
  return grpo_factor_of(logp, old, old_logp != nullptr, ref, A, dloss, beta, lo, hi, T);
}

// All of a row's scalars are loaded before any of them is used, so the row waits for
// one round trip to memory before its first logits load, not several.  `kept` tells
// whether the GRPO forward read the row with L2 priority evict_last.
__device__ __forceinline__ float grpo_row_factor(const BwdParams& p, int64_t r, int64_t b, bool& kept) {
  const bool live = p.mask == nullptr || p.mask[r] != 0;
  const float logp = p.logp[r];
  const float old = p.old_logp ? p.old_logp[r] : logp;
  const float ref = p.beta != 0.f ? p.ref_logp[r] : 0.f;
  const float A = p.adv[b];
  const float dloss = p.dloss[r];
  kept = live && !(p.beta == 0.f && A == 0.f);
  if (!live) return 0.f;
  return grpo_factor_of(logp, old, p.old_logp != nullptr, ref, A, dloss, p.beta, p.lo, p.hi, p.T);
}

// The part of a row one CTA handles: vectors [v0, v1), plus the scalar head and tail.
struct Span {
  int v0, v1;
  bool head, tail;
};

__device__ __forceinline__ Span whole_row(const RowSplit& sp) { return Span{0, sp.nvec, true, true}; }

template <class E, int THREADS>
__device__ __forceinline__ void fill_span(typename E::storage* out, const RowSplit& sp, const Span& sn,
                                          uint32_t pair) {
  const int tid = threadIdx.x;
  if (sn.head && tid < sp.head) E::store_bits(out + tid, pair);
  if (sn.tail && tid < sp.tail) E::store_bits(out + sp.head + sp.nvec * E::kVec + tid, pair);
  uint4* vb = reinterpret_cast<uint4*>(out + sp.head);
  const uint4 v = make_uint4(pair, pair, pair, pair);
#pragma unroll 4
  for (int i = sn.v0 + tid; i < sn.v1; i += THREADS) st_v4_evict_first(vb + i, v);
}

// Load the VEC input elements of output vector i (input rows may be out of phase with
// the output rows; then the elements are loaded one by one).
// LAST_READ: with L2 priority evict_first.
template <class E, bool SAME_PHASE, bool LAST_READ = false>
__device__ __forceinline__ uint4 load_vec(const typename E::storage* in_body, int i) {
  if constexpr (SAME_PHASE) {
    const uint4* q = reinterpret_cast<const uint4*>(in_body) + i;
    return LAST_READ ? ld_v4_evict_first(q) : ld_v4(q);
  } else {
    float f[E::kVec];
#pragma unroll
    for (int q = 0; q < E::kVec; ++q) f[q] = E::load_scalar_coherent(in_body + i * E::kVec + q);
    return E::pack(f, 0u);  // exact: the values came from this format
  }
}

// Stream one row with g != 0: out_j = -sign(g) |g| p_j (NEG: g > 0), accumulating
// sum_{j != idx} |g| p_j for the idx element.  Returns this thread's partial sum and
// whether it wrote the idx element.  The gradient is stored with L2 priority evict_first;
// LAST_READ loads the logits with evict_first too.
// With kept_vecs > 0, body vectors [0, kept_vecs) come from `kept` (a copy the caller made in
// shared memory) instead of global memory.
template <class E, int THREADS, int UNROLL, bool SAME_PHASE, bool NEG, bool LAST_READ = false>
__device__ __forceinline__ float stream_span(const typename E::storage* in, typename E::storage* out,
                                             const RowSplit& sp, const Span& sn, int idx, float c, float nK,
                                             bool& owner, const uint4* kept = nullptr, int kept_vecs = 0) {
  constexpr int VEC = E::kVec;
  using S = typename E::storage;
  const int tid = threadIdx.x;
  float q_acc = 0.f;
  float2 q2 = make_float2(0.f, 0.f);

  auto scalar = [&](int j) {
    const float x = E::load_scalar_coherent(in + j);
    const float e = ex2(fmaf(x, c, nK));
    if (j == idx) owner = true; else q_acc += e;
    E::store_scalar(out + j, NEG ? -e : e);
  };
  if (sn.head && tid < sp.head) scalar(tid);
  if (sn.tail && tid < sp.tail) scalar(sp.head + sp.nvec * VEC + tid);

  const S* in_body = in + sp.head;
  uint4* ob = reinterpret_cast<uint4*>(out + sp.head);
  const int idx_body = idx - sp.head;  // idx relative to the body start
  const float2 c2 = make_float2(c, c), nK2 = make_float2(nK, nK);

  auto process = [&](const uint4& v, int i) {
    float2 e[E::kPairs];
#pragma unroll
    for (int q = 0; q < E::kPairs; ++q) {
      const float2 t = __ffma2_rn(E::pair(v, q), c2, nK2);
      e[q] = make_float2(ex2(t.x), ex2(t.y));
    }
    const unsigned k = static_cast<unsigned>(idx_body - i * VEC);
    if (k < static_cast<unsigned>(VEC)) {  // this vector holds idx: leave it out of the sum
      owner = true;
#pragma unroll
      for (int q = 0; q < E::kPairs; ++q) {
        if (2 * q != static_cast<int>(k)) q_acc += e[q].x;
        if (2 * q + 1 != static_cast<int>(k)) q_acc += e[q].y;
      }
    } else {
#pragma unroll
      for (int q = 0; q < E::kPairs; ++q) q2 = __fadd2_rn(q2, e[q]);
    }
    st_v4_evict_first(ob + i, E::template pack_pairs<NEG>(e));
  };

  // the part read from global memory first (L2, while it is still there), then the part kept in
  // shared memory
  auto sweep = [&](auto load, int i, int n) {
    for (; i + (UNROLL - 1) * THREADS < n; i += UNROLL * THREADS) {
      uint4 v[UNROLL];
#pragma unroll
      for (int k = 0; k < UNROLL; ++k) v[k] = load(i + k * THREADS);
#pragma unroll
      for (int k = 0; k < UNROLL; ++k) process(v[k], i + k * THREADS);
    }
    for (; i < n; i += THREADS) process(load(i), i);
  };
  const int g0 = sn.v0 > kept_vecs ? sn.v0 : kept_vecs;
  sweep([&](int j) { return load_vec<E, SAME_PHASE, LAST_READ>(in_body, j); }, g0 + tid, sn.v1);
  if (kept_vecs > sn.v0) sweep([&](int j) { return kept[j]; }, sn.v0 + tid, kept_vecs < sn.v1 ? kept_vecs : sn.v1);
  return q_acc + (q2.x + q2.y);
}

// SHARD: the logits rows are one vocabulary shard (columns [vocab_start, vocab_start + V)
// of rows of vocab_total columns).  The idx element is written only by the shard that
// holds idx, as sign(g) (|g| sum of the shard's other p_j + |g| p_rest).
template <class E, int THREADS, int UNROLL, bool GRPO, bool SAME_PHASE, bool SHARD>
__global__ void __launch_bounds__(THREADS) rowgrad_kernel(const BwdParams p) {
  using S = typename E::storage;
  wait_for_previous_grids();
  const int64_t r = blockIdx.x;
  const int64_t b = r / p.x.L;
  const int64_t l = r - b * p.x.L;
  const int tid = threadIdx.x;
  const int V = p.x.V;

  // row factor, computed redundantly by every thread from broadcast loads; idx and lse
  // are loaded in the same round trip (they are only used when g != 0)
  const int64_t id64 = p.idx[r];
  const float lse = p.lse[r];
  const float prest = SHARD && p.p_rest != nullptr ? p.p_rest[r] : 0.f;
  bool kept = false;  // the GRPO forward read this row with evict_last
  const float g = GRPO ? grpo_row_factor(p, r, b, kept) : p.dlogp_up[r] / p.T;
  S* out = static_cast<S*>(p.dx.ptr) + b * p.dx.sb + l * p.dx.sl;
  const RowSplit sp = split_row<E>(out, V);
  const Span sn = whole_row(sp);
  const S* in = static_cast<const S*>(p.x.ptr) + b * p.x.sb + l * p.x.sl;

  if (g == 0.f) {  // early-out: +0.0 over the row, nothing read
    fill_span<E, THREADS>(out, sp, sn, 0u);
    if (kept) l2_demote<THREADS>(in, static_cast<int64_t>(V) * sizeof(S));
    return;
  }
  if (id64 < 0 || id64 >= (SHARD ? p.vocab_total : static_cast<int64_t>(V))) {
    fill_span<E, THREADS>(out, sp, sn, E::kNaNPair);
    if (kept) l2_demote<THREADS>(in, static_cast<int64_t>(V) * sizeof(S));
    if (tid == 0 && p.dev_err) atomicOr(p.dev_err, GRPO_DEVERR_IDX_OUT_OF_RANGE_BIT);
    return;
  }
  int idx = static_cast<int>(id64);
  if constexpr (SHARD) {  // -1: idx is in another shard, no element of this one is excluded
    const int64_t loc = id64 - p.vocab_start;
    idx = loc >= 0 && loc < V ? static_cast<int>(loc) : -1;
  }
  const float nK = fmaf(-lse, kLog2e, log2f(fabsf(g)));  // -(lse*log2e - log2|g|)
  bool owner = false;
  // d_j = -sign(g) |g| p_j: negated when g > 0.  After a GRPO forward this is the row's
  // last read: evict_first.
  const float q_part =
      g > 0.f ? stream_span<E, THREADS, UNROLL, SAME_PHASE, true, GRPO>(in, out, sp, sn, idx, p.c, nK, owner)
              : stream_span<E, THREADS, UNROLL, SAME_PHASE, false, GRPO>(in, out, sp, sn, idx, p.c, nK, owner);

  // g (1 - p_idx) = sign(g) * sum_{j != idx} |g| p_j; written by the thread that wrote
  // the idx element's provisional value, so its two stores stay in program order.
  float q_total = block_sum_all<THREADS>(q_part);
  if (SHARD) q_total += fabsf(g) * prest;
  if (owner) E::store_scalar(out + idx, g > 0.f ? q_total : -q_total);
}

// Entropy backward: d_j = g p_j (log p_j + H), g = -dH / T.  With |g| folded into the
// exponent, |g| p_j = 2^{t_j}, t_j = x_j c - K, and log p_j + H = ln2 t_j + (H - ln|g|),
// so each element costs a packed FMA, one ex2, a packed FMA and a packed multiply.  A
// -inf logit is raised to -2^60 first, so that a p_j = 0 term is 0 and not 0 * -inf.
template <class E, int THREADS, int UNROLL, bool SAME_PHASE, bool NEG>
__device__ __forceinline__ void stream_span_entropy(const typename E::storage* in, typename E::storage* out,
                                                    const RowSplit& sp, const Span& sn, float c, float nK,
                                                    float h_shift) {
  constexpr int VEC = E::kVec;
  using S = typename E::storage;
  constexpr float kNeg = -1.152921504606847e18f;  // -2^60
  const int tid = threadIdx.x;
  auto scalar = [&](int j) {
    float x = E::load_scalar_coherent(in + j);
    if (x < kNeg) x = kNeg;
    const float t = fmaf(x, c, nK);
    const float d = ex2(t) * fmaf(kLn2, t, h_shift);
    E::store_scalar(out + j, NEG ? -d : d);
  };
  if (sn.head && tid < sp.head) scalar(tid);
  if (sn.tail && tid < sp.tail) scalar(sp.head + sp.nvec * VEC + tid);
  const S* in_body = in + sp.head;
  uint4* ob = reinterpret_cast<uint4*>(out + sp.head);
  const float2 c2 = make_float2(c, c), nK2 = make_float2(nK, nK);
  const float2 ln2 = make_float2(kLn2, kLn2), hs2 = make_float2(h_shift, h_shift);
  auto process = [&](uint4 v, int i) {
    E::clamp_low(v);
    float2 d[E::kPairs];
#pragma unroll
    for (int q = 0; q < E::kPairs; ++q) {
      const float2 t = __ffma2_rn(E::pair(v, q), c2, nK2);
      const float2 e = make_float2(ex2(t.x), ex2(t.y));
      d[q] = __fmul2_rn(e, __ffma2_rn(ln2, t, hs2));
    }
    st_v4_evict_first(ob + i, E::template pack_pairs<NEG>(d));
  };
  int i = sn.v0 + tid;
  for (; i + (UNROLL - 1) * THREADS < sn.v1; i += UNROLL * THREADS) {
    uint4 v[UNROLL];
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) v[k] = load_vec<E, SAME_PHASE>(in_body, i + k * THREADS);
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) process(v[k], i + k * THREADS);
  }
  for (; i < sn.v1; i += THREADS) process(load_vec<E, SAME_PHASE>(in_body, i), i);
}

template <class E, int THREADS, int UNROLL, bool SAME_PHASE>
__global__ void __launch_bounds__(THREADS) entgrad_kernel(const BwdParams p) {
  using S = typename E::storage;
  wait_for_previous_grids();
  const int64_t r = blockIdx.x;
  const int64_t b = r / p.x.L;
  const int64_t l = r - b * p.x.L;
  const int V = p.x.V;
  const float lse = p.lse[r];  // same round trip as dentropy (used only when g != 0)
  const float H = p.entropy[r];
  const float g = -p.dentropy[r] / p.T;
  S* out = static_cast<S*>(p.dx.ptr) + b * p.dx.sb + l * p.dx.sl;
  const RowSplit sp = split_row<E>(out, V);
  const Span sn = whole_row(sp);
  if (g == 0.f) {  // early-out: +0.0 over the row, nothing read
    fill_span<E, THREADS>(out, sp, sn, 0u);
    return;
  }
  const S* in = static_cast<const S*>(p.x.ptr) + b * p.x.sb + l * p.x.sl;
  const float lg = log2f(fabsf(g));
  const float nK = fmaf(-lse, kLog2e, lg);        // -(lse*log2e - log2|g|)
  const float h_shift = fmaf(-kLn2, lg, H);       // H - ln|g|
  if (g < 0.f) stream_span_entropy<E, THREADS, UNROLL, SAME_PHASE, true>(in, out, sp, sn, p.c, nK, h_shift);
  else stream_span_entropy<E, THREADS, UNROLL, SAME_PHASE, false>(in, out, sp, sn, p.c, nK, h_shift);
}

template <class E>
cudaError_t launch_entgrad_dtype(bool same_phase, const BwdParams& p, int64_t rows, int sms, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>(rows));
  if (pick_threads_bwd(p.x.V, sizeof(typename E::storage), rows, sms) == 64) {
    return same_phase ? launch_after_previous(entgrad_kernel<E, 64, kUnroll, true>, grid, dim3(64), s, p)
                      : launch_after_previous(entgrad_kernel<E, 64, kUnroll, false>, grid, dim3(64), s, p);
  } else {
    return same_phase ? launch_after_previous(entgrad_kernel<E, 256, kUnroll, true>, grid, dim3(256), s, p)
                      : launch_after_previous(entgrad_kernel<E, 256, kUnroll, false>, grid, dim3(256), s, p);
  }
}

template <class E, int THREADS, int U, bool GRPO, bool SAME_PHASE, bool SHARD>
cudaError_t launch4(const BwdParams& p, int64_t rows, cudaStream_t s) {
  return launch_after_previous(rowgrad_kernel<E, THREADS, U, GRPO, SAME_PHASE, SHARD>,
                               dim3(static_cast<unsigned>(rows)), dim3(THREADS), s, p);
}

template <class E, int THREADS, int U, bool SHARD>
cudaError_t launch3(bool grpo, bool same_phase, const BwdParams& p, int64_t rows, cudaStream_t s) {
  if (grpo) return same_phase ? launch4<E, THREADS, U, true, true, SHARD>(p, rows, s)
                              : launch4<E, THREADS, U, true, false, SHARD>(p, rows, s);
  return same_phase ? launch4<E, THREADS, U, false, true, SHARD>(p, rows, s)
                    : launch4<E, THREADS, U, false, false, SHARD>(p, rows, s);
}

// pick_threads_bwd chooses 64 or 256 threads.
template <class E, bool SHARD = false>
cudaError_t launch2(bool grpo, bool same_phase, const BwdParams& p, int64_t rows, int sms, cudaStream_t s) {
  if (pick_threads_bwd(p.x.V, sizeof(typename E::storage), rows, sms) == 64)
    return launch3<E, 64, kUnroll, SHARD>(grpo, same_phase, p, rows, s);
  return launch3<E, 256, kUnroll, SHARD>(grpo, same_phase, p, rows, s);
}

}  // namespace
}  // namespace grpo
