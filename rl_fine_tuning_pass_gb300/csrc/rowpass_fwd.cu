// Forward row kernels: one pass over each row's logits computes the online softmax
// statistic (running max, sum of exponentials, entropy accumulator) and, in the
// epilogue, lse, the selective log-prob, the entropy and the GRPO token loss.
//
// Definitions follow "Axolotl: entropy and selective log-softmax with Triton kernels"
// (sections "1. benchmarks/bench_entropy.py" and "2. ...bench_selective_logsoftmax.py")
// and, for the loss, the clipped-ratio objective with the k3 KL term whose gradient
// "LinkedIn Liger-Kernel GRPO Loss Backward optimisation", section "Code analysis",
// prints.  One CTA per row; each thread streams 16-byte vectors, UNROLL of them in
// flight, and folds each chunk into its statistic with one rescale per chunk.
#include <cmath>

#include "rowpass_common.cuh"

namespace grpo {
namespace {

// Running state of one thread: the maximum m seen so far (raw logits, exact) decides
// when to move the offset; the statistic itself is kept relative to a = m * c.
struct Running {
  float m;
  Stat st;
};

template <bool kH>
__device__ __forceinline__ void stat_rescale(Running& rs, float newm, float c) {
  const float a_new = newm * c;
  if (rs.st.s != 0.f) {
    const float delta = rs.st.a - a_new;  // <= 0
    const float alpha = ex2(delta);
    if (kH) rs.st.u = alpha * fmaf(delta, rs.st.s, rs.st.u);
    rs.st.s *= alpha;
  }
  rs.m = newm;
  rs.st.a = a_new;
}

// Fold elements f[0..N) into the statistic (the running max already covers them).
template <bool kH, int N>
__device__ __forceinline__ void stat_accumulate(Stat& st, const float (&f)[N], float c) {
  const float na = -st.a;
#pragma unroll
  for (int q = 0; q < N; ++q) {
    const float t = fmaf(f[q], c, na);
    const float e = ex2(t);
    st.s += e;
    if (kH) st.u = fmaf(e, t, st.u);
  }
}

template <bool kH>
__device__ __forceinline__ void stat_scalar(Running& rs, float x, float c) {
  if (x > rs.m) stat_rescale<kH>(rs, x, c);
  // entropy: a -inf logit must add 0, not 0 * -inf (see clamp_low)
  float f[1] = {kH && x < -1.152921504606847e18f ? -1.152921504606847e18f : x};
  stat_accumulate<kH>(rs.st, f, c);
}

template <class E, int THREADS, int UNROLL, int MODE>
__global__ void __launch_bounds__(THREADS) rowstats_kernel(const FwdParams p) {
  constexpr bool kIdx = MODE != kFwdEntropy;
  constexpr bool kH = MODE == kFwdEntropy || MODE == kFwdGrpoH;
  constexpr bool kGrpo = MODE == kFwdGrpo || MODE == kFwdGrpoH;
  constexpr int VEC = E::kVec;
  using S = typename E::storage;

  const int64_t r = blockIdx.x;
  const int64_t b = r / p.x.L;
  const int64_t l = r - b * p.x.L;
  const int tid = threadIdx.x;

  if (kGrpo && p.mask != nullptr && p.mask[r] == 0) {
    // masked token: not part of the objective; every output is +0.0, no logits read
    if (tid == 0) {
      p.loss[r] = 0.f;
      p.logp[r] = 0.f;
      p.lse[r] = 0.f;
      if (p.kl) p.kl[r] = 0.f;
      if (p.is_clipped) p.is_clipped[r] = 0;
      if (p.entropy) p.entropy[r] = 0.f;
    }
    return;
  }

  const S* row = static_cast<const S*>(p.x.ptr) + b * p.x.sb + l * p.x.sl;
  const int V = p.x.V;
  const float c = p.c;

  // the selected logit: one scalar load, issued before the stream so it overlaps it
  int idx = 0;
  bool bad_idx = false;
  float x_idx = 0.f;
  if (kIdx && tid == 0) {
    const int64_t id = p.idx[r];
    bad_idx = id < 0 || id >= V;
    idx = bad_idx ? 0 : static_cast<int>(id);
    x_idx = E::load_scalar(row + idx);
  }

  Running rs{-INFINITY, Stat{0.f, 0.f, 0.f}};
  const RowSplit sp = split_row<E>(row, V);
  if (tid < sp.head) stat_scalar<kH>(rs, E::load_scalar(row + tid), c);
  if (tid < sp.tail) stat_scalar<kH>(rs, E::load_scalar(row + sp.head + sp.nvec * VEC + tid), c);

  const uint4* vb = reinterpret_cast<const uint4*>(row + sp.head);
  int i = tid;
  for (; i + (UNROLL - 1) * THREADS < sp.nvec; i += UNROLL * THREADS) {
    uint4 v[UNROLL];
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) v[k] = ld_nc_v4(vb + i + k * THREADS);
    const float cm = E::template chunk_max<UNROLL>(v);
    if (cm > rs.m) stat_rescale<kH>(rs, cm, c);
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) {
      if (kH) E::clamp_low(v[k]);
      float f[VEC];
      E::unpack(v[k], f);
      stat_accumulate<kH>(rs.st, f, c);
    }
  }
  for (; i < sp.nvec; i += THREADS) {
    uint4 v[1];
    v[0] = ld_nc_v4(vb + i);
    const float cm = E::template chunk_max<1>(v);
    if (cm > rs.m) stat_rescale<kH>(rs, cm, c);
    if (kH) E::clamp_low(v[0]);
    float f[VEC];
    E::unpack(v[0], f);
    stat_accumulate<kH>(rs.st, f, c);
  }

  const Stat st = stat_block_reduce<THREADS>(rs.st);
  if (tid != 0) return;

  const float ln_s = logf(st.s);
  const float lse = fmaf(st.a, kLn2, ln_s);  // ln2 * a + ln s
  float H = 0.f;
  if (kH) H = ln_s - kLn2 * st.u / st.s;
  if (MODE == kFwdEntropy) {
    p.entropy[r] = H;
    return;
  }
  // z_idx - lse = ln2 * (x_idx * c - a) - ln s, with the same offset a as the stream
  const float logp = bad_idx ? __int_as_float(0x7FC00000) : fmaf(kLn2, fmaf(x_idx, c, -st.a), -ln_s);
  if (bad_idx && p.dev_err) atomicOr(p.dev_err, GRPO_DEVERR_IDX_OUT_OF_RANGE_BIT);
  p.logp[r] = logp;
  p.lse[r] = lse;
  if (!kGrpo) return;

  const float ratio = p.old_logp ? expf(logp - p.old_logp[r]) : 1.f;
  const float A = p.adv[b];
  // clip(ratio, lo, hi) written with comparisons so that a NaN ratio stays NaN
  const float clipped = ratio < p.lo ? p.lo : (ratio > p.hi ? p.hi : ratio);
  const float obj = ratio * A, obj_clipped = clipped * A;
  const bool is_clipped = obj_clipped < obj;
  const float pg = is_clipped ? -obj_clipped : -obj;
  float kl = 0.f;
  if (p.beta != 0.f) {
    const float d = p.ref_logp[r] - logp;
    kl = p.beta * (expm1f(d) - d);  // beta (e^d - d - 1), no cancellation for small d
  }
  if (bad_idx) kl = __int_as_float(0x7FC00000);
  p.loss[r] = pg + kl;
  if (p.kl) p.kl[r] = kl;
  if (p.is_clipped) p.is_clipped[r] = is_clipped ? 1 : 0;
  if (kH) p.entropy[r] = H;
}

template <class E, int THREADS>
cudaError_t launch_mode(int mode, const FwdParams& p, int64_t rows, cudaStream_t s) {
  constexpr int U = 4;
  const dim3 grid(static_cast<unsigned>(rows));
  switch (mode) {
    case kFwdSlsm: rowstats_kernel<E, THREADS, U, kFwdSlsm><<<grid, THREADS, 0, s>>>(p); break;
    case kFwdEntropy: rowstats_kernel<E, THREADS, U, kFwdEntropy><<<grid, THREADS, 0, s>>>(p); break;
    case kFwdGrpo: rowstats_kernel<E, THREADS, U, kFwdGrpo><<<grid, THREADS, 0, s>>>(p); break;
    case kFwdGrpoH: rowstats_kernel<E, THREADS, U, kFwdGrpoH><<<grid, THREADS, 0, s>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

template <class E>
cudaError_t launch_dtype(int mode, const FwdParams& p, int64_t rows, cudaStream_t s) {
  switch (pick_threads(p.x.V, sizeof(typename E::storage))) {
    case 128: return launch_mode<E, 128>(mode, p, rows, s);
    case 256: return launch_mode<E, 256>(mode, p, rows, s);
    case 512: return launch_mode<E, 512>(mode, p, rows, s);
    default: return launch_mode<E, 1024>(mode, p, rows, s);
  }
}

}  // namespace

cudaError_t launch_fwd(int mode, int dtype, const FwdParams& p, int64_t rows, cudaStream_t stream) {
  return dtype == 1 ? launch_dtype<BF16>(mode, p, rows, stream)
                    : launch_dtype<F32>(mode, p, rows, stream);
}

}  // namespace grpo
