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
// so each element costs one FMA and one ex2; the sign of -g is XOR-ed into the packed
// output.  The idx element needs g * (1 - p_idx); 1 - p_idx is formed as the sum of the
// other columns' p_j (accumulated on the way, reduced over the CTA at the end), which
// keeps full relative accuracy when p_idx is close to 1.
#include <cmath>

#include "rowpass_common.cuh"

namespace grpo {
namespace {

// Per-row factor g of the GRPO loss (fp32, same operation order as the definition).
__device__ __forceinline__ float grpo_row_factor(const BwdParams& p, int64_t r, int64_t b) {
  if (p.mask != nullptr && p.mask[r] == 0) return 0.f;
  const float logp = p.logp[r];
  const float ratio = p.old_logp ? expf(logp - p.old_logp[r]) : 1.f;
  const float A = p.adv[b];
  const float clipped = ratio < p.lo ? p.lo : (ratio > p.hi ? p.hi : ratio);
  // unclipped branch is the minimum (ties included): d(-ratio*A)/dlogp; else constant
  const float dpg = (ratio * A <= clipped * A) ? -A * ratio : 0.f;
  float dkl = 0.f;
  if (p.beta != 0.f) dkl = -p.beta * expm1f(p.ref_logp[r] - logp);  // beta (1 - e^(ref - logp))
  return (dpg + dkl) * p.dloss[r] / p.T;
}

template <class E, int THREADS>
__device__ __forceinline__ void fill_row(typename E::storage* out, int V, uint32_t pair) {
  const RowSplit sp = split_row<E>(out, V);
  const int tid = threadIdx.x;
  if (tid < sp.head) E::store_bits(out + tid, pair);
  if (tid < sp.tail) E::store_bits(out + sp.head + sp.nvec * E::kVec + tid, pair);
  uint4* vb = reinterpret_cast<uint4*>(out + sp.head);
  const uint4 v = make_uint4(pair, pair, pair, pair);
#pragma unroll 4
  for (int i = tid; i < sp.nvec; i += THREADS) st_v4(vb + i, v);
}

// Load the VEC input elements of output vector i (input rows may be out of phase with
// the output rows; then the elements are loaded one by one).
template <class E, bool SAME_PHASE>
__device__ __forceinline__ uint4 load_vec(const typename E::storage* in_body, int i) {
  if (SAME_PHASE) return ld_v4(reinterpret_cast<const uint4*>(in_body) + i);
  float f[E::kVec];
#pragma unroll
  for (int q = 0; q < E::kVec; ++q) f[q] = E::load_scalar_coherent(in_body + i * E::kVec + q);
  return E::pack(f, 0u);  // exact: the values came from this format
}

template <class E, int THREADS, int UNROLL, bool GRPO, bool SAME_PHASE>
__global__ void __launch_bounds__(THREADS) rowgrad_kernel(const BwdParams p) {
  constexpr int VEC = E::kVec;
  using S = typename E::storage;
  const int64_t r = blockIdx.x;
  const int64_t b = r / p.x.L;
  const int64_t l = r - b * p.x.L;
  const int tid = threadIdx.x;
  const int V = p.x.V;

  // row factor, computed redundantly by every thread from broadcast loads
  const float g = GRPO ? grpo_row_factor(p, r, b) : p.dlogp_up[r] / p.T;
  S* out = static_cast<S*>(p.dx.ptr) + b * p.dx.sb + l * p.dx.sl;

  if (g == 0.f) {  // early-out: +0.0 over the row, nothing read
    fill_row<E, THREADS>(out, V, 0u);
    return;
  }
  const int64_t id64 = p.idx[r];
  if (id64 < 0 || id64 >= V) {
    fill_row<E, THREADS>(out, V, E::kNaNPair);
    if (tid == 0 && p.dev_err) atomicOr(p.dev_err, GRPO_DEVERR_IDX_OUT_OF_RANGE_BIT);
    return;
  }
  const int idx = static_cast<int>(id64);
  const S* in = static_cast<const S*>(p.x.ptr) + b * p.x.sb + l * p.x.sl;
  const float c = p.c;
  const float nK = fmaf(-p.lse[r], kLog2e, log2f(fabsf(g)));  // -(lse*log2e - log2|g|)
  const uint32_t flip = g > 0.f ? E::kSignPair : 0u;            // d_j = -sign(g) |g| p_j

  float q_acc = 0.f;  // sum over j != idx of |g| p_j
  bool owner = false;

  const RowSplit sp = split_row<E>(out, V);
  auto scalar = [&](int j) {
    const float x = E::load_scalar_coherent(in + j);
    const float e = ex2(fmaf(x, c, nK));
    if (j == idx) owner = true; else q_acc += e;
    E::store_scalar(out + j, flip ? -e : e);
  };
  if (tid < sp.head) scalar(tid);
  if (tid < sp.tail) scalar(sp.head + sp.nvec * VEC + tid);

  const S* in_body = in + sp.head;
  uint4* ob = reinterpret_cast<uint4*>(out + sp.head);
  const int idx_body = idx - sp.head;  // idx relative to the body start

  auto process = [&](const uint4& v, int i) {
    float f[VEC], e[VEC];
    E::unpack(v, f);
#pragma unroll
    for (int q = 0; q < VEC; ++q) e[q] = ex2(fmaf(f[q], c, nK));
    const unsigned k = static_cast<unsigned>(idx_body - i * VEC);
    if (k < static_cast<unsigned>(VEC)) {
      owner = true;
#pragma unroll
      for (int q = 0; q < VEC; ++q)
        if (q != static_cast<int>(k)) q_acc += e[q];
    } else {
#pragma unroll
      for (int q = 0; q < VEC; ++q) q_acc += e[q];
    }
    st_v4(ob + i, E::pack(e, flip));
  };

  int i = tid;
  for (; i + (UNROLL - 1) * THREADS < sp.nvec; i += UNROLL * THREADS) {
    uint4 v[UNROLL];
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) v[k] = load_vec<E, SAME_PHASE>(in_body, i + k * THREADS);
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) process(v[k], i + k * THREADS);
  }
  for (; i < sp.nvec; i += THREADS) process(load_vec<E, SAME_PHASE>(in_body, i), i);

  // g (1 - p_idx) = sign(g) * sum_{j != idx} |g| p_j; written by the thread that wrote
  // the idx element's provisional value, so its two stores stay in program order.
  const float q_total = block_sum_all<THREADS>(q_acc);
  if (owner) E::store_scalar(out + idx, g > 0.f ? q_total : -q_total);
}

template <class E, int THREADS, bool GRPO, bool SAME_PHASE>
cudaError_t launch4(const BwdParams& p, int64_t rows, cudaStream_t s) {
  constexpr int U = 4;
  rowgrad_kernel<E, THREADS, U, GRPO, SAME_PHASE><<<dim3(static_cast<unsigned>(rows)), THREADS, 0, s>>>(p);
  return cudaGetLastError();
}

template <class E, int THREADS>
cudaError_t launch3(bool grpo, bool same_phase, const BwdParams& p, int64_t rows, cudaStream_t s) {
  if (grpo) return same_phase ? launch4<E, THREADS, true, true>(p, rows, s)
                              : launch4<E, THREADS, true, false>(p, rows, s);
  return same_phase ? launch4<E, THREADS, false, true>(p, rows, s)
                    : launch4<E, THREADS, false, false>(p, rows, s);
}

template <class E>
cudaError_t launch2(bool grpo, bool same_phase, const BwdParams& p, int64_t rows, cudaStream_t s) {
  switch (pick_threads(p.x.V, sizeof(typename E::storage))) {
    case 128: return launch3<E, 128>(grpo, same_phase, p, rows, s);
    case 256: return launch3<E, 256>(grpo, same_phase, p, rows, s);
    case 512: return launch3<E, 512>(grpo, same_phase, p, rows, s);
    default: return launch3<E, 1024>(grpo, same_phase, p, rows, s);
  }
}

}  // namespace

cudaError_t launch_bwd(bool grpo, int dtype, bool same_phase, const BwdParams& p, int64_t rows,
                       cudaStream_t stream) {
  return dtype == 1 ? launch2<BF16>(grpo, same_phase, p, rows, stream)
                    : launch2<F32>(grpo, same_phase, p, rows, stream);
}

}  // namespace grpo
