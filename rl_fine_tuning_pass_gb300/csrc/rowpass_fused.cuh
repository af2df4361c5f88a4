// Fused single-read GRPO forward + backward, for per-token loss weights (dloss) that are
// known before the forward ("Liger GRPO meets TRL", section 4: the chunked loss computes
// the gradients during the forward, so the logits never have to be kept for a later
// backward).  One CTA per row: the row is streamed once for the statistic and the
// forward outputs; thread 0 decides the row factor g from this row's own logp (the same
// fp32 value the forward writes); a row with g == 0 is filled with +0.0, any other row
// is swept a second time to write g * (1[j == idx] - p_j).  The second sweep re-reads
// the row the same CTA has just read, so on the GPU it is mostly served by L2.
#pragma once

#include "rowpass_bwd.cuh"
#include "rowpass_fwd.cuh"

namespace grpo {
namespace {

// keep_vecs > 0 (rows whose logits and dlogits share their phase): the first keep_vecs 16-byte
// vectors of the row's body are kept in (dynamic) shared memory by the first sweep and read
// back from there by the second, so only the rest of the row has to stay in L2 between them.
template <class E, int THREADS, int UNROLL, bool kH, bool SAME_PHASE>
__global__ void __launch_bounds__(THREADS) fused_kernel(const FusedParams q, int keep_vecs) {
  extern __shared__ uint4 fused_kept[];
  wait_for_previous_grids();
  constexpr int MODE = kH ? kFwdGrpoH : kFwdGrpo;
  constexpr int VEC = E::kVec;
  using S = typename E::storage;
  const FwdParams& p = q.f;

  const int64_t r = blockIdx.x;
  const int64_t b = r / p.x.L;
  const int64_t l = r - b * p.x.L;
  const int tid = threadIdx.x;
  const int V = p.x.V;
  const float c = p.c;
  S* out = static_cast<S*>(q.dx.ptr) + b * q.dx.sb + l * q.dx.sl;
  const RowSplit osp = split_row<E>(out, V);
  const Span osn = whole_row(osp);

  const int64_t id64 = p.idx[r];  // loaded with the mask, before either is waited on
  const float A_pre = p.beta == 0.f ? p.adv[b] : 1.f;
  if (p.mask != nullptr && p.mask[r] == 0) {  // masked token: zero outputs, zero gradient row
    if (tid == 0) masked_row_outputs(p, r);
    fill_span<E, THREADS>(out, osp, osn, 0u);
    return;
  }

  const S* row = static_cast<const S*>(p.x.ptr) + b * p.x.sb + l * p.x.sl;
  const bool bad_idx = id64 < 0 || id64 >= V;
  const int idx = bad_idx ? 0 : static_cast<int>(id64);

  // sweep 1: the online statistic (as in rowstats_kernel)
  Running rs{-INFINITY, 0.f, make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  const RowSplit sp = split_row<E>(row, V);
  if (tid < sp.head) run_scalar<kH>(rs, E::load_scalar(row + tid), c);
  if (tid < sp.tail) run_scalar<kH>(rs, E::load_scalar(row + sp.head + sp.nvec * VEC + tid), c);
  const uint4* vb = reinterpret_cast<const uint4*>(row + sp.head);
  // L2: a row whose gradient is zero in advance (A == 0 with beta == 0) is not read again;
  // any other row is kept (evict_last) for the second sweep, which lets it go.
  // Coherent loads: dlogits may alias the logits.
  const bool kept = A_pre != 0.f;
  // the shared-memory copy: only for a row that is swept again (its first kv vectors are then
  // loaded evict_first, as their last read from L2)
  const int kv = (SAME_PHASE && kept) ? min(keep_vecs, sp.nvec) : 0;
  auto sweep1 = [&](auto load) {
    int i = tid;
    for (; i + (UNROLL - 1) * THREADS < sp.nvec; i += UNROLL * THREADS) {
      uint4 v[UNROLL];
#pragma unroll
      for (int k = 0; k < UNROLL; ++k) {
        const int j = i + k * THREADS;
        if (j < kv) {
          v[k] = ld_v4_evict_first(vb + j);
          fused_kept[j] = v[k];
        } else {
          v[k] = load(vb + j);
        }
      }
      run_vectors<E, kH>(rs, v, c);
    }
    for (; i < sp.nvec; i += THREADS) {
      uint4 v[1];
      if (i < kv) {
        v[0] = ld_v4_evict_first(vb + i);
        fused_kept[i] = v[0];
      } else {
        v[0] = load(vb + i);
      }
      run_vectors<E, kH>(rs, v, c);
    }
  };
  if (kept) sweep1([](const uint4* q) { return ld_v4_evict_last(q); });
  else sweep1([](const uint4* q) { return ld_v4_evict_first(q); });
  // the selected logit, loaded after the stream so that no dependent load delays it
  const float x_idx = tid == 0 ? E::load_scalar_coherent(row + idx) : 0.f;
  Stat mine;
  mine.a = rs.a;
  mine.s = rs.s.x + rs.s.y;
  mine.u = rs.u.x + rs.u.y;
  const Stat st = stat_block_reduce<THREADS>(mine);

  // forward outputs and the row factor, decided once and shared with the CTA
  __shared__ float sh_g, sh_nK;
  __shared__ int sh_idx;
  if (tid == 0) {
    float logp = 0.f, lse = 0.f;
    row_epilogue<MODE>(p, r, b, st, c, x_idx, bad_idx, &logp, &lse);
    const float g = grpo_factor(logp, p.old_logp, p.ref_logp, p.adv[b], q.dloss[r], p.beta, p.lo, p.hi, q.T, r);
    sh_g = g;
    sh_nK = fmaf(-lse, kLog2e, log2f(fabsf(g)));  // -(lse*log2e - log2|g|)
    sh_idx = bad_idx ? -1 : idx;
  }
  __syncthreads();
  const float g = sh_g;
  if (g == 0.f) {  // early-out: +0.0 over the row
    fill_span<E, THREADS>(out, osp, osn, 0u);
    if (kept) l2_demote<THREADS>(row, static_cast<int64_t>(V) * sizeof(S));
    return;
  }
  const int gidx = sh_idx;
  if (gidx < 0) {  // out-of-range idx (already reported by the forward outputs)
    fill_span<E, THREADS>(out, osp, osn, E::kNaNPair);
    if (kept) l2_demote<THREADS>(row, static_cast<int64_t>(V) * sizeof(S));
    return;
  }

  // sweep 2: dlogits (d_j = -sign(g) |g| p_j, and g (1 - p_idx) at idx)
  bool owner = false;
  const float nK = sh_nK;
  const float q_part =
      g > 0.f ? stream_span<E, THREADS, UNROLL, SAME_PHASE, true, true>(row, out, osp, osn, gidx, c, nK, owner,
                                                                         fused_kept, kv)
              : stream_span<E, THREADS, UNROLL, SAME_PHASE, false, true>(row, out, osp, osn, gidx, c, nK, owner,
                                                                          fused_kept, kv);
  const float q_total = block_sum_all<THREADS>(q_part);
  if (owner) E::store_scalar(out + gidx, g > 0.f ? q_total : -q_total);
}

// Shared memory a 512-thread CTA keeps of its row: two such CTAs fit on an SM, and the rest of
// the ~300 rows in flight (at V = 151936, 193 KB each) then fits in L2.
constexpr int kFusedKeepBytes = 104 * 1024;

template <class E, int THREADS, int U, bool kH>
cudaError_t launch_fused_h(const FusedParams& q, int64_t rows, bool same_phase, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>(rows));
  if (!same_phase) return launch_after_previous(fused_kernel<E, THREADS, U, kH, false>, grid, dim3(THREADS), s, q, 0);
  int keep = 0;
  if (THREADS == 512) {  // rows of 128 KB and more
    keep = kFusedKeepBytes / 16;
    const cudaError_t e = cudaFuncSetAttribute(fused_kernel<E, THREADS, U, kH, true>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, kFusedKeepBytes);
    if (e != cudaSuccess) return e;
  }
  return launch_after_previous_smem(fused_kernel<E, THREADS, U, kH, true>, grid, dim3(THREADS),
                                    static_cast<size_t>(keep) * 16, s, q, keep);
}

template <class E, int THREADS, int U>
cudaError_t launch_fused_t(const FusedParams& q, int64_t rows, bool same_phase, cudaStream_t s) {
  return q.f.entropy ? launch_fused_h<E, THREADS, U, true>(q, rows, same_phase, s)
                     : launch_fused_h<E, THREADS, U, false>(q, rows, same_phase, s);
}

template <class E>
cudaError_t launch_fused_dtype(const FusedParams& q, int64_t rows, bool same_phase, int sms, cudaStream_t s) {
  switch (pick_threads_fused(q.f.x.V, sizeof(typename E::storage), rows, sms)) {
    case 64: return launch_fused_t<E, 64, kUnroll>(q, rows, same_phase, s);
    case 128: return launch_fused_t<E, 128, kUnroll>(q, rows, same_phase, s);
    case 512: return launch_fused_t<E, 512, kUnroll>(q, rows, same_phase, s);
    default: return launch_fused_t<E, 256, kUnroll>(q, rows, same_phase, s);
  }
}

}  // namespace
}  // namespace grpo
