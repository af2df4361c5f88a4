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

// The kept part of a row comes into shared memory by 1-D bulk copies (TMA) that thread 0
// issues: `bytes` (a multiple of 16) from the 16-byte aligned `src`, in pieces of 16 KB, each
// counted on the CTA's mbarrier `bar` (initialised here for one arrival with the byte count).
// These bytes are not needed in L2 again, so the copies read them with priority evict_first.
__device__ __forceinline__ void kept_copy_issue(uint32_t bar, uint32_t dst, const void* src, uint32_t bytes) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
  const char* s = static_cast<const char*>(src);
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  for (uint32_t off = 0; off < bytes; off += 16384u) {
    const uint32_t n = bytes - off < 16384u ? bytes - off : 16384u;
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            dst + off),
        "l"(s + off), "r"(n), "r"(bar), "l"(pol)
        : "memory");
  }
}
// Wait for the kept part to land: false after about two seconds (4e9 cycles) without it.
__device__ __forceinline__ bool kept_copy_wait(uint32_t bar) {
  const long long t0 = clock64();
  while (true) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(bar)
        : "memory");
    if (done != 0) return true;
    if (clock64() - t0 > 4000000000LL) return false;
  }
}

// A row of +0.0 written by bulk copies (TMA) from a zeroed 16 KB block `buf` of shared memory
// (evict_first); the scalar head and tail by plain stores.  Thread 0 waits until the copies
// have read the block, so the CTA may exit or reuse it afterwards.
template <class E, int THREADS>
__device__ __forceinline__ void zero_row_bulk(typename E::storage* out, const RowSplit& sp, uint4* buf) {
  const int tid = threadIdx.x;
  for (int i = tid; i < 1024; i += THREADS) buf[i] = make_uint4(0u, 0u, 0u, 0u);
  if (tid < sp.head) E::store_bits(out + tid, 0u);
  if (tid < sp.tail) E::store_bits(out + sp.head + sp.nvec * E::kVec + tid, 0u);
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncthreads();
  if (tid == 0) {
    char* dst = reinterpret_cast<char*>(out + sp.head);
    const uint32_t src = smem_addr(buf);
    const uint32_t bytes = static_cast<uint32_t>(sp.nvec) * 16u;
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    for (uint32_t off = 0; off < bytes; off += 16384u) {
      const uint32_t n = bytes - off < 16384u ? bytes - off : 16384u;
      asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(dst + off),
                   "r"(src), "r"(n), "l"(pol)
                   : "memory");
    }
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
  }
}

// keep_vecs > 0 (rows whose logits and dlogits share their phase): the first keep_vecs 16-byte
// vectors of the row's body are copied into (dynamic) shared memory by bulk copies issued
// before the first sweep, which streams the rest of the row meanwhile and then takes the kept
// part from shared memory; the second sweep reads it back from there too (after the rest, which
// it takes from L2 first, while it is still there), so only the rest of the row has to stay in
// L2 between the sweeps.
template <class E, int THREADS, int UNROLL, bool kH, bool SAME_PHASE>
__global__ void __launch_bounds__(THREADS) fused_kernel(const FusedParams q, int keep_vecs) {
  extern __shared__ uint4 fused_kept[];
  __shared__ __align__(8) uint64_t kept_bar;
  wait_for_previous_grids();
  constexpr int MODE = kH ? kFwdGrpoH : kFwdGrpo;
  constexpr int VEC = E::kVec;
  using S = typename E::storage;
  const FwdParams& p = q.f;

  // Long rows (512-thread CTAs, several waves of them): CTAs in launch order take the j-th token
  // position of every sequence in turn (the grid has one CTA per row), so the rows in flight at
  // any time come from all the sequences.  With a mask, whose masked rows sit at the ends of the
  // sequences, the positions are taken alternately from the start and the end (l = j / 2, then
  // L - 1 - j / 2), so that masked (write-only) and unmasked rows stay mixed over the launch.
  // Shorter rows go in row order.
  const int64_t nseq = gridDim.x / p.x.L;
  const int64_t j = blockIdx.x / nseq;
  const int64_t b = THREADS == 512 ? blockIdx.x % nseq : blockIdx.x / p.x.L;
  const int64_t l = THREADS != 512      ? blockIdx.x % p.x.L
                    : p.mask == nullptr ? j
                    : (j & 1)           ? p.x.L - 1 - (j >> 1)
                                        : (j >> 1);
  const int64_t r = b * p.x.L + l;
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
    if (SAME_PHASE && keep_vecs >= 1024) zero_row_bulk<E, THREADS>(out, osp, fused_kept);
    else fill_span<E, THREADS>(out, osp, osn, 0u);
    return;
  }

  // the row's scalars for thread 0's epilogue, loaded now so that their latency is hidden
  // behind the stream
  RowScalars pre{0.f, 0.f, 0.f};
  float pre_dloss = 0.f;
  if (tid == 0) {
    if (p.old_logp) pre.old = p.old_logp[r];
    if (p.beta != 0.f) pre.ref = p.ref_logp[r];
    pre.A = p.adv[b];
    pre_dloss = q.dloss[r];
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
  // the shared-memory copy: only for a row that is swept again
  const int kv = (SAME_PHASE && kept) ? min(keep_vecs, sp.nvec) : 0;
  const uint32_t bar = smem_addr(&kept_bar);
  if (kv > 0) {
    if (tid == 0) kept_copy_issue(bar, smem_addr(fused_kept), vb, static_cast<uint32_t>(kv) * 16u);
    __syncthreads();  // the mbarrier is initialised before anyone waits on it
  }
  // a long row swept again: while the CTA loads one step of UNROLL x THREADS vectors, thread 0
  // asks L2 for the next step (a bulk prefetch, evict_last), one step ahead and no more
  uint64_t pf_pol = 0;
  if (tid == 0) asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pf_pol));
  auto sweep1 = [&](auto load, const uint4* src, int i, int n, bool prefetch) {
    constexpr int kStep = UNROLL * THREADS;
    for (; i + (UNROLL - 1) * THREADS < n; i += kStep) {
      if (prefetch && tid == 0 && i + kStep < n) {
        const int e = i + 2 * kStep < n ? i + 2 * kStep : n;
        asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(src + i + kStep),
                     "r"(static_cast<uint32_t>(e - i - kStep) * 16u), "l"(pf_pol)
                     : "memory");
      }
      uint4 v[UNROLL];
#pragma unroll
      for (int k = 0; k < UNROLL; ++k) v[k] = load(src + i + k * THREADS);
      run_vectors<E, kH>(rs, v, c);
    }
    for (; i < n; i += THREADS) {
      uint4 v[1] = {load(src + i)};
      run_vectors<E, kH>(rs, v, c);
    }
  };
  if (kept) sweep1([](const uint4* a) { return ld_v4_evict_last(a); }, vb, kv + tid, sp.nvec, THREADS == 512);
  else sweep1([](const uint4* a) { return ld_v4_evict_first(a); }, vb, tid, sp.nvec, false);
  // the selected logit, loaded after the stream from global memory so that no dependent load
  // delays it, and before the kept part is processed, which hides its latency
  const float x_idx = tid == 0 ? E::load_scalar_coherent(row + idx) : 0.f;
  if (kv > 0) {
    if (!kept_copy_wait(bar)) {  // the row's outputs are not valid; wait once more for the copies in flight
      if (tid == 0 && p.dev_err != nullptr) atomicOr(p.dev_err, GRPO_DEVERR_TIMEOUT_BIT);
      kept_copy_wait(bar);
    }
    sweep1([](const uint4* a) { return *a; }, fused_kept, tid, kv, false);
  }
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
    row_epilogue<MODE>(p, r, b, st, c, x_idx, bad_idx, &logp, &lse, &pre);
    const float g = grpo_factor_of(logp, p.old_logp ? pre.old : logp, p.old_logp != nullptr, pre.ref, pre.A,
                                   pre_dloss, p.beta, p.lo, p.hi, q.T);
    sh_g = g;
    sh_nK = fmaf(-lse, kLog2e, log2f(fabsf(g)));  // -(lse*log2e - log2|g|)
    sh_idx = bad_idx ? -1 : idx;
  }
  __syncthreads();
  const float g = sh_g;
  if (g == 0.f) {  // early-out: +0.0 over the row
    if (SAME_PHASE && keep_vecs >= 1024) zero_row_bulk<E, THREADS>(out, osp, fused_kept);
    else fill_span<E, THREADS>(out, osp, osn, 0u);
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
