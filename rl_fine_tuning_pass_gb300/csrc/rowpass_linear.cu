// The GRPO loss on top of the LM head, in chunks of rows ("Liger GRPO meets TRL",
// sections 3 and 4): for each chunk of rows, its logits x = h W^T are formed, the row pass
// turns them into the loss, the forward outputs and dlogits, and the gradients of the
// chunk's hidden states (dlogits W) and of the head weight (+= dlogits^T h) are formed
// before the next chunk, so the logits of the whole batch never exist at once.
//
// The three contractions are this library's tcgen05 GEMMs (lmhead_gemm.cuh: bf16 operands
// staged by TMA, fp32 accumulation in tensor memory).  The logits GEMM forms, in its
// epilogue, the softmax statistic of every 128 columns of every row from its fp32 results,
// and stores, in place of the logits, their exponentials relative to each 128-column maximum
// (fp16, scaled by 2^15): half the bytes of fp32 logits, and no exponential left for the row
// pass.  The row
// pass between the GEMMs is this file's kernel: one CTA per row of the chunk merges the row's
// statistics, forms x[idx] in fp32 from the row's hidden state and the head weight, runs the
// forward epilogue, decides the row factor g, and scales the row's exponentials into bf16
// dlogits in place, the operand type of the two backward GEMMs.  The idx element is
// g (1 - p_idx) formed as the complementary sum, as in the unsplit backward.
// grad_hidden's contraction runs over the whole vocabulary, so it is split along K; the
// splits are summed in a fixed order by a small kernel, so results do not depend on timing.
//
// The chunks hold unmasked rows only.  A masked row's outputs and gradients are zero by
// definition, so it is given them once per call and never enters a chunk.  Before each chunk a
// one-CTA kernel picks the next unmasked rows from the device-side mask, and a gather kernel
// copies their hidden states into consecutive rows.  The GEMMs read the chunk's row count from
// the device.  Nothing goes back to the host, so a call can be captured in a CUDA graph and
// follows the mask a replay finds.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include <cuda_fp16.h>

#include "grpo_rowpass.h"
#include "lmhead_gemm.cuh"
#include "rowpass_bwd.cuh"
#include "rowpass_linear.h"

namespace grpo {
namespace {

// Threads of the row-pass CTA (one row each).
constexpr int kLinearThreads = 512;

// The row pass's sweep over one row of the chunk, in place: the logits GEMM left the
// exponentials e_j = 2^(x_j c - a_t) of each 128-column part t (a_t = c max x over the part, the
// statistic's .x) as fp16 scaled by 2^15; with nK = log2|g| - lse log2 e,
// |g| p_j = e_j 2^(a_t + nK), written back as bf16 dlogits d_j = -sign(g) |g| p_j.  Returns
// this thread's share of sum_{j != idx} |g| p_j.
__device__ __forceinline__ float2 unpack_h2(uint32_t w) {
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
}
template <int THREADS, int UNROLL, bool NEG>
__device__ __forceinline__ float linear_sweep_e(uint16_t* row, const float4* __restrict__ st_row, int V, int idx,
                                                float nK, bool& owner) {
  constexpr float kUnscale = -15.f;  // log2 of the exponentials' 2^-15 scale
  const int tid = threadIdx.x;
  uint4* vb = reinterpret_cast<uint4*>(row);
  float q_acc = 0.f;
  float2 q2 = make_float2(0.f, 0.f);
  const int groups = V / 8;  // 8 exponentials (one 16-byte vector) -> 8 dlogits, in place
  auto process = [&](const uint4& w, float a, int i) {
    const float sc = ex2(a + (nK + kUnscale));
    const float2 s2 = make_float2(sc, sc);
    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
    float2 e[BF16::kPairs];
#pragma unroll
    for (int q = 0; q < BF16::kPairs; ++q) e[q] = __fmul2_rn(unpack_h2(wv[q]), s2);
    const unsigned k = static_cast<unsigned>(idx - 8 * i);
    if (k < 8u) {  // this vector holds idx: leave it out of the sum
      owner = true;
#pragma unroll
      for (int q = 0; q < BF16::kPairs; ++q) {
        if (2 * q != static_cast<int>(k)) q_acc += e[q].x;
        if (2 * q + 1 != static_cast<int>(k)) q_acc += e[q].y;
      }
    } else {
#pragma unroll
      for (int q = 0; q < BF16::kPairs; ++q) q2 = __fadd2_rn(q2, e[q]);
    }
    vb[i] = BF16::template pack_pairs<NEG>(e);
  };
  // UNROLL vectors a thread (and their parts' offsets) loaded before any is written back;
  // meanwhile thread 0 asks L2 for the CTA's next step (a bulk prefetch), one step ahead
  constexpr int kStep = UNROLL * THREADS;
  int i = tid;
  for (; i + (UNROLL - 1) * THREADS < groups; i += kStep) {
    if (tid == 0 && i + kStep < groups) {
      const int e = i + 2 * kStep < groups ? i + 2 * kStep : groups;
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(vb + i + kStep),
                   "r"(static_cast<uint32_t>(e - i - kStep) * 16u)
                   : "memory");
    }
    uint4 w[UNROLL];
    float a[UNROLL];
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) w[k] = vb[i + k * THREADS];
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) a[k] = st_row[(i + k * THREADS) >> 4].x;  // 16 vectors a 128-column part
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) process(w[k], a[k], i + k * THREADS);
  }
  for (; i < groups; i += THREADS) process(vb[i], st_row[i >> 4].x, i);
  const int j = 8 * groups + tid;  // the last V % 8 elements
  if (j < V) {
    const __half hj = *reinterpret_cast<const __half*>(row + j);
    const float d = __half2float(hj) * ex2(st_row[j >> 7].x + (nK + kUnscale));
    if (j == idx) owner = true;
    else q_acc += d;
    BF16::store_scalar(row + j, NEG ? -d : d);
  }
  return q_acc + (q2.x + q2.y);
}

// x[idx] of one row: its hidden state times row idx of the head weight, in fp32 (one warp).
// The logits GEMM forms the same value (exact bf16 products, fp32 sums) in another order.
__device__ __forceinline__ float linear_x_idx(const uint16_t* __restrict__ h, const uint16_t* __restrict__ w,
                                              int64_t H, int lane) {
  const uint4* hv = reinterpret_cast<const uint4*>(h);
  const uint4* wv = reinterpret_cast<const uint4*>(w);
  float acc = 0.f;
  for (int64_t k = lane; k < H / 8; k += 32) {
    const uint4 a = hv[k], b = wv[k];
#pragma unroll
    for (int q = 0; q < BF16::kPairs; ++q) {
      const float2 x = BF16::pair(a, q), y = BF16::pair(b, q);
      acc = fmaf(x.x, y.x, acc);
      acc = fmaf(x.y, y.y, acc);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, off);
  return acc;
}

__device__ __forceinline__ void fill_bf16_row(uint16_t* out, int V, uint32_t pair, int nthreads) {
  uint4* ob = reinterpret_cast<uint4*>(out);
  const uint4 v = make_uint4(pair, pair, pair, pair);
  for (int i = threadIdx.x; i < V / 8; i += nthreads) st_v4_evict_first(ob + i, v);
  const int j = (V / 8) * 8 + static_cast<int>(threadIdx.x);
  if (j < V) out[j] = static_cast<uint16_t>(pair & 0xFFFFu);
}

// One CTA per row of the chunk: merge the row's statistics, the forward epilogue and the row
// factor, then one sweep over the row's fp16 exponentials turning them into bf16 dlogits in
// place.  Row i of the chunk is batch row list[i]; the chunk holds state[0] rows, and the rows
// after them up to the next multiple of 64 get zero dlogits, since grad_weight's GEMM reads
// its K (row) dimension in blocks of 64.
template <int THREADS, int UNROLL, bool kH>
__global__ void __launch_bounds__(THREADS) linear_rows_kernel(const LinearChunkParams q) {
  wait_for_previous_grids();
  constexpr int MODE = kH ? kFwdGrpoH : kFwdGrpo;
  const FwdParams& p = q.f;
  const int64_t rl = blockIdx.x;  // row within the chunk
  const int n = q.state[0];
  const int tid = threadIdx.x;
  const int V = p.x.V;
  uint16_t* out = q.dlogits + rl * q.ld;
  if (rl >= n) {
    if (rl < ((static_cast<int64_t>(n) + 63) & ~int64_t(63))) fill_bf16_row(out, V, 0u, THREADS);
    return;
  }
  const int64_t r = q.list[rl];  // row of the batch (never a masked one)
  const int64_t b = r / p.x.L;
  const float c = p.c;

  const int64_t id64 = p.idx[r];
  // the row's scalars for thread 0's epilogue, loaded now so that their latency is hidden
  RowScalars pre{0.f, 0.f, 0.f};
  float pre_dloss = 0.f;
  if (tid == 0) {
    if (p.old_logp) pre.old = p.old_logp[r];
    if (p.beta != 0.f) pre.ref = p.ref_logp[r];
    pre.A = p.adv[b];
    pre_dloss = q.dloss[r];
  }
  const bool bad_idx = id64 < 0 || id64 >= V;
  const int idx = bad_idx ? 0 : static_cast<int>(id64);
  // the selected logit, from the row's hidden state and the head weight (warp 0), while the
  // other warps start on the statistics
  float x_idx = 0.f;
  if (tid < 32 && !bad_idx) x_idx = linear_x_idx(q.hidden_rows + rl * q.H, q.weight + idx * q.H, q.H, tid);

  // the row's statistic: its 128-column parts, merged in a fixed order
  const int n_valid = (V + 127) / 128;
  const float4* st_row = q.stats + rl * q.n_stat;
  Stat mine{-INFINITY, 0.f, 0.f};
  for (int k = tid; k < n_valid; k += THREADS) {
    const float4 e = st_row[k];
    mine = stat_combine(mine, Stat{e.x, e.y, e.z});
  }
  const Stat st = stat_block_reduce<THREADS>(mine);

  __shared__ float sh_g, sh_nK;
  if (tid == 0) {
    float logp = 0.f, lse = 0.f;
    row_epilogue<MODE>(p, r, b, st, c, x_idx, bad_idx, &logp, &lse, &pre);
    const float g = grpo_factor_of(logp, p.old_logp ? pre.old : logp, p.old_logp != nullptr, pre.ref, pre.A,
                                   pre_dloss, p.beta, p.lo, p.hi, q.T);
    sh_g = g;
    sh_nK = fmaf(-lse, kLog2e, log2f(fabsf(g)));  // -(lse*log2e - log2|g|)
  }
  __syncthreads();
  const float g = sh_g;
  if (g == 0.f) {  // early-out: +0.0 over the row, its logits never read
    fill_bf16_row(out, V, 0u, THREADS);
    return;
  }
  if (bad_idx) {
    fill_bf16_row(out, V, BF16::kNaNPair, THREADS);
    return;
  }
  // the sweep: d_j = -sign(g) |g| p_j in bf16, and g (1 - p_idx) at idx
  bool owner = false;
  const float nK = sh_nK;
  const float q_part = g > 0.f ? linear_sweep_e<THREADS, UNROLL, true>(out, st_row, V, idx, nK, owner)
                               : linear_sweep_e<THREADS, UNROLL, false>(out, st_row, V, idx, nK, owner);
  const float q_total = block_sum_all<THREADS>(q_part);
  if (owner) BF16::store_scalar(out + idx, g > 0.f ? q_total : -q_total);
}

// grad_hidden row list[i] = the sum of the K splits of the chunk's row i, in split order,
// for the chunk's state[0] rows.
__global__ void __launch_bounds__(256) split_sum_kernel(const float4* __restrict__ part, float4* __restrict__ out,
                                                        const int32_t* __restrict__ list,
                                                        const int32_t* __restrict__ state, int64_t h4, int splits,
                                                        int64_t split4) {
  wait_for_previous_grids();
  const int64_t n4 = static_cast<int64_t>(state[0]) * h4;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n4; i += int64_t(gridDim.x) * blockDim.x) {
    float4 a = part[i];
    for (int s = 1; s < splits; ++s) {
      const float4 v = part[s * split4 + i];
      a.x += v.x;
      a.y += v.y;
      a.z += v.z;
      a.w += v.w;
    }
    const int64_t rl = i / h4;
    out[static_cast<int64_t>(list[rl]) * h4 + (i - rl * h4)] = a;
  }
}

// Masked rows: their forward outputs and their grad_hidden rows are zero, and nothing else of
// the call touches them (one warp per row).
__global__ void __launch_bounds__(256) linear_masked_kernel(const FwdParams p, float4* __restrict__ grad_hidden,
                                                            int64_t rows, int64_t h4) {
  wait_for_previous_grids();
  const int64_t r = blockIdx.x * int64_t(8) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows || p.mask[r] != 0) return;
  if (lane == 0) masked_row_outputs(p, r);
  if (grad_hidden != nullptr)
    for (int64_t i = lane; i < h4; i += 32) grad_hidden[r * h4 + i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// The rows of the next chunk: up to `chunk` unmasked rows, in batch order, from the batch row
// where the previous chunk stopped (state[1]; row 0 for the first chunk).  One CTA scans the
// mask, 16 rows a thread per pass; state[0] = the rows found, state[1] = the row after the
// last of them (or `rows` when the batch is used up).
constexpr int kSelectThreads = 1024;
__global__ void __launch_bounds__(kSelectThreads) linear_select_kernel(const uint8_t* __restrict__ mask,
                                                                       int64_t rows, int chunk, int first,
                                                                       int32_t* __restrict__ list,
                                                                       int32_t* __restrict__ state) {
  wait_for_previous_grids();
  __shared__ int warp_sum[kSelectThreads / 32];
  __shared__ int sh_total, sh_cursor;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int64_t pos = first ? 0 : state[1];
  int found = 0;
  if (tid == 0) sh_cursor = -1;
  while (pos < rows && found < chunk) {
    const int64_t r0 = pos + 16 * static_cast<int64_t>(tid);
    uint32_t bits = 0;  // bit j: row r0 + j is in the batch and unmasked
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int64_t r = r0 + j;
      if (r < rows && (mask == nullptr || mask[r] != 0)) bits |= 1u << j;
    }
    const int cnt = __popc(bits);
    int incl = cnt;  // inclusive scan over the warp, then over the warps
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int w = warp_sum[lane];
      int wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xFFFFFFFFu, wi, o);
        if (lane >= o) wi += v;
      }
      warp_sum[lane] = wi - w;  // exclusive
      if (lane == 31) sh_total = wi;
    }
    __syncthreads();
    int k = found + warp_sum[warp] + incl - cnt;  // this thread's first slot
    for (uint32_t m = bits; m != 0u; m &= m - 1u) {
      const int j = __ffs(m) - 1;
      if (k < chunk) list[k] = static_cast<int32_t>(r0 + j);
      if (k == chunk - 1) sh_cursor = static_cast<int>(r0 + j + 1);
      ++k;
    }
    found += sh_total;
    pos += 16 * static_cast<int64_t>(kSelectThreads);
    __syncthreads();  // warp_sum and sh_total are rewritten by the next pass
  }
  if (tid == 0) {
    state[0] = found < chunk ? found : chunk;
    state[1] = found < chunk ? static_cast<int32_t>(rows) : sh_cursor;
  }
}

// The chunk's hidden states in consecutive rows: row i = hidden row list[i] for the state[0]
// rows of the chunk, zero after them up to the next multiple of 64 (within the chunk).
__global__ void __launch_bounds__(256) linear_gather_kernel(const uint4* __restrict__ hidden,
                                                            uint4* __restrict__ out,
                                                            const int32_t* __restrict__ list,
                                                            const int32_t* __restrict__ state, int64_t h8,
                                                            int64_t chunk) {
  wait_for_previous_grids();
  const int64_t n = state[0];
  const int64_t upto = std::min(chunk, (n + 63) & ~int64_t(63));
  const int64_t total = upto * h8;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total; i += int64_t(gridDim.x) * blockDim.x) {
    const int64_t rl = i / h8;
    out[i] = rl < n ? hidden[static_cast<int64_t>(list[rl]) * h8 + (i - rl * h8)] : make_uint4(0u, 0u, 0u, 0u);
  }
}

// K splits of grad_hidden's GEMM: as many as the workspace holds (at most 32), picked so
// that the split tiles fill the persistent CTA pairs' passes most evenly.
int grad_hidden_splits(int64_t tiles, int64_t k_blocks, uint64_t part_bytes, uint64_t split_bytes, int pairs) {
  int best = 1;
  double best_eff = 0.0;
  const int64_t cap = std::min<int64_t>(32, std::min<int64_t>(k_blocks, static_cast<int64_t>(part_bytes / split_bytes)));
  for (int s = 1; s <= cap; ++s) {
    const int64_t units = tiles * s;
    const int64_t grid = std::min<int64_t>(units, pairs);
    const int64_t passes = (units + grid - 1) / grid;
    const double eff = static_cast<double>(units) / static_cast<double>(passes * pairs);
    if (eff > best_eff + 1e-3) {
      best_eff = eff;
      best = s;
    }
  }
  return best;
}

}  // namespace

namespace {

// The launches of one fused-linear call: the tensor maps of the head weight and of the chunk
// buffers, made once, and one function per stage of a chunk.  Every chunk is sized for
// q.chunk rows on the host; how many it holds is known only on the device (state[0]), where
// the kernels read it.
struct LinearLauncher {
  const FusedLinearParams& q;
  bool kH;
  int sms;
  CUtensorMap tW_k, tW_mn;  // the head weight K-major (logits) and MN-major (grad_hidden)
  CUtensorMap tHc_k, tHc_mn;  // the chunk's gathered hidden rows: K-major (logits), MN-major (grad_weight)
  CUtensorMap tD_k, tD_mn;  // the chunk's dlogits: K-major (grad_hidden), MN-major (grad_weight)

  explicit LinearLauncher(const FusedLinearParams& params) : q(params) {
    kH = q.chunk_params.f.entropy != nullptr;
    sms = gemm::sm_count();
  }
  bool init() {
    using namespace gemm;
    if (sms <= 0) return false;
    const LinearChunkBufs& b = q.bufs;
    return make_operand_map(&tW_k, q.weight, false, q.V, q.H, q.H, BNH) &&
           make_operand_map(&tW_mn, q.weight, true, q.H, q.V, q.H, BNH) &&
           make_operand_map(&tHc_k, b.hidden, false, q.chunk, q.H, q.H, BM) &&
           make_operand_map(&tHc_mn, b.hidden, true, q.H, q.chunk, q.H, BNH) &&
           make_operand_map(&tD_k, b.dlogits, false, q.chunk, q.V, q.ld, BM) &&
           make_operand_map(&tD_mn, b.dlogits, true, q.V, q.chunk, q.ld, BM);
  }

  // masked rows: zero outputs and zero grad_hidden rows, once per call
  cudaError_t masked(cudaStream_t s) const {
    const FwdParams& f = q.chunk_params.f;
    if (f.mask == nullptr) return cudaSuccess;
    const dim3 grid(static_cast<unsigned>((q.rows + 7) / 8));
    return launch_after_previous(linear_masked_kernel, grid, dim3(256), s, f,
                                 reinterpret_cast<float4*>(q.grad_hidden), q.rows, q.H / 4);
  }

  // the chunk's rows (the next unmasked ones) and their hidden states, gathered
  cudaError_t select(bool first, cudaStream_t s) const {
    const LinearChunkBufs& b = q.bufs;
    cudaError_t e = launch_after_previous(linear_select_kernel, dim3(1), dim3(kSelectThreads), s,
                                          q.chunk_params.f.mask, q.rows, static_cast<int>(q.chunk),
                                          first ? 1 : 0, b.list, b.state);
    if (e != cudaSuccess) return e;
    const int64_t h8 = q.H / 8, n = q.chunk * h8;
    const unsigned blocks = static_cast<unsigned>(std::min<int64_t>((n + 255) / 256, int64_t(sms) * 8));
    return launch_after_previous(linear_gather_kernel, dim3(blocks), dim3(256), s,
                                 reinterpret_cast<const uint4*>(q.hidden), reinterpret_cast<uint4*>(b.hidden),
                                 static_cast<const int32_t*>(b.list), static_cast<const int32_t*>(b.state), h8,
                                 q.chunk);
  }

  // logits [n, V] fp32 = h_chunk W^T, with the statistics of every 128 columns
  cudaError_t logits(cudaStream_t s) const {
    using namespace gemm;
    const LinearChunkBufs& b = q.bufs;
    Params pl{};
    pl.M = static_cast<int>(q.chunk);
    pl.N = static_cast<int>(q.V);
    pl.k_blocks = static_cast<int>((q.H + BK - 1) / BK);
    pl.m_tiles = static_cast<int>((q.chunk + 2 * BM - 1) / (2 * BM));
    pl.n_tiles = static_cast<int>((q.V + BN - 1) / BN);
    pl.splits = 1;
    pl.m_fastest = 1;
    pl.C = reinterpret_cast<float*>(b.dlogits);  // bf16 exponentials (kEpiLogits)
    pl.ldc = q.ld;
    pl.stats = b.stats;
    pl.c = q.chunk_params.f.c;
    pl.err = q.chunk_params.f.dev_err;
    pl.dyn = b.state;
    return kH ? launch_gemm<kEpiLogits, false, false, true>(tHc_k, tW_k, pl, s)
              : launch_gemm<kEpiLogits, false, false, false>(tHc_k, tW_k, pl, s);
  }

  // the row pass: forward outputs and bf16 dlogits of the chunk
  cudaError_t rows(cudaStream_t s) const {
    const LinearChunkBufs& b = q.bufs;
    LinearChunkParams lp = q.chunk_params;
    lp.stats = b.stats;
    lp.hidden_rows = b.hidden;
    lp.weight = q.weight;
    lp.H = q.H;
    lp.dlogits = b.dlogits;
    lp.ld = q.ld;
    lp.n_stat = static_cast<int>(linear_n_stat(q.V));
    lp.list = b.list;
    lp.state = b.state;
    lp.chunk = q.chunk;
    const dim3 grid(static_cast<unsigned>(q.chunk));
    return kH ? launch_after_previous(linear_rows_kernel<kLinearThreads, kUnroll, true>, grid,
                                      dim3(kLinearThreads), s, lp)
              : launch_after_previous(linear_rows_kernel<kLinearThreads, kUnroll, false>, grid,
                                      dim3(kLinearThreads), s, lp);
  }

  // grad_h [n, H] = dlogits W (split along the vocabulary, the splits summed in order into
  // the chunk's rows of grad_hidden) and grad_W [V, H] += dlogits^T h_chunk (vector
  // reduce-adds into the caller's fp32 gradient)
  cudaError_t grads(cudaStream_t s) const {
    using namespace gemm;
    const LinearChunkBufs& b = q.bufs;
    const int64_t H = q.H, V = q.V, c = q.chunk;
    cudaError_t e = cudaSuccess;
    if (q.grad_hidden != nullptr) {
      Params ph{};
      ph.M = static_cast<int>(c);
      ph.N = static_cast<int>(H);
      ph.k_blocks = static_cast<int>((V + BK - 1) / BK);
      ph.m_tiles = static_cast<int>((c + 2 * BM - 1) / (2 * BM));
      ph.n_tiles = static_cast<int>((H + BN - 1) / BN);
      const uint64_t split_bytes = static_cast<uint64_t>(c) * H * 4;
      ph.splits = grad_hidden_splits(int64_t(ph.m_tiles) * ph.n_tiles, ph.k_blocks, q.part_bytes, split_bytes,
                                     sms / 2);
      ph.m_fastest = 1;
      ph.C = q.part;
      ph.ldc = H;
      ph.split_stride = c * H;
      ph.err = q.chunk_params.f.dev_err;
      ph.dyn = b.state;
      e = launch_gemm<kEpiStore, false, true, false>(tD_k, tW_mn, ph, s);
      if (e != cudaSuccess) return e;
      const int64_t h4 = H / 4, n4 = c * h4;
      const unsigned blocks = static_cast<unsigned>(std::min<int64_t>((n4 + 255) / 256, int64_t(sms) * 8));
      e = launch_after_previous(split_sum_kernel, dim3(blocks), dim3(256), s,
                                reinterpret_cast<const float4*>(q.part), reinterpret_cast<float4*>(q.grad_hidden),
                                static_cast<const int32_t*>(b.list), static_cast<const int32_t*>(b.state), h4,
                                ph.splits, n4);
      if (e != cudaSuccess) return e;
    }
    if (q.grad_weight != nullptr) {
      Params pw{};
      pw.M = static_cast<int>(V);
      pw.N = static_cast<int>(H);
      pw.k_blocks = static_cast<int>((c + BK - 1) / BK);
      pw.m_tiles = static_cast<int>((V + 2 * BM - 1) / (2 * BM));
      pw.n_tiles = static_cast<int>((H + BN - 1) / BN);
      pw.splits = 1;
      pw.m_fastest = 0;
      pw.C = q.grad_weight;
      pw.ldc = H;
      pw.err = q.chunk_params.f.dev_err;
      pw.dyn = b.state;
      pw.dyn_k = 1;
      e = launch_gemm<kEpiAccum, true, true, false>(tD_mn, tHc_mn, pw, s);
    }
    return e;
  }
};

}  // namespace

cudaError_t launch_fused_linear(const FusedLinearParams& q, cudaStream_t stream) {
  LinearLauncher run(q);
  if (!run.init()) return cudaErrorInvalidValue;
  // Masked rows are left out of every chunk: their outputs and gradients are zero by
  // definition, so the GEMMs and the row pass see only the unmasked rows, packed into
  // chunks in batch order (the zero-gradient early-out of "LinkedIn Liger-Kernel GRPO Loss
  // Backward optimisation", applied to whole masked rows before their logits exist).  The
  // host sizes the loop for an unmasked batch; chunks past the last unmasked row find no
  // rows on the device and their kernels return at once.
  // (Running a chunk's row pass on a second stream next to its neighbours' GEMMs, with two
  // sets of chunk buffers, measured no faster: the GEMMs and the row pass both lean on the L2
  // and DRAM bandwidth they share.)
  cudaError_t e = run.masked(stream);
  for (int64_t r0 = 0; e == cudaSuccess && r0 < q.rows; r0 += q.chunk) {
    e = run.select(r0 == 0, stream);
    if (e == cudaSuccess) e = run.logits(stream);
    if (e == cudaSuccess) e = run.rows(stream);
    if (e == cudaSuccess) e = run.grads(stream);
  }
  return e;
}

}  // namespace grpo

// ---------------------------------------------------------------------------
// grpo_fused_linear_noalloc: the same computation with its scratch in a fixed device array
// ---------------------------------------------------------------------------
//
// For callers that must not allocate device memory at call time (an allocator-free
// runtime, a host process that has handed all device memory to a pool it does not own, a
// code path that must not synchronise on an allocation).  The scratch grpo_fused_linear
// takes from the caller (one chunk's 16-bit exponentials / dlogits, statistics, gathered hidden
// rows and row list, and the K splits of grad_hidden) lives here in one array of kNoallocScratchBytes, reserved in every
// device context that loads this library and held until the process exits.  Every call uses
// the whole array: calls that run at the same time on the GPU (different streams, threads or
// host processes sharing the context) race on it.  Nothing in it has to start at zero: each
// call writes every part before reading it.

namespace grpo {
namespace {

constexpr uint64_t kNoallocScratchBytes = uint64_t(32) << 20;  // 32 MiB per device

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CUcontext current_context() {
  static const CtxGetCurrentFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<CtxGetCurrentFn>(nullptr);
    return reinterpret_cast<CtxGetCurrentFn>(f);
  }();
  CUcontext ctx = nullptr;
  if (fn == nullptr || fn(&ctx) != CUDA_SUCCESS) return nullptr;
  return ctx;
}

// The array's device address, looked up with the device current the first time a device
// (context) calls, and again whenever the device's context has changed since (a
// cudaDeviceReset makes a new one, where the array lives at a new address).
void* noalloc_scratch_address() {
  struct Entry {
    CUcontext ctx;
    void* addr;
  };
  static Entry cache[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  cudaFree(nullptr);  // makes the device's primary context current (allocates nothing)
  const CUcontext ctx = current_context();
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev].addr == nullptr || cache[dev].ctx != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
    cache[dev] = Entry{ctx, p};
  }
  return cache[dev].addr;
}

bool noalloc_f32(const void* p, bool required) {
  return p == nullptr ? !required : (reinterpret_cast<uintptr_t>(p) % 4) == 0;
}

}  // namespace
}  // namespace grpo

extern "C" grpo_status grpo_fused_linear_noalloc(
    const void* hidden, const void* weight, int64_t B, int64_t L, int64_t H, int64_t V, const int64_t* idx,
    const float* old_logp, const float* ref_logp, const float* adv, const uint8_t* mask, const float* dloss, float T,
    float beta, float eps_low, float eps_high, int64_t chunk_rows, float* loss, float* logp, float* lse, float* kl,
    uint8_t* is_clipped, float* entropy, float* grad_hidden, float* grad_weight, int32_t* dev_err,
    grpo_stream_t stream) {
  using grpo::noalloc_f32;
  // the arguments, checked as grpo_fused_linear checks them, before any CUDA call
  if (!(std::isfinite(T) && T > 0.f) || !std::isfinite(beta) || beta < 0.f || !std::isfinite(eps_low) ||
      eps_low < 0.f || eps_low > 1.f || !std::isfinite(eps_high) || eps_high < 0.f)
    return GRPO_ERR_INVALID_ARG;
  if (B < 0 || L < 0 || H < 8 || H % 8 != 0 || V < 1 || chunk_rows < 1) return GRPO_ERR_INVALID_ARG;
  if (V > (int64_t(1) << 30) || static_cast<long double>(B) * L > ((int64_t(1) << 31) - 1) || H > (int64_t(1) << 24))
    return GRPO_ERR_UNSUPPORTED;
  const int64_t rows = B * L;
  if (rows == 0) return GRPO_OK;
  const int64_t chunk = chunk_rows < rows ? chunk_rows : rows;
  // the fixed array's limit: the chunk's buffers (16-bit exponentials / dlogits, statistics,
  // gathered bf16 hidden rows, row list and state, each rounded up to 256 bytes) and one
  // split of grad_hidden (chunk * H fp32) <= 32 MiB
  const uint64_t chunk_bytes = grpo::linear_chunk_bytes(H, V, chunk);
  if (chunk_bytes + static_cast<uint64_t>(chunk) * H * 4 > grpo::kNoallocScratchBytes) return GRPO_ERR_UNSUPPORTED;
  auto a16 = [](const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) % 16) == 0; };
  if (!a16(hidden) || !a16(weight)) return GRPO_ERR_INVALID_ARG;
  if (idx == nullptr || (reinterpret_cast<uintptr_t>(idx) % 8) != 0 || !noalloc_f32(old_logp, false) ||
      !noalloc_f32(adv, true) || !noalloc_f32(dloss, true) || !noalloc_f32(loss, true) || !noalloc_f32(logp, true) ||
      !noalloc_f32(lse, true) || !noalloc_f32(kl, false) || !noalloc_f32(entropy, false) ||
      !noalloc_f32(dev_err, false))
    return GRPO_ERR_INVALID_ARG;
  if ((grad_hidden != nullptr && !a16(grad_hidden)) || (grad_weight != nullptr && !a16(grad_weight)))
    return GRPO_ERR_INVALID_ARG;
  if (beta != 0.f && !noalloc_f32(ref_logp, true)) return GRPO_ERR_INVALID_ARG;
  if (!noalloc_f32(ref_logp, false)) return GRPO_ERR_INVALID_ARG;

  // set-up on this device's first call (and after a device reset): the array's address
  char* scratch = static_cast<char*>(grpo::noalloc_scratch_address());
  if (scratch == nullptr) return GRPO_ERR_CUDA;

  grpo::FusedLinearParams q{};
  q.hidden = static_cast<const uint16_t*>(hidden);
  q.weight = static_cast<const uint16_t*>(weight);
  q.rows = rows;
  q.H = H;
  q.V = V;
  q.chunk = chunk;
  q.ld = grpo::linear_ld(V);
  grpo::linear_carve(q, scratch, grpo::kNoallocScratchBytes);
  q.grad_hidden = grad_hidden;
  q.grad_weight = grad_weight;
  grpo::LinearChunkParams& cp = q.chunk_params;
  grpo::FwdParams& p = cp.f;
  p.x = grpo::RowsView{nullptr, L, 0, 0, static_cast<int>(V)};
  p.idx = idx;
  p.old_logp = old_logp;
  p.ref_logp = ref_logp;
  p.adv = adv;
  p.mask = mask;
  p.c = static_cast<float>(1.4426950408889634074 / static_cast<double>(T));
  p.invT = static_cast<float>(1.0 / static_cast<double>(T));
  p.beta = beta;
  p.lo = static_cast<float>(1.0 - static_cast<double>(eps_low));
  p.hi = static_cast<float>(1.0 + static_cast<double>(eps_high));
  p.loss = loss;
  p.logp = logp;
  p.lse = lse;
  p.kl = kl;
  p.is_clipped = is_clipped;
  p.entropy = entropy;
  p.dev_err = dev_err;
  cp.dloss = dloss;
  cp.T = T;
  return grpo::launch_fused_linear(q, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? GRPO_OK
                                                                                              : GRPO_ERR_CUDA;
}
