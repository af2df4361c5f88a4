// The GRPO loss on top of the LM head, in chunks of rows ("Liger GRPO meets TRL",
// sections 3 and 4): for each chunk of rows, its logits x = h W^T are formed, the row pass
// turns them into the loss, the forward outputs and dlogits, and the gradients of the
// chunk's hidden states (dlogits W) and of the head weight (+= dlogits^T h) are formed
// before the next chunk, so the logits of the whole batch never exist at once.
//
// The three contractions are plain GEMMs on the tensor cores through cuBLASLt (bf16
// operands, fp32 accumulation).  The row pass between them is this file's kernel: one CTA
// per row of the chunk reads the chunk's fp32 logits (just written, mostly from L2) for
// the online statistic and the epilogue, decides the row factor g, and sweeps the row again
// to write dlogits in bf16, the operand type of the two backward GEMMs.  The idx element
// is g (1 - p_idx) formed as the complementary sum, as in the unsplit backward.
#include <cublasLt.h>

#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "grpo_rowpass.h"
#include "rowpass_bwd.cuh"
#include "rowpass_fwd.cuh"

namespace grpo {
namespace {

// Row pass over one chunk: fp32 logits [rows][ld] in, bf16 dlogits [rows][ld] out.
template <int THREADS, int UNROLL, bool kH, bool NEG>
__device__ __forceinline__ float linear_sweep2(const float* row, uint16_t* out, int V, int idx, float c, float nK,
                                               bool& owner) {
  const int tid = threadIdx.x;
  const uint4* vb = reinterpret_cast<const uint4*>(row);
  uint4* ob = reinterpret_cast<uint4*>(out);
  const float2 c2 = make_float2(c, c), nK2 = make_float2(nK, nK);
  float q_acc = 0.f;
  float2 q2 = make_float2(0.f, 0.f);
  const int groups = V / 8;  // 8 logits (two 16-byte fp32 vectors) -> one 16-byte bf16 vector
  for (int i = tid; i < groups; i += THREADS) {
    const uint4 a = ld_v4_evict_first(vb + 2 * i), b = ld_v4_evict_first(vb + 2 * i + 1);
    float2 e[4];
    const float2 x[4] = {make_float2(__uint_as_float(a.x), __uint_as_float(a.y)),
                         make_float2(__uint_as_float(a.z), __uint_as_float(a.w)),
                         make_float2(__uint_as_float(b.x), __uint_as_float(b.y)),
                         make_float2(__uint_as_float(b.z), __uint_as_float(b.w))};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 t = __ffma2_rn(x[q], c2, nK2);
      e[q] = make_float2(ex2(t.x), ex2(t.y));
    }
    const unsigned k = static_cast<unsigned>(idx - 8 * i);
    if (k < 8u) {  // this group holds idx: leave it out of the sum
      owner = true;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (2 * q != static_cast<int>(k)) q_acc += e[q].x;
        if (2 * q + 1 != static_cast<int>(k)) q_acc += e[q].y;
      }
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) q2 = __fadd2_rn(q2, e[q]);
    }
    st_v4_evict_first(ob + i, BF16::pack_pairs<NEG>(e));
  }
  const int j = 8 * groups + tid;  // the last V % 8 elements
  if (j < V) {
    const float e = ex2(fmaf(row[j], c, nK));
    if (j == idx) owner = true;
    else q_acc += e;
    BF16::store_scalar(out + j, NEG ? -e : e);
  }
  return q_acc + (q2.x + q2.y);
}

__device__ __forceinline__ void fill_bf16_row(uint16_t* out, int V, uint32_t pair, int nthreads) {
  uint4* ob = reinterpret_cast<uint4*>(out);
  const uint4 v = make_uint4(pair, pair, pair, pair);
  for (int i = threadIdx.x; i < V / 8; i += nthreads) st_v4_evict_first(ob + i, v);
  const int j = (V / 8) * 8 + static_cast<int>(threadIdx.x);
  if (j < V) out[j] = static_cast<uint16_t>(pair & 0xFFFFu);
}

template <int THREADS, int UNROLL, bool kH>
__global__ void __launch_bounds__(THREADS) linear_chunk_kernel(const LinearChunkParams q) {
  wait_for_previous_grids();
  constexpr int MODE = kH ? kFwdGrpoH : kFwdGrpo;
  const FwdParams& p = q.f;
  const int64_t rl = blockIdx.x;  // row within the chunk
  const int64_t r = q.row0 + rl;  // row of the batch
  const int64_t b = r / p.x.L;
  const int tid = threadIdx.x;
  const int V = p.x.V;
  const float c = p.c;
  const float* row = q.logits + rl * q.ld;
  uint16_t* out = q.dlogits + rl * q.ld;

  const int64_t id64 = p.idx[r];  // loaded with the mask, before either is waited on
  if (p.mask != nullptr && p.mask[r] == 0) {  // masked token: zero outputs, zero gradient row
    if (tid == 0) masked_row_outputs(p, r);
    fill_bf16_row(out, V, 0u, THREADS);
    return;
  }
  const bool bad_idx = id64 < 0 || id64 >= V;
  const int idx = bad_idx ? 0 : static_cast<int>(id64);

  // sweep 1: the online statistic of the fp32 row (16-byte aligned: ld % 8 == 0).  The row
  // is kept in L2 (evict_last) for sweep 2, which lets it go (evict_first); one CTA of 1024
  // threads per SM keeps some 150 rows in flight, few enough for L2 to hold them.
  Running rs{-INFINITY, 0.f, make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  const uint4* vb = reinterpret_cast<const uint4*>(row);
  const int nvec = V / 4;
  if (tid < V - 4 * nvec) run_scalar<kH>(rs, row[4 * nvec + tid], c);
  int i = tid;
  for (; i + (UNROLL - 1) * THREADS < nvec; i += UNROLL * THREADS) {
    uint4 v[UNROLL];
#pragma unroll
    for (int k = 0; k < UNROLL; ++k) v[k] = ld_v4_evict_last(vb + i + k * THREADS);
    run_vectors<F32, kH>(rs, v, c);
  }
  for (; i < nvec; i += THREADS) {
    uint4 v[1];
    v[0] = ld_v4_evict_last(vb + i);
    run_vectors<F32, kH>(rs, v, c);
  }
  const float x_idx = tid == 0 ? row[idx] : 0.f;
  Stat mine;
  mine.a = rs.a;
  mine.s = rs.s.x + rs.s.y;
  mine.u = rs.u.x + rs.u.y;
  const Stat st = stat_block_reduce<THREADS>(mine);

  __shared__ float sh_g, sh_nK;
  if (tid == 0) {
    float logp = 0.f, lse = 0.f;
    row_epilogue<MODE>(p, r, b, st, c, x_idx, bad_idx, &logp, &lse);
    const float g = grpo_factor(logp, p.old_logp, p.ref_logp, p.adv[b], q.dloss[r], p.beta, p.lo, p.hi, q.T, r);
    sh_g = g;
    sh_nK = fmaf(-lse, kLog2e, log2f(fabsf(g)));  // -(lse*log2e - log2|g|)
  }
  __syncthreads();
  const float g = sh_g;
  if (g == 0.f) {  // early-out: +0.0 over the row
    fill_bf16_row(out, V, 0u, THREADS);
    l2_demote<THREADS>(row, static_cast<int64_t>(V) * 4);
    return;
  }
  if (bad_idx) {
    fill_bf16_row(out, V, BF16::kNaNPair, THREADS);
    l2_demote<THREADS>(row, static_cast<int64_t>(V) * 4);
    return;
  }
  // sweep 2: d_j = -sign(g) |g| p_j in bf16, and g (1 - p_idx) at idx
  bool owner = false;
  const float nK = sh_nK;
  const float q_part = g > 0.f ? linear_sweep2<THREADS, UNROLL, kH, true>(row, out, V, idx, c, nK, owner)
                               : linear_sweep2<THREADS, UNROLL, kH, false>(row, out, V, idx, c, nK, owner);
  const float q_total = block_sum_all<THREADS>(q_part);
  if (owner) BF16::store_scalar(out + idx, g > 0.f ? q_total : -q_total);
}

// ---------------------------------------------------------------------------
// cuBLASLt: one handle per device, the heuristic's algorithm cached per problem
// ---------------------------------------------------------------------------

struct LtHandle {
  cublasLtHandle_t h = nullptr;
  bool ok = false;
};

cublasLtHandle_t lt_handle() {
  static LtHandle handles[64];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!handles[dev].ok) {
    if (cublasLtCreate(&handles[dev].h) != CUBLAS_STATUS_SUCCESS) return nullptr;
    handles[dev].ok = true;
  }
  return handles[dev].h;
}

// Column-major D[m, n] = alpha op(A) op(B) + beta C (C = D), A, B bf16, D fp32 or bf16,
// fp32 accumulation.
struct GemmKey {
  int dev, ta, tb, dtype_d;
  int64_t m, n, k, lda, ldb, ldd;
  size_t ws;
  bool operator<(const GemmKey& o) const {
    return std::tie(dev, ta, tb, dtype_d, m, n, k, lda, ldb, ldd, ws) <
           std::tie(o.dev, o.ta, o.tb, o.dtype_d, o.m, o.n, o.k, o.lda, o.ldb, o.ldd, o.ws);
  }
};

cudaError_t lt_gemm(bool ta, bool tb, int64_t m, int64_t n, int64_t k, const void* A, int64_t lda, const void* B,
                    int64_t ldb, void* D, int64_t ldd, cudaDataType_t dtype_d, float beta, void* ws,
                    size_t ws_bytes, cudaStream_t stream) {
  cublasLtHandle_t h = lt_handle();
  if (h == nullptr) return cudaErrorNotSupported;
  cublasLtMatmulDesc_t op = nullptr;
  cublasLtMatrixLayout_t la = nullptr, lb = nullptr, ld = nullptr;
  cudaError_t err = cudaErrorUnknown;
  const cublasOperation_t opa = ta ? CUBLAS_OP_T : CUBLAS_OP_N, opb = tb ? CUBLAS_OP_T : CUBLAS_OP_N;
  do {
    if (cublasLtMatmulDescCreate(&op, CUBLAS_COMPUTE_32F, CUDA_R_32F) != CUBLAS_STATUS_SUCCESS) break;
    if (cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSA, &opa, sizeof(opa)) != CUBLAS_STATUS_SUCCESS) break;
    if (cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSB, &opb, sizeof(opb)) != CUBLAS_STATUS_SUCCESS) break;
    if (cublasLtMatrixLayoutCreate(&la, CUDA_R_16BF, ta ? k : m, ta ? m : k, lda) != CUBLAS_STATUS_SUCCESS) break;
    if (cublasLtMatrixLayoutCreate(&lb, CUDA_R_16BF, tb ? n : k, tb ? k : n, ldb) != CUBLAS_STATUS_SUCCESS) break;
    if (cublasLtMatrixLayoutCreate(&ld, dtype_d, m, n, ldd) != CUBLAS_STATUS_SUCCESS) break;
    int dev = 0;
    cudaGetDevice(&dev);
    const GemmKey key{dev, ta, tb, static_cast<int>(dtype_d), m, n, k, lda, ldb, ldd, ws_bytes};
    static std::map<GemmKey, cublasLtMatmulAlgo_t> cache;
    static std::mutex mu;
    cublasLtMatmulAlgo_t algo;
    bool have = false;
    {
      std::lock_guard<std::mutex> lock(mu);
      auto it = cache.find(key);
      if (it != cache.end()) {
        algo = it->second;
        have = true;
      }
    }
    if (!have) {
      cublasLtMatmulPreference_t pref = nullptr;
      if (cublasLtMatmulPreferenceCreate(&pref) != CUBLAS_STATUS_SUCCESS) break;
      cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &ws_bytes,
                                           sizeof(ws_bytes));
      cublasLtMatmulHeuristicResult_t res;
      int found = 0;
      const cublasStatus_t hs = cublasLtMatmulAlgoGetHeuristic(h, op, la, lb, ld, ld, pref, 1, &res, &found);
      cublasLtMatmulPreferenceDestroy(pref);
      if (hs != CUBLAS_STATUS_SUCCESS || found < 1) {
        err = cudaErrorNotSupported;
        break;
      }
      algo = res.algo;
      std::lock_guard<std::mutex> lock(mu);
      cache[key] = algo;
    }
    const float alpha = 1.f;
    const cublasStatus_t s = cublasLtMatmul(h, op, &alpha, A, la, B, lb, &beta, D, ld, D, ld, &algo, ws, ws_bytes,
                                            stream);
    err = s == CUBLAS_STATUS_SUCCESS ? cudaSuccess : cudaErrorLaunchFailure;
  } while (false);
  if (ld) cublasLtMatrixLayoutDestroy(ld);
  if (lb) cublasLtMatrixLayoutDestroy(lb);
  if (la) cublasLtMatrixLayoutDestroy(la);
  if (op) cublasLtMatmulDescDestroy(op);
  return err;
}

}  // namespace

cudaError_t launch_fused_linear(const FusedLinearParams& q, cudaStream_t stream) {
  const int64_t R = q.rows, H = q.H, V = q.V, ld = q.ld;
  for (int64_t r0 = 0; r0 < R; r0 += q.chunk) {
    const int64_t c = R - r0 < q.chunk ? R - r0 : q.chunk;
    const uint16_t* h = q.hidden + r0 * H;
    // logits^T [V, c] (column-major, ld) = W [V, H] h^T: W is the column-major [H, V] matrix
    cudaError_t e = lt_gemm(true, false, V, c, H, q.weight, H, h, H, q.logits, ld, CUDA_R_32F, 0.f, q.ws,
                            q.ws_bytes, stream);
    if (e != cudaSuccess) return e;
    LinearChunkParams lp = q.chunk_params;
    lp.row0 = r0;
    const dim3 grid(static_cast<unsigned>(c));
    e = lp.f.entropy ? launch_after_previous(linear_chunk_kernel<1024, kUnroll, true>, grid, dim3(1024), stream, lp)
                     : launch_after_previous(linear_chunk_kernel<1024, kUnroll, false>, grid, dim3(1024), stream, lp);
    if (e != cudaSuccess) return e;
    if (q.grad_hidden != nullptr) {
      // grad_h^T [H, c] = W^T-as-[H, V] x dlogits^T [V, c]
      e = lt_gemm(false, false, H, c, V, q.weight, H, q.dlogits, ld, q.grad_hidden + r0 * H, H, CUDA_R_32F, 0.f,
                  q.ws, q.ws_bytes, stream);
      if (e != cudaSuccess) return e;
    }
    if (q.grad_weight != nullptr) {
      // grad_W^T [H, V] += h^T [H, c] x dlogits [c, V]
      e = lt_gemm(false, true, H, V, c, h, H, q.dlogits, ld, q.grad_weight, H, CUDA_R_32F, 1.f, q.ws,
                  q.ws_bytes, stream);
      if (e != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

}  // namespace grpo

// ---------------------------------------------------------------------------
// grpo_fused_linear_noalloc: the same computation with its scratch in a fixed device array
// ---------------------------------------------------------------------------
//
// For callers that must not allocate device memory at call time (an allocator-free
// runtime, a host process that has handed all device memory to a pool it does not own, a
// code path that must not synchronise on an allocation).  The scratch grpo_fused_linear
// takes from the caller (one chunk's fp32 logits and bf16 dlogits, and the GEMMs'
// workspace) lives here in one array of kNoallocScratchBytes, reserved in every device
// context that loads this library and held until the process exits.  Every call uses the
// whole array: calls that run at the same time on the GPU (different streams, threads or
// host processes sharing the context) race on it.  Nothing in it has to start at zero: each
// call writes every part before reading it.

namespace grpo {
namespace {

constexpr uint64_t kNoallocScratchBytes = uint64_t(32) << 20;  // 32 MiB per device
constexpr uint64_t kNoallocGemmWs = uint64_t(4) << 20;         // of which the GEMMs' workspace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

// The array's device address, looked up once per device with that device current.
void* noalloc_scratch_address() {
  static void* addr[64] = {nullptr};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

// lt_gemm with its descriptors in caller-provided (stack) storage and the chosen
// algorithms in a fixed table, so that a call allocates nothing, on the host either.
cudaError_t lt_gemm_noalloc(bool ta, bool tb, int64_t m, int64_t n, int64_t k, const void* A, int64_t lda,
                            const void* B, int64_t ldb, void* D, int64_t ldd, float beta, void* ws, size_t ws_bytes,
                            cudaStream_t stream) {
  cublasLtHandle_t h = lt_handle();
  if (h == nullptr) return cudaErrorNotSupported;
  cublasLtMatmulDescOpaque_t op_s;
  cublasLtMatrixLayoutOpaque_t la_s, lb_s, ld_s;
  cublasLtMatmulDesc_t op = &op_s;
  cublasLtMatrixLayout_t la = &la_s, lb = &lb_s, ldl = &ld_s;
  const cublasOperation_t opa = ta ? CUBLAS_OP_T : CUBLAS_OP_N, opb = tb ? CUBLAS_OP_T : CUBLAS_OP_N;
  if (cublasLtMatmulDescInit(op, CUBLAS_COMPUTE_32F, CUDA_R_32F) != CUBLAS_STATUS_SUCCESS ||
      cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSA, &opa, sizeof(opa)) != CUBLAS_STATUS_SUCCESS ||
      cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSB, &opb, sizeof(opb)) != CUBLAS_STATUS_SUCCESS ||
      cublasLtMatrixLayoutInit(la, CUDA_R_16BF, ta ? k : m, ta ? m : k, lda) != CUBLAS_STATUS_SUCCESS ||
      cublasLtMatrixLayoutInit(lb, CUDA_R_16BF, tb ? n : k, tb ? k : n, ldb) != CUBLAS_STATUS_SUCCESS ||
      cublasLtMatrixLayoutInit(ldl, CUDA_R_32F, m, n, ldd) != CUBLAS_STATUS_SUCCESS)
    return cudaErrorNotSupported;
  int dev = 0;
  cudaGetDevice(&dev);
  const GemmKey key{dev, ta, tb, static_cast<int>(CUDA_R_32F), m, n, k, lda, ldb, ldd, ws_bytes};
  struct Entry {
    GemmKey key;
    cublasLtMatmulAlgo_t algo;
    bool used;
  };
  static Entry table[64];
  static int next = 0;
  static std::mutex mu;
  cublasLtMatmulAlgo_t algo;
  bool have = false;
  {
    std::lock_guard<std::mutex> lock(mu);
    for (const Entry& e : table)
      if (e.used && !(e.key < key) && !(key < e.key)) {
        algo = e.algo;
        have = true;
        break;
      }
  }
  if (!have) {
    cublasLtMatmulPreferenceOpaque_t pref_s;
    cublasLtMatmulPreference_t pref = &pref_s;
    if (cublasLtMatmulPreferenceInit(pref) != CUBLAS_STATUS_SUCCESS) return cudaErrorNotSupported;
    cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &ws_bytes,
                                         sizeof(ws_bytes));
    cublasLtMatmulHeuristicResult_t res;
    int found = 0;
    if (cublasLtMatmulAlgoGetHeuristic(h, op, la, lb, ldl, ldl, pref, 1, &res, &found) != CUBLAS_STATUS_SUCCESS ||
        found < 1)
      return cudaErrorNotSupported;
    algo = res.algo;
    std::lock_guard<std::mutex> lock(mu);
    table[next] = Entry{key, algo, true};  // a fixed table: the oldest entry makes room
    next = (next + 1) % 64;
  }
  const float alpha = 1.f;
  return cublasLtMatmul(h, op, &alpha, A, la, B, lb, &beta, D, ldl, D, ldl, &algo, ws, ws_bytes, stream) ==
                 CUBLAS_STATUS_SUCCESS
             ? cudaSuccess
             : cudaErrorLaunchFailure;
}

cudaError_t launch_fused_linear_noalloc(const FusedLinearParams& q, cudaStream_t stream) {
  const int64_t R = q.rows, H = q.H, V = q.V, ld = q.ld;
  for (int64_t r0 = 0; r0 < R; r0 += q.chunk) {
    const int64_t c = R - r0 < q.chunk ? R - r0 : q.chunk;
    const uint16_t* h = q.hidden + r0 * H;
    cudaError_t e = lt_gemm_noalloc(true, false, V, c, H, q.weight, H, h, H, q.logits, ld, 0.f, q.ws, q.ws_bytes,
                                    stream);
    if (e != cudaSuccess) return e;
    LinearChunkParams lp = q.chunk_params;
    lp.row0 = r0;
    const dim3 grid(static_cast<unsigned>(c));
    e = lp.f.entropy ? launch_after_previous(linear_chunk_kernel<1024, kUnroll, true>, grid, dim3(1024), stream, lp)
                     : launch_after_previous(linear_chunk_kernel<1024, kUnroll, false>, grid, dim3(1024), stream, lp);
    if (e != cudaSuccess) return e;
    if (q.grad_hidden != nullptr) {
      e = lt_gemm_noalloc(false, false, H, c, V, q.weight, H, q.dlogits, ld, q.grad_hidden + r0 * H, H, 0.f, q.ws,
                          q.ws_bytes, stream);
      if (e != cudaSuccess) return e;
    }
    if (q.grad_weight != nullptr) {
      e = lt_gemm_noalloc(false, true, H, V, c, h, H, q.dlogits, ld, q.grad_weight, H, 1.f, q.ws, q.ws_bytes,
                          stream);
      if (e != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
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
  const int64_t ld = (V + 7) / 8 * 8;
  const int64_t chunk = chunk_rows < rows ? chunk_rows : rows;
  const uint64_t logits_bytes = (static_cast<uint64_t>(ld) * chunk * 4 + 255) & ~uint64_t(255);
  const uint64_t dlogits_bytes = (static_cast<uint64_t>(ld) * chunk * 2 + 255) & ~uint64_t(255);
  // the fixed array's limit: chunk * 6 * ld bytes (rounded to 256) + the GEMMs' 4 MiB <= 32 MiB
  if (logits_bytes + dlogits_bytes + grpo::kNoallocGemmWs > grpo::kNoallocScratchBytes) return GRPO_ERR_UNSUPPORTED;
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

  // set-up on this device's first call: the array's address (and the library's cuBLASLt
  // handle for the device, created on first use by every GEMM path of this library)
  char* scratch = static_cast<char*>(grpo::noalloc_scratch_address());
  if (scratch == nullptr) return GRPO_ERR_CUDA;

  grpo::FusedLinearParams q{};
  q.hidden = static_cast<const uint16_t*>(hidden);
  q.weight = static_cast<const uint16_t*>(weight);
  q.rows = rows;
  q.H = H;
  q.V = V;
  q.chunk = chunk;
  q.ld = ld;
  q.logits = reinterpret_cast<float*>(scratch);
  q.dlogits = reinterpret_cast<uint16_t*>(scratch + logits_bytes);
  q.ws = scratch + logits_bytes + dlogits_bytes;
  q.ws_bytes = grpo::kNoallocGemmWs;
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
  cp.logits = q.logits;
  cp.dlogits = q.dlogits;
  cp.ld = ld;
  cp.dloss = dloss;
  cp.T = T;
  return grpo::launch_fused_linear_noalloc(q, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? GRPO_OK
             : GRPO_ERR_CUDA;
}
