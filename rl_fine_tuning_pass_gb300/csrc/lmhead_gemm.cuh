// The three contractions of the GRPO loss on top of the LM head ("Liger GRPO meets TRL",
// sections 3 and 4: the chunk's logits are its hidden states times the head weight, and the
// gradients of the hidden states and of the head weight are formed from the chunk's
// dlogits), as one tcgen05 GEMM kernel for sm_103a:
//
//   D[M, N] = A[M, K] B[K, N]    bf16 operands, fp32 accumulation in tensor memory
//
// with three epilogues:
//   kEpiLogits  D is the chunk's logits (M = rows, N = V, K = H), kept in registers: each
//               tile forms the softmax statistic (a, s, u) of each half (128 columns) of
//               every row, a = c max x_j, and stores, in place of the logits, the
//               exponentials e_j = 2^(x_j c - a) as fp16 scaled by 2^15 (C is then a 16-bit
//               matrix), half the bytes of fp32 logits.  The row pass turns them into bf16
//               dlogits in place: |g| p_j = e_j 2^(a - lse log2 e + log2 |g|);
//   kEpiStore   D is stored (one K split of grad_hidden: M = rows, N = H, K = V);
//   kEpiAccum   D is added to the fp32 output (grad_weight += dlogits^T h: M = V, N = H,
//               K = rows) by TMA reduce-adds.
//
// Layout and pipeline.  The kernel runs on pairs of CTAs (a cluster of two SMs); a pair
// computes one 256 x 256 output tile at a time with tcgen05.mma.cta_group::2 (M = 256,
// N = 256, K = 16): each CTA stages its 128 rows of A and its 128 columns of B, so each SM
// moves a third less operand data through shared memory than a one-SM 128 x 256 tile would.
// In each CTA, warp 0 streams that CTA's halves with TMA into a 6-stage ring of
// 128-byte-swizzled tiles (64 K-elements deep: 16 KB of A and 16 KB of B), signalling the
// pair's leader (cluster rank 0); warp 1 holds 512 TMEM columns (two 256-column fp32
// accumulators, allocated for the pair), and one thread of the leader's warp 1 issues the
// MMAs and commits them to both CTAs' barriers.  Warps 2-9 of each CTA read its 128 rows
// of the finished accumulator back with tcgen05.ld (a warp reaches the 32 TMEM lanes of its
// quarter; two warps share a quarter, one for each half of the columns) while the MMAs of
// the next tile fill the other accumulator.  Each warp passes its 32 x 32 boxes through a
// swizzled staging buffer (one row per lane in) and hands it to the TMA: kEpiLogits (16-bit
// boxes, 64-byte swizzle) and kEpiStore (fp32 boxes, 128-byte swizzle, one split per z) by a
// tensor store, kEpiAccum by a tensor reduce-add (the buffer's swizzle is the tensor map's).
// That is one instruction where a lane's shared loads and global stores (or 16 vector
// reduce-adds) were; the fewer instructions the epilogue warps issue, the less they slow the
// MMA thread that shares an SM sub-partition with two of them.  Operands may be K-major (K contiguous: h, W in the logits GEMM, dlogits in
// grad_hidden) or MN-major (M or N contiguous: W in grad_hidden, dlogits^T and h in
// grad_weight); the MN-major tiles are loaded as 64-wide boxes and described to the MMA
// with the MN-major bit.
//
// Every wait on an mbarrier gives up after about two seconds: it sets the CTA's abort flag,
// every role leaves its loop, the in-flight copies and MMAs are waited for (again with a
// limit), both CTAs of the pair meet at a cluster barrier, TMEM is freed and the kernel
// returns with GRPO_DEVERR_TIMEOUT_BIT set in the caller's error word.  Nothing traps.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "rowpass_fwd.cuh"

namespace grpo {
namespace gemm {

constexpr int BM = 128;     // rows of a CTA's half tile (TMEM lanes); the pair's tile has 2 BM
constexpr int BN = 256;     // columns of a tile (TMEM columns of one accumulator)
constexpr int BNH = BN / 2;  // columns of B each CTA of the pair stages
constexpr int BK = 64;      // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int kStages = 6;
constexpr int kEpiWarps = 8;   // two per TMEM lane quarter, each half of the tile's columns
constexpr int kThreads = 32 * (2 + kEpiWarps);  // warp 0 TMA, warp 1 MMA, warps 2-9 epilogue
constexpr uint32_t kStageA = BM * BK * 2;   // 16 KB
constexpr uint32_t kStageB = BNH * BK * 2;  // 16 KB
constexpr uint32_t kTmemCols = 2 * BN;
constexpr uint32_t kStageC = 32 * 32 * 4;        // one epilogue warp's 32 x 32 fp32 output box
constexpr uint32_t kSmemC = kEpiWarps * kStageC;  // one staging box per epilogue warp
constexpr uint32_t kBarBytes = 256;
constexpr uint32_t kSmemBytes = 1024 + kStages * (kStageA + kStageB) + kSmemC + kBarBytes;
constexpr long long kWaitCycles = 4000000000LL;  // about 2 s at 2 GHz

enum Epi : int { kEpiLogits = 0, kEpiStore = 1, kEpiAccum = 2 };

struct Params {
  int M, N;            // output rows and columns
  int k_blocks;        // ceil(K / 64)
  int m_tiles, n_tiles, splits;  // m_tiles counts the pair's 256-row tiles
  int m_fastest;       // 1: consecutive tiles share a B tile; 0: share an A tile
  float* C;            // fp32 output [M][ldc] (+ split * split_stride); ldc a multiple of 4
                       // (kEpiLogits: 16-bit [M][ldc], ldc a multiple of 8)
  int64_t ldc, split_stride;
  // kEpiLogits only
  float4* stats;       // [M][2 n_tiles]: (a, s, u, 0) of each half tile's 128 columns
  float c;             // log2(e) / T
  int* err;            // device error word (nullable)
  int pair_limit;      // at most this many CTA pairs (0: as many as fit on the GPU)
  // A extent known only on the device (the rows a chunk holds after the masked rows are
  // left out), read when the kernel starts, after the grids before it have completed:
  // null, or *dyn rows (dyn_k = 0: M = min(M, *dyn), m_tiles follows) or *dyn K elements
  // (dyn_k = 1: k_blocks = ceil(*dyn / 64); splits must be 1).  M and m_tiles (k_blocks)
  // above are then the upper bounds the launch is sized for.  Zero rows or zero K blocks:
  // no tiles.
  const int32_t* dyn;
  int dyn_k;
};

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for the phase of parity `parity` to complete.  Gives up (false) when the CTA's abort
// flag is set (if honor_abort) or after kWaitCycles, which sets the flag.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          bool honor_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 127u) == 0u) {
      if (honor_abort && *abort_flag) return false;
      if (clock64() - t0 > kWaitCycles) {
        *abort_flag = 1;
        return false;
      }
    }
  }
}
// A TMA load into this CTA's shared memory whose completion is signalled on `bar`, a
// shared::cluster address that may be the pair leader's barrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
// Add the 32 x 32 fp32 box at shared address `src` to the tensor at box coordinates (x, y);
// rows and columns outside the tensor are left out.  One bulk group per call.
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(src)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Store the 32 x 32 16-bit box at shared address `src` (64-byte rows, the map's 64-byte swizzle)
// to the tensor at box coordinates (x, y); rows and columns outside the tensor are left out.
// One bulk group per call.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(src)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Store the 32 x 32 fp32 box at shared address `src` (128-byte rows, the map's 128-byte swizzle)
// to split z of the tensor at box coordinates (x, y); rows and columns outside are left out.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z), "r"(src)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// At most one bulk group of this thread still reading shared memory.
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// No bulk group of this thread still reading shared memory / none still in flight.
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Order this thread's shared-memory writes before the async proxy (TMA) reads them.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// An arrival that orders nothing but this thread's completed tcgen05 reads before it (the
// tcgen05.fence::before_thread_sync ahead of it): relaxed, so that it does not wait for the
// thread's global stores still in flight.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

// Shared-memory matrix descriptor of a 128-byte-swizzled tile (start, leading and stride
// byte offsets in 16-byte units, descriptor version 1, swizzle mode 2 = 128 B).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}
// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, their majorness,
// N / 8 and M / 16 (M = 256: the pair's tile).
template <bool A_MN, bool B_MN>
__host__ __device__ constexpr uint32_t idesc_bf16() {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((A_MN ? 1u : 0u) << 15) | ((B_MN ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>((2 * BM) >> 4) << 24);
}
// Issued by one thread of the pair's leader: D[256 x 256] (+)= A B, A's rows 0-127 and B's
// columns 0-127 from this CTA's shared memory, the rest from the peer's at the same offsets;
// each CTA's TMEM receives its 128 rows.
__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(
          tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// Arrive on the barrier at offset `bar` in both CTAs of the pair once every MMA this thread
// issued so far has completed.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}
// Arrive on this CTA's barrier `bar` once every MMA this thread issued has completed.
__device__ __forceinline__ void umma_commit_local(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
// 32 consecutive fp32 columns of this warp's 32 TMEM lanes (one lane per thread), without
// waiting for them (tmem_wait_ld).
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, float (&v)[32]) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// The extents of this launch: Params' own, or with the device-side extent applied.
struct Dims {
  int M, m_tiles, k_blocks, total;
};
__device__ __forceinline__ Dims dims_of(const Params& p) {
  Dims d{p.M, p.m_tiles, p.k_blocks, 0};
  if (p.dyn != nullptr) {
    const int n = max(*p.dyn, 0);
    if (p.dyn_k) {
      d.k_blocks = min(p.k_blocks, (n + BK - 1) / BK);
    } else {
      d.M = min(p.M, n);
      d.m_tiles = (d.M + 2 * BM - 1) / (2 * BM);
    }
  }
  d.total = (d.M > 0 && d.k_blocks > 0) ? d.m_tiles * p.n_tiles * p.splits : 0;
  return d;
}

// The tile list: tile t -> (m, n, split) and the split's K blocks [kb0, kb1).
struct Tile {
  int m, n, s, kb0, kb1;
};
__device__ __forceinline__ Tile tile_of(const Params& p, const Dims& d, int t) {
  Tile u;
  const int mn = d.m_tiles * p.n_tiles;
  u.s = t / mn;
  const int r = t - u.s * mn;
  if (p.m_fastest) {
    u.m = r % d.m_tiles;
    u.n = r / d.m_tiles;
  } else {
    u.n = r % p.n_tiles;
    u.m = r / p.n_tiles;
  }
  u.kb0 = static_cast<int>(static_cast<int64_t>(d.k_blocks) * u.s / p.splits);
  u.kb1 = static_cast<int>(static_cast<int64_t>(d.k_blocks) * (u.s + 1) / p.splits);
  return u;
}

// ---------------------------------------------------------------------------
// epilogues (one thread = one row of the tile, 32 columns at a time)
// ---------------------------------------------------------------------------
// Row `lane` of a warp's 32 x 32 fp32 box into its 128-byte-swizzled staging buffer: the
// 16-byte chunk q of row r sits at chunk q ^ (r % 8), so the eight rows a quarter-warp
// writes at once fall in eight different bank groups.
__device__ __forceinline__ void stage_row(uint32_t buf, int lane, const float (&v)[32]) {
  const uint32_t row = buf + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const uint32_t dst = row + static_cast<uint32_t>((q ^ (lane & 7)) * 16);
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "f"(v[4 * q]), "f"(v[4 * q + 1]),
                 "f"(v[4 * q + 2]), "f"(v[4 * q + 3])
                 : "memory");
  }
}

// The logits epilogue's statistic over one row's 128 columns of the tile (the first `cols`
// of them inside the matrix): the maximum m (tile_max), then, box by box, e_j = 2^(x_j c - a)
// with a = m c, and s = sum e_j, u = sum e_j (x_j c - a) (box_exp).  Columns at or past N get
// e = 0.  (The same (a, s, u) the row kernels form, here in two passes over values already in
// registers, so no rescale.)  box_exp writes e_j 2^15 over the box, the scaled form that is
// stored (fp16, below), by shifting the exponent: t' = x_j c - a + 15, so the scale costs no
// multiply; s and u are taken back to the unscaled e at the end (tile_sums).
__device__ __forceinline__ float tile_max(const float (&v)[BN / 64][32], int cols) {
  float m = -INFINITY;
  if (cols >= BN / 2) {
#pragma unroll
    for (int j = 0; j < BN / 64; ++j)
#pragma unroll
      for (int i = 0; i < 32; ++i) m = fmaxf(m, v[j][i]);
  } else {
#pragma unroll
    for (int j = 0; j < BN / 64; ++j)
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (32 * j + i < cols) m = fmaxf(m, v[j][i]);
  }
  return m;
}
constexpr float kExpScaleLog2 = 15.f;  // the stored exponentials are e 2^15
template <bool kH>
__device__ __forceinline__ void box_exp(float (&v)[32], int cols, float2 c2, float2 na2, float2& s2, float2& u2) {
  if (cols < 32) {  // the ragged end of the row: columns past N add nothing
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i >= cols) v[i] = -INFINITY;
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float2 x = make_float2(v[2 * i], v[2 * i + 1]);
    if (kH) {
      x.x = fmaxf(x.x, kNegClamp);  // -inf adds 0 to u, not 0 * -inf
      x.y = fmaxf(x.y, kNegClamp);
    }
    const float2 t = __ffma2_rn(x, c2, na2);  // x c - a + 15
    const float2 e = make_float2(ex2(t.x), ex2(t.y));
    s2 = __fadd2_rn(s2, e);
    if (kH) u2 = __ffma2_rn(e, t, u2);
    v[2 * i] = e.x;
    v[2 * i + 1] = e.y;
  }
}
// s = 2^-15 sum e', u = 2^-15 (sum e' t' - 15 sum e')  (e' = e 2^15, t' = t + 15)
__device__ __forceinline__ float2 tile_sums(float2 s2, float2 u2) {
  const float s = s2.x + s2.y, u = u2.x + u2.y;
  constexpr float kInv = 1.f / 32768.f;
  return make_float2(s * kInv, fmaf(-kExpScaleLog2, s, u) * kInv);
}

// The exponentials are stored as fp16 scaled by 2^15: e <= 1 becomes at most 32768, below
// fp16's 65504, and fp16's normal range then reaches down to e = 2^-29, so the relative
// rounding is 2^-11 for every e that can matter.
__device__ __forceinline__ uint32_t pack_h2(float a, float b) {  // a, b already scaled
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Row `lane` of a warp's 32 x 32 box of exponentials, as fp16, into its staging buffer (64
// bytes a row): the 16-byte chunk q of row r sits at chunk q ^ ((r / 2) % 4), so the eight
// rows a quarter-warp writes at once cover all 32 banks.  This is the TMA's 64-byte swizzle
// (address bits 4-5 XOR bits 7-8), so the buffer goes out as one tensor store.
__device__ __forceinline__ void stage_row_h16(uint32_t buf, int lane, const float (&v)[32]) {
  const uint32_t row = buf + static_cast<uint32_t>(lane) * 64u;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 w = make_uint4(pack_h2(v[8 * q], v[8 * q + 1]), pack_h2(v[8 * q + 2], v[8 * q + 3]),
                               pack_h2(v[8 * q + 4], v[8 * q + 5]), pack_h2(v[8 * q + 6], v[8 * q + 7]));
    const uint32_t dst = row + static_cast<uint32_t>((q ^ ((lane >> 1) & 3)) * 16);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int EPI, bool A_MN, bool B_MN, bool kH>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const Params p,
                const __grid_constant__ CUtensorMap tmC) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem =
      reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char* sA = smem;
  unsigned char* sB = smem + kStages * kStageA;
  unsigned char* sC = sB + kStages * kStageB;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sC + kSmemC);
  // full[s] (the leader's are used), empty[s], tmem_full[2], tmem_empty[2] (the leader's),
  // drain
  const uint32_t full0 = smem_addr(bars), empty0 = smem_addr(bars + kStages);
  const uint32_t tfull0 = smem_addr(bars + 2 * kStages), tempty0 = smem_addr(bars + 2 * kStages + 2);
  const uint32_t drain = smem_addr(bars + 2 * kStages + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();  // 0: the pair's leader, which issues the MMAs
  const bool leader = rank == 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 2 * kEpiWarps);  // one arrival per epilogue warp of the pair
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
    prefetch_tensormap(&tmC);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  wait_for_previous_grids();
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers are initialised before either signals the other's
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const Dims dims = dims_of(p);
  const int total = dims.total;
  const int first = static_cast<int>(cluster_id()), step = static_cast<int>(cluster_count());

  if (warp == 0) {
    // ---- TMA producer (each CTA its halves of A and B) ----
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;  // stages filled and not yet known to be consumed (for the abort path)
      bool ok = true;
      for (int t = first; t < total && ok; t += step) {
        const Tile u = tile_of(p, dims, t);
        const int arow = u.m * 2 * BM + static_cast<int>(rank) * BM;  // this CTA's A rows
        const int bcol = u.n * BN + static_cast<int>(rank) * BNH;      // this CTA's B columns
        for (int kb = u.kb0; kb < u.kb1; ++kb) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          // both CTAs' copies complete on the leader's full barrier, which expects them all
          const uint32_t fb = map_to_rank(full0 + 8 * stage, 0);
          if (leader) mbar_expect_tx(full0 + 8 * stage, 2 * (kStageA + kStageB));
          const uint32_t a_dst = smem_addr(sA + stage * kStageA), b_dst = smem_addr(sB + stage * kStageB);
          const int k0 = kb * BK;
          if constexpr (A_MN) {
            tma_load_2d(a_dst, &tmA, arow, k0, fb);
            tma_load_2d(a_dst + 8192, &tmA, arow + 64, k0, fb);
          } else {
            tma_load_2d(a_dst, &tmA, k0, arow, fb);
          }
          if constexpr (B_MN) {
            tma_load_2d(b_dst, &tmB, bcol, k0, fb);
            tma_load_2d(b_dst + 8192, &tmB, bcol + 64, k0, fb);
          } else {
            tma_load_2d(b_dst, &tmB, k0, bcol, fb);
          }
          issued = issued < kStages ? issued + 1 : kStages;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && leader) {
        // copies may still be landing in the ring: wait (bounded) for each stage's full
        // phase before the CTA's shared memory can go away
        for (int i = 0; i < issued; ++i) {
          if (--stage < 0) {
            stage = kStages - 1;
            phase ^= 1u;
          }
          mbar_wait(full0 + 8 * stage, phase, abort_flag, false);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- MMA issuer: one thread of the leader ----
    if (lane == 0 && leader) {
      constexpr uint32_t idesc = idesc_bf16<A_MN, B_MN>();
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      for (int t = first; t < total && ok; t += step, ++local) {
        const Tile u = tile_of(p, dims, t);
        const int acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        if (!mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1u, abort_flag)) break;
        tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(acc * BN);
        for (int kb = u.kb0; kb < u.kb1; ++kb) {
          if (!mbar_wait(full0 + 8 * stage, phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_addr(sA + stage * kStageA), b_base = smem_addr(sB + stage * kStageB);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = A_MN ? sw128_desc(a_base + kk * 2048, 8192, 1024) : sw128_desc(a_base + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? sw128_desc(b_base + kk * 2048, 8192, 1024) : sw128_desc(b_base + kk * 32, 16, 1024);
            umma_bf16(d, ad, bd, idesc, (kb > u.kb0 || kk > 0) ? 1u : 0u);
          }
          umma_commit_pair(empty0 + 8 * stage);  // both CTAs' stage is free once these MMAs are done
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) umma_commit_pair(tfull0 + 8 * acc);  // both CTAs' accumulator halves are ready
      }
      // no MMA may still be writing either CTA's TMEM when it is freed (a launch whose
      // device-side extent left it no tiles issued none)
      if (local > 0) {
        umma_commit_local(drain);
        mbar_wait(drain, 0, abort_flag, false);
      }
    }
    __syncwarp();
  } else {
    // ---- epilogue: warps 2..9; TMEM lanes 32 * (warp % 4) ..., columns half * 128 ... ----
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;
    const uint32_t buf = smem_addr(sC) + static_cast<uint32_t>(warp - 2) * kStageC;
    uint32_t nbox = 0;  // kEpiLogits: boxes this warp has stored (they alternate between two 2 KB halves)
    int local = 0;
    for (int t = first; t < total; t += step, ++local) {
      const Tile u = tile_of(p, dims, t);
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      const bool ok = mbar_wait(tfull0 + 8 * acc, acc_phase, abort_flag);
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
      tc_fence_after();
      const int row0 = u.m * 2 * BM + static_cast<int>(rank) * BM + quarter * 32;  // this warp's first row
      const int row = row0 + lane;
      const bool row_ok = row < dims.M;
      const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>(acc * BN + half * (BN / 2));
      const int col_base = u.n * BN + half * (BN / 2);
      const int boxes = min(BN / 64, (p.N - col_base + 31) / 32);  // boxes with columns below N
      // all of this warp's 128 accumulator columns into registers with one wait, then the
      // accumulator goes back to the MMA while the statistic and the stores proceed
      float v[BN / 64][32];
#pragma unroll
      for (int j = 0; j < BN / 64; ++j) tmem_ld32_async(taddr + 32 * j, v[j]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(map_to_rank(tempty0 + 8 * acc, 0));  // done with it
      if constexpr (EPI == kEpiLogits) {
        // the statistic of the row's 128 columns, and the exponentials relative to their
        // maximum stored (fp16, scaled by 2^15) in place of the logits
        const float m = tile_max(v, p.N - col_base);
        const float st_a = m * p.c;
        // every logit -inf: e = 0 and nothing to add, with a finite shift (no -inf - -inf)
        const float shift = (m == -INFINITY ? 0.f : st_a) - kExpScaleLog2;
        const float2 c2 = make_float2(p.c, p.c), na2 = make_float2(-shift, -shift);
        float2 s2 = make_float2(0.f, 0.f), u2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < BN / 64; ++j) {
          if (j >= boxes) break;
          const int col0 = col_base + 32 * j;
          box_exp<kH>(v[j], p.N - col0, c2, na2, s2, u2);
          const uint32_t hb = buf + (nbox & 1u) * 2048u;
          if (lane == 0) bulk_wait_read1();  // the store before the last one has read this half
          __syncwarp();
          stage_row_h16(hb, lane, v[j]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && row0 < p.M) tma_store_2d(&tmC, hb, col0, row0);
          ++nbox;
        }
        if (row_ok && col_base < p.N) {
          const float2 su = tile_sums(s2, u2);
          p.stats[static_cast<int64_t>(row) * (2 * p.n_tiles) + 2 * u.n + half] = make_float4(st_a, su.x, su.y, 0.f);
        }
      } else if constexpr (EPI == kEpiAccum) {
        // each 32 x 32 box staged (128-byte swizzle, the tensor map's) and added to the output
        // by a TMA reduce-add, so the adds cost one instruction a box; the box's buffer is
        // restaged only once the previous reduce has read it
#pragma unroll
        for (int j = 0; j < BN / 64; ++j) {
          if (j >= boxes) break;
          const int col0 = col_base + 32 * j;
          if (lane == 0) bulk_wait_read0();
          __syncwarp();
          stage_row(buf, lane, v[j]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) tma_reduce_add_2d(&tmC, buf, col0, row0);
        }
      } else {
        // each 32 x 32 box staged (128-byte swizzle, the tensor map's) and stored to split u.s
        // by one TMA store; the buffer is restaged only once the previous store has read it
#pragma unroll
        for (int j = 0; j < BN / 64; ++j) {
          if (j >= boxes) break;
          const int col0 = col_base + 32 * j;
          if (lane == 0) bulk_wait_read0();
          __syncwarp();
          stage_row(buf, lane, v[j]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && row0 < p.M) tma_store_3d(&tmC, buf, col0, row0, u.s);
        }
      }
    }
  }
  if (warp >= 2 && lane == 0) bulk_wait_all();  // the epilogue's stores / adds are done
  __syncthreads();
  tc_fence_before();
  cluster_sync();  // neither CTA leaves while the other's copies, MMAs or arrivals may target it
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
  if (threadIdx.x == 0 && *abort_flag && p.err != nullptr) atomicOr(p.err, GRPO_DEVERR_TIMEOUT_BIT);
}

// ---------------------------------------------------------------------------
// host side: tensor maps and the launch
// ---------------------------------------------------------------------------
using TensorMapEncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                       const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                       CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled, looked up once through the runtime (no link against the driver
// library).
inline TensorMapEncodeFn tensor_map_encoder() {
  static const TensorMapEncodeFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<TensorMapEncodeFn>(nullptr);
    return reinterpret_cast<TensorMapEncodeFn>(f);
  }();
  return fn;
}

// A bf16 matrix of `outer` rows of `inner` elements, `row_elems` apart (a multiple of 8),
// read in boxes of box_outer rows x box_inner elements (box_inner = 64: one 128-byte
// swizzle row).  Elements outside [0, inner) x [0, outer) read as zero.
inline bool make_bf16_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_elems,
                          uint32_t box_inner, uint32_t box_outer) {
  const TensorMapEncodeFn enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_elems * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t elem_strides[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, elem_strides,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The tensor map of one operand: K-major (K contiguous: [MN rows][K], one box of `mn_box`
// rows x 64) or MN-major (MN contiguous: [K rows][MN], boxes of 64 rows x 64).
inline bool make_operand_map(CUtensorMap* map, const void* base, bool mn_major, uint64_t mn, uint64_t k,
                             uint64_t row_elems, uint32_t mn_box) {
  return mn_major ? make_bf16_map(map, base, mn, k, row_elems, 64, BK)
                  : make_bf16_map(map, base, k, mn, row_elems, BK, mn_box);
}

inline int sm_count() {
  static int count_of_device[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (count_of_device[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    count_of_device[dev] = n;
  }
  return count_of_device[dev];
}

// Launch one GEMM: min(tiles, the pairs that fit at once) persistent CTA pairs.  The
// kernel's shared-memory attribute and its number of co-resident pairs are set up once per
// device (the occupancy query costs far more host time than a launch).
template <int EPI, bool A_MN, bool B_MN, bool kH>
cudaError_t launch_gemm(const CUtensorMap& a, const CUtensorMap& b, const Params& p, cudaStream_t stream) {
  auto kernel = gemm_kernel<EPI, A_MN, B_MN, kH>;
  const int total = p.m_tiles * p.n_tiles * p.splits;
  if (total <= 0) return cudaSuccess;
  static int pairs_of_device[64] = {};  // 0: not yet known
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  int pairs = pairs_of_device[dev];
  if (pairs == 0) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    cfg.numAttrs = 1;  // the occupancy query takes the cluster shape only
    cfg.gridDim = dim3(2 * 512);
    e = cudaOccupancyMaxActiveClusters(&pairs, kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (pairs <= 0) return cudaErrorInvalidConfiguration;
    pairs_of_device[dev] = pairs;
  }
  if (p.pair_limit > 0 && p.pair_limit < pairs) pairs = p.pair_limit;
  cfg.numAttrs = 2;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * (total < pairs ? total : pairs)));
  // kEpiAccum: the output's tensor map, 32 x 32 fp32 boxes with the staging buffer's swizzle
  CUtensorMap c{};
  if (EPI == kEpiLogits) {  // 32 x 32 boxes of the 16-bit exponentials, 64-byte swizzle (the staging's)
    const TensorMapEncodeFn enc = tensor_map_encoder();
    if (enc == nullptr || p.ldc % 8 != 0) return cudaErrorInvalidValue;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.N), static_cast<cuuint64_t>(p.M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.ldc) * 2};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t elem_strides[2] = {1, 1};
    if (enc(&c, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, p.C, dims, strides, box, elem_strides,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  if (EPI == kEpiStore) {  // [splits][M][ldc] fp32, 32 x 32 boxes with the staging buffer's swizzle
    const TensorMapEncodeFn enc = tensor_map_encoder();
    if (enc == nullptr || p.ldc % 4 != 0) return cudaErrorInvalidValue;
    const int64_t zs = p.splits > 1 ? p.split_stride : p.ldc * p.M;
    if (zs % 4 != 0) return cudaErrorInvalidValue;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(p.N), static_cast<cuuint64_t>(p.M),
                                static_cast<cuuint64_t>(p.splits)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(p.ldc) * 4, static_cast<cuuint64_t>(zs) * 4};
    const cuuint32_t box[3] = {32, 32, 1};
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    if (enc(&c, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p.C, dims, strides, box, elem_strides,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  if (EPI == kEpiAccum) {
    const TensorMapEncodeFn enc = tensor_map_encoder();
    if (enc == nullptr || p.ldc % 4 != 0) return cudaErrorInvalidValue;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.N), static_cast<cuuint64_t>(p.M)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.ldc) * 4};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t elem_strides[2] = {1, 1};
    if (enc(&c, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, p.C, dims, strides, box, elem_strides,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  return cudaLaunchKernelEx(&cfg, kernel, a, b, p, c);
}

}  // namespace gemm
}  // namespace grpo
