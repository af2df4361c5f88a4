// Device helpers shared by the forward and backward row kernels (sm_103a).
//
// Element formats: bf16 (8 per 16-byte vector) and fp32 (4 per vector).  A row of V
// elements is split, by the alignment of ITS OWN start address, into a scalar head
// (elements before the first 16-byte boundary), a body of 16-byte vectors, and a
// scalar tail.  Rows of a contiguous [R, V] tensor with V*size a multiple of 16 have
// no head and no tail.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "rowpass_internal.h"

namespace grpo {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;

// First statement of every kernel: wait until the grids launched before this one in the
// stream have completed and their memory is visible (see launch_after_previous).
__device__ __forceinline__ void wait_for_previous_grids() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Thread-block clusters: this CTA's rank, the shared::cluster address of one of this CTA's
// shared variables in CTA `rank` of the cluster, remote stores there, and the cluster-wide
// barrier (every thread of every CTA of the cluster), also split into its two halves.
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_count() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void st_cluster_f32(uint32_t cluster_addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(cluster_addr), "f"(v) : "memory");
}
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_sync() {
  cluster_arrive();
  cluster_wait();
}

// 2^x on the SFU (PTX ex2.approx.ftz.f32).  Results below 2^-126 flush to zero.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 16-byte loads.  The forward kernels never write the logits, so they use the
// non-coherent read-only path; the backward may write the same addresses it reads
// (in-place dlogits), so it uses the coherent path.  Neither allocates in L1: every
// byte is touched once.
__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}
__device__ __forceinline__ uint4 ld_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p)
               : "memory");
  return r;
}
__device__ __forceinline__ void st_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// The same accesses with an L2 eviction priority (createpolicy + .L2::cache_hint, the
// policy made next to each access so that no 64-bit policy register stays live across
// the streaming loops).  The priority steers which lines the L2 gives up first and
// changes no result:
//   evict_first - data touched for the last time in this pass: the logits of a row whose
//                 gradient is known to be zero, a row's last read, every gradient store;
//   evict_last  - logits that will be read again soon: a GRPO row in the forward (the
//                 backward reads it next) and in the fused kernel's first sweep.  The
//                 re-read lets them go (evict_first); a row that turns out to need no
//                 re-read is put back to normal priority by l2_demote.
__device__ __forceinline__ uint4 ld_nc_v4_evict_first(const void* p) {
  uint4 r;
  asm("{\n\t.reg .b64 pol;\n\t"
      "createpolicy.fractional.L2::evict_first.b64 pol, 1.0;\n\t"
      "ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], pol;\n\t}"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}
__device__ __forceinline__ uint4 ld_v4_evict_first(const void* p) {
  uint4 r;
  asm volatile("{\n\t.reg .b64 pol;\n\t"
               "createpolicy.fractional.L2::evict_first.b64 pol, 1.0;\n\t"
               "ld.global.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], pol;\n\t}"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p)
               : "memory");
  return r;
}
__device__ __forceinline__ uint4 ld_nc_v4_evict_last(const void* p) {
  uint4 r;
  asm("{\n\t.reg .b64 pol;\n\t"
      "createpolicy.fractional.L2::evict_last.b64 pol, 1.0;\n\t"
      "ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], pol;\n\t}"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}
__device__ __forceinline__ uint4 ld_v4_evict_last(const void* p) {
  uint4 r;
  asm volatile("{\n\t.reg .b64 pol;\n\t"
               "createpolicy.fractional.L2::evict_last.b64 pol, 1.0;\n\t"
               "ld.global.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], pol;\n\t}"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p)
               : "memory");
  return r;
}
__device__ __forceinline__ void st_v4_evict_first(void* p, uint4 v) {
  asm volatile("{\n\t.reg .b64 pol;\n\t"
               "createpolicy.fractional.L2::evict_first.b64 pol, 1.0;\n\t"
               "st.global.L1::no_allocate.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, pol;\n\t}"
               ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Put the L2 lines of [p, p + bytes) that are present back to normal priority, without
// reading them.  The 128-byte line addresses are rounded down from p; they stay inside
// the memory page that holds p, since pages are larger than and aligned to 128 bytes.
template <int THREADS>
__device__ __forceinline__ void l2_demote(const void* p, int64_t bytes) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(p) & ~static_cast<uintptr_t>(127);
  const uintptr_t end = reinterpret_cast<uintptr_t>(p) + static_cast<uintptr_t>(bytes);
  for (uintptr_t a = a0 + 128u * threadIdx.x; a < end; a += 128u * THREADS)
    asm volatile("applypriority.global.L2::evict_normal [%0], 128;" ::"l"(a) : "memory");
}

// ---------------------------------------------------------------------------
// element traits
// ---------------------------------------------------------------------------
struct BF16 {
  using storage = uint16_t;
  static constexpr int kVec = 8;
  static constexpr uint32_t kSignPair = 0x80008000u;  // sign bits of both halves of a word
  static constexpr uint32_t kNaNPair = 0x7FC07FC0u;
  __device__ __forceinline__ static float lo(uint32_t w) { return __uint_as_float(w << 16); }
  __device__ __forceinline__ static float hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
  __device__ __forceinline__ static float load_scalar(const storage* p) {
    return __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(p))) << 16);
  }
  __device__ __forceinline__ static float load_scalar_coherent(const storage* p) {
    return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const volatile unsigned short*>(p)) << 16);
  }
  __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[kVec]) {
    f[0] = lo(v.x); f[1] = hi(v.x); f[2] = lo(v.y); f[3] = hi(v.y);
    f[4] = lo(v.z); f[5] = hi(v.z); f[6] = lo(v.w); f[7] = hi(v.w);
  }
  // the vector as kVec / 2 pairs of floats (elements 2i, 2i+1), for the packed f32x2 math
  static constexpr int kPairs = 4;
  __device__ __forceinline__ static float2 pair(const uint4& v, int i) {
    const uint32_t w = i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
    return make_float2(lo(w), hi(w));
  }
  // pairs -> one 16-byte vector, RNE; NEG stores the negated values
  template <bool NEG>
  __device__ __forceinline__ static uint4 pack_pairs(const float2 (&e)[kPairs]) {
    uint4 o;
    o.x = NEG ? pack2(-e[0].x, -e[0].y) : pack2(e[0].x, e[0].y);
    o.y = NEG ? pack2(-e[1].x, -e[1].y) : pack2(e[1].x, e[1].y);
    o.z = NEG ? pack2(-e[2].x, -e[2].y) : pack2(e[2].x, e[2].y);
    o.w = NEG ? pack2(-e[3].x, -e[3].y) : pack2(e[3].x, e[3].y);
    return o;
  }
  // Maximum of the vectors' elements.  max.bf16x2 is exact and returns the non-NaN
  // operand when one operand is NaN (NaN rows still end as NaN through the sums).
  template <int N>
  __device__ __forceinline__ static float chunk_max(const uint4 (&v)[N]) {
    __nv_bfloat162 m = *reinterpret_cast<const __nv_bfloat162*>(&v[0].x);
#pragma unroll
    for (int k = 0; k < N; ++k) {
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v[k]);
      m = __hmax2(m, __hmax2(__hmax2(h[0], h[1]), __hmax2(h[2], h[3])));
    }
    return fmaxf(__low2float(m), __high2float(m));
  }
  // Raise every element below -2^60 (i.e. -inf) to -2^60; NaN stays NaN.  Used before
  // the entropy accumulation so that a -inf logit adds 2^t * t = 0 instead of 0 * -inf.
  __device__ __forceinline__ static void clamp_low(uint4& v) {
    const __nv_bfloat162 lo2 = __floats2bfloat162_rn(-1.152921504606847e18f, -1.152921504606847e18f);
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&v);
    h[0] = __hmax2_nan(h[0], lo2); h[1] = __hmax2_nan(h[1], lo2);
    h[2] = __hmax2_nan(h[2], lo2); h[3] = __hmax2_nan(h[3], lo2);
  }
  __device__ __forceinline__ static uint32_t pack2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // RNE; a -> low half
    return *reinterpret_cast<uint32_t*>(&h);
  }
  // eight floats -> one 16-byte vector, with `flip` XOR-ed into every sign bit pair
  __device__ __forceinline__ static uint4 pack(const float (&e)[kVec], uint32_t flip) {
    uint4 o;
    o.x = pack2(e[0], e[1]) ^ flip; o.y = pack2(e[2], e[3]) ^ flip;
    o.z = pack2(e[4], e[5]) ^ flip; o.w = pack2(e[6], e[7]) ^ flip;
    return o;
  }
  __device__ __forceinline__ static void store_scalar(storage* p, float v) {
    __nv_bfloat16 h = __float2bfloat16_rn(v);
    *reinterpret_cast<__nv_bfloat16*>(p) = h;
  }
  __device__ __forceinline__ static void store_bits(storage* p, uint32_t pair) {
    *p = static_cast<uint16_t>(pair & 0xFFFFu);
  }
};

struct F32 {
  using storage = float;
  static constexpr int kVec = 4;
  static constexpr uint32_t kSignPair = 0x80000000u;
  static constexpr uint32_t kNaNPair = 0x7FC00000u;
  __device__ __forceinline__ static float load_scalar(const storage* p) { return __ldg(p); }
  __device__ __forceinline__ static float load_scalar_coherent(const storage* p) {
    return *reinterpret_cast<const volatile float*>(p);
  }
  __device__ __forceinline__ static void unpack(const uint4& v, float (&f)[kVec]) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
  }
  static constexpr int kPairs = 2;
  __device__ __forceinline__ static float2 pair(const uint4& v, int i) {
    return i == 0 ? make_float2(__uint_as_float(v.x), __uint_as_float(v.y))
                  : make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
  }
  template <bool NEG>
  __device__ __forceinline__ static uint4 pack_pairs(const float2 (&e)[kPairs]) {
    return NEG ? make_uint4(__float_as_uint(-e[0].x), __float_as_uint(-e[0].y), __float_as_uint(-e[1].x),
                            __float_as_uint(-e[1].y))
               : make_uint4(__float_as_uint(e[0].x), __float_as_uint(e[0].y), __float_as_uint(e[1].x),
                            __float_as_uint(e[1].y));
  }
  template <int N>
  __device__ __forceinline__ static float chunk_max(const uint4 (&v)[N]) {
    float m = __uint_as_float(v[0].x);
#pragma unroll
    for (int k = 0; k < N; ++k)
      m = fmaxf(m, fmaxf(fmaxf(__uint_as_float(v[k].x), __uint_as_float(v[k].y)),
                         fmaxf(__uint_as_float(v[k].z), __uint_as_float(v[k].w))));
    return m;
  }
  __device__ __forceinline__ static void clamp_low(uint4& v) {
    constexpr float lo = -1.152921504606847e18f;  // -2^60
    float* f = reinterpret_cast<float*>(&v);
#pragma unroll
    for (int q = 0; q < 4; ++q) f[q] = f[q] < lo ? lo : f[q];  // NaN stays NaN
  }
  __device__ __forceinline__ static uint4 pack(const float (&e)[kVec], uint32_t flip) {
    return make_uint4(__float_as_uint(e[0]) ^ flip, __float_as_uint(e[1]) ^ flip,
                      __float_as_uint(e[2]) ^ flip, __float_as_uint(e[3]) ^ flip);
  }
  __device__ __forceinline__ static void store_scalar(storage* p, float v) { *p = v; }
  __device__ __forceinline__ static void store_bits(storage* p, uint32_t bits) {
    *reinterpret_cast<uint32_t*>(p) = bits;
  }
};

// Split of one row into scalar head, 16-byte vector body and scalar tail.
struct RowSplit {
  int head;  // elements before the first 16-byte boundary
  int nvec;  // 16-byte vectors in the body
  int tail;  // elements after the body
};

template <class E>
__device__ __forceinline__ RowSplit split_row(const void* row, int V) {
  const int mis = static_cast<int>(reinterpret_cast<uintptr_t>(row) & 15u);
  int head = mis ? (16 - mis) / static_cast<int>(sizeof(typename E::storage)) : 0;
  head = head < V ? head : V;
  const int rest = V - head;
  RowSplit s;
  s.head = head;
  s.nvec = rest / E::kVec;
  s.tail = rest - s.nvec * E::kVec;
  return s;
}

// ---------------------------------------------------------------------------
// online softmax statistic of a set of logits x_j, relative to an offset a (log2 units;
// a is the running maximum times c, rounded to fp32, and is used exactly as stored):
//   t_j = x_j * c - a  (one FMA),  s = sum_j 2^{t_j},  u = sum_j 2^{t_j} t_j,
//   c = log2(e) / T.
// Then  lse = ln2 * a + ln s  and  H = ln s - ln2 * u / s,  whatever the rounding of a.
// ---------------------------------------------------------------------------
struct Stat {
  float a, s, u;
};

// Merge two partial statistics.  An empty partial (s == 0) is the identity; NaN
// partials propagate.
__device__ __forceinline__ Stat stat_combine(const Stat& x, const Stat& y) {
  if (y.s == 0.f) return x;
  if (x.s == 0.f) return y;
  const float A = fmaxf(x.a, y.a);
  const float dx = x.a - A, dy = y.a - A;
  const float ex = ex2(dx), ey = ex2(dy);
  Stat r;
  r.a = A;
  r.s = ex * x.s + ey * y.s;
  r.u = ex * fmaf(dx, x.s, x.u) + ey * fmaf(dy, y.s, y.u);
  return r;
}

// Re-express a partial relative to the offset A >= v.a (empty partials stay empty).
__device__ __forceinline__ Stat stat_shift(const Stat& v, float A) {
  if (v.s == 0.f) return Stat{A, 0.f, 0.f};
  const float d = v.a - A;
  const float e = ex2(d);
  return Stat{A, e * v.s, e * fmaf(d, v.s, v.u)};
}

// Warp-wide merge, result in every lane: the largest offset first (one max per
// round), then every lane moves to it once, then plain sums.
__device__ __forceinline__ Stat stat_warp_reduce(Stat v) {
  float A = v.s == 0.f ? -INFINITY : v.a;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) A = fmaxf(A, __shfl_xor_sync(0xFFFFFFFFu, A, off));
  if (A == -INFINITY) return Stat{-INFINITY, 0.f, 0.f};  // every lane empty
  v = stat_shift(v, A);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    v.s += __shfl_xor_sync(0xFFFFFFFFu, v.s, off);
    v.u += __shfl_xor_sync(0xFFFFFFFFu, v.u, off);
  }
  return v;
}

// CTA-wide merge; the result is valid in thread 0.
template <int THREADS>
__device__ __forceinline__ Stat stat_block_reduce(Stat v) {
  constexpr int kWarps = THREADS / 32;
  v = stat_warp_reduce(v);
  if (kWarps == 1) return v;
  __shared__ Stat sh[kWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < kWarps ? sh[lane] : Stat{-INFINITY, 0.f, 0.f};
    v = stat_warp_reduce(v);
  }
  return v;
}

// CTA-wide float sum, broadcast to every thread.
template <int THREADS>
__device__ __forceinline__ float block_sum_all(float v) {
  constexpr int kWarps = THREADS / 32;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
  if (kWarps == 1) return v;
  __shared__ float sh[kWarps];
  __shared__ float total;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) sh[warp] = v;
  __syncthreads();
  if (warp == 0) {
    v = lane < kWarps ? sh[lane] : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
    if (lane == 0) total = v;
  }
  __syncthreads();
  return total;
}

}  // namespace grpo
