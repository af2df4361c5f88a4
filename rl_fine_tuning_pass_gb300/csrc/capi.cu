// C-ABI entry points declared in include/grpo_rowpass.h.  Host-side validation runs
// completely before any CUDA call, so a rejected call has no effect on the device.
#include <algorithm>
#include <cmath>
#include <cstdint>

#include "grpo_rowpass.h"
#include "rowpass_internal.h"
#include "rowpass_linear.h"

namespace {

using grpo::BwdParams;
using grpo::FwdParams;

constexpr double kLog2eD = 1.4426950408889634074;
constexpr int64_t kMaxRows = (int64_t(1) << 31) - 1;  // one CTA per row, 1-D grid
constexpr int64_t kMaxV = (int64_t(1) << 30);         // in-row indices are 32-bit

int elem_size(int32_t dtype) { return dtype == GRPO_BF16 ? 2 : 4; }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Offset (elements) of the last element of the last row, +1; -1 on overflow.
int64_t extent_elems(const grpo_rows* t) {
  const long double e = static_cast<long double>(t->B - 1) * t->stride_b +
                        static_cast<long double>(t->L - 1) * t->stride_l + t->V;
  if (e > 4.0e18L) return -1;
  return (t->B - 1) * t->stride_b + (t->L - 1) * t->stride_l + t->V;
}

// Rows of an output tensor must not overlap: one of the two strides is the inner one.
bool rows_disjoint(const grpo_rows* t) {
  auto nested = [&](int64_t si, int64_t ni, int64_t so, int64_t no) {
    if (ni > 1 && si < t->V) return false;
    const int64_t span = (ni > 0 ? ni - 1 : 0) * si + t->V;
    return !(no > 1 && so < span);
  };
  return nested(t->stride_l, t->L, t->stride_b, t->B) || nested(t->stride_b, t->B, t->stride_l, t->L);
}

int64_t rows_of(const grpo_rows* t) { return t->B * t->L; }

grpo_status check_rows(const grpo_rows* t) {
  if (t == nullptr) return GRPO_ERR_INVALID_ARG;
  if (t->ptr == nullptr && !(t->B == 0 || t->L == 0)) return GRPO_ERR_INVALID_ARG;
  if (t->dtype != GRPO_FP32 && t->dtype != GRPO_BF16) return GRPO_ERR_INVALID_ARG;
  if (t->reserved != 0) return GRPO_ERR_INVALID_ARG;
  if (t->B < 0 || t->L < 0 || t->V < 1) return GRPO_ERR_INVALID_ARG;
  if (t->stride_b < 0 || t->stride_l < 0) return GRPO_ERR_INVALID_ARG;
  if (!aligned(t->ptr, elem_size(t->dtype))) return GRPO_ERR_INVALID_ARG;
  if (t->V > kMaxV) return GRPO_ERR_UNSUPPORTED;
  if (t->B > 0 && t->L > 0) {
    if (static_cast<long double>(t->B) * t->L > kMaxRows) return GRPO_ERR_UNSUPPORTED;
    if (extent_elems(t) < 0) return GRPO_ERR_INVALID_ARG;
  }
  return GRPO_OK;
}

bool finite_pos(float v) { return std::isfinite(v) && v > 0.f; }

grpo_status check_scalars_grpo(float T, float beta, float eps_low, float eps_high) {
  if (!finite_pos(T)) return GRPO_ERR_INVALID_ARG;
  if (!std::isfinite(beta) || beta < 0.f) return GRPO_ERR_INVALID_ARG;
  if (!std::isfinite(eps_low) || eps_low < 0.f || eps_low > 1.f) return GRPO_ERR_INVALID_ARG;
  if (!std::isfinite(eps_high) || eps_high < 0.f) return GRPO_ERR_INVALID_ARG;
  return GRPO_OK;
}

bool ok_f32(const void* p) { return p != nullptr && aligned(p, 4); }
bool ok_i64(const void* p) { return p != nullptr && aligned(p, 8); }
bool ok_opt_f32(const void* p) { return p == nullptr || aligned(p, 4); }
bool ok_opt_i32(const void* p) { return p == nullptr || aligned(p, 4); }

grpo::RowsView view_of(const grpo_rows* t) {
  return grpo::RowsView{t->ptr, t->L, t->stride_b, t->stride_l, static_cast<int>(t->V)};
}

// dlogits: same dtype and shape as logits, disjoint rows, and either exactly the same
// tensor (in-place) or no byte in common with it.
grpo_status check_dlogits(const grpo_rows* x, const grpo_rows* dx, bool* same_phase) {
  grpo_status st = check_rows(dx);
  if (st != GRPO_OK) return st;
  if (dx->dtype != x->dtype || dx->B != x->B || dx->L != x->L || dx->V != x->V)
    return GRPO_ERR_INVALID_ARG;
  const int es = elem_size(x->dtype);
  const int64_t rows = x->B * x->L;
  if (rows > 1 && !rows_disjoint(dx)) return GRPO_ERR_INVALID_ARG;
  if (rows > 0) {
    const uintptr_t xa = reinterpret_cast<uintptr_t>(x->ptr);
    const uintptr_t da = reinterpret_cast<uintptr_t>(dx->ptr);
    const uintptr_t xe = xa + static_cast<uintptr_t>(extent_elems(x)) * es;
    const uintptr_t de = da + static_cast<uintptr_t>(extent_elems(dx)) * es;
    const bool overlap = xa < de && da < xe;
    const bool same = xa == da && (x->B <= 1 || x->stride_b == dx->stride_b) &&
                      (x->L <= 1 || x->stride_l == dx->stride_l);
    if (overlap && !same) return GRPO_ERR_INVALID_ARG;
  }
  // every row of dx starts at the same address mod 16 as the matching row of x
  const int64_t ph = (static_cast<int64_t>(reinterpret_cast<uintptr_t>(x->ptr) & 15) -
                      static_cast<int64_t>(reinterpret_cast<uintptr_t>(dx->ptr) & 15));
  const bool b_ok = x->B <= 1 || ((x->stride_b - dx->stride_b) * es) % 16 == 0;
  const bool l_ok = x->L <= 1 || ((x->stride_l - dx->stride_l) * es) % 16 == 0;
  *same_phase = ph == 0 && b_ok && l_ok;
  return GRPO_OK;
}

grpo_status from_cuda(cudaError_t e) { return e == cudaSuccess ? GRPO_OK : GRPO_ERR_CUDA; }

// Streaming multiprocessors of the current device (queried once per device; the
// launch shape depends on how many rows can be resident at once).
int device_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    cache[dev] = n;
  }
  return cache[dev];
}

}  // namespace

extern "C" {

grpo_status grpo_loss_fwd(const grpo_rows* logits, const int64_t* idx, const float* old_logp,
                          const float* ref_logp, const float* adv, const uint8_t* mask, float T,
                          float beta, float eps_low, float eps_high, float* loss, float* logp,
                          float* lse, float* kl, uint8_t* is_clipped, float* entropy, int32_t* dev_err,
                          grpo_stream_t stream) {
  grpo_status st = check_rows(logits);
  if (st != GRPO_OK) return st;
  if ((st = check_scalars_grpo(T, beta, eps_low, eps_high)) != GRPO_OK) return st;
  if (rows_of(logits) == 0) return GRPO_OK;  // nothing to read or write; pointers may be NULL
  if (!ok_i64(idx) || !ok_opt_f32(old_logp) || !ok_f32(adv) || !ok_f32(loss) || !ok_f32(logp) ||
      !ok_f32(lse) || !ok_opt_f32(kl) || !ok_opt_f32(entropy) || !ok_opt_i32(dev_err))
    return GRPO_ERR_INVALID_ARG;
  if (beta != 0.f && !ok_f32(ref_logp)) return GRPO_ERR_INVALID_ARG;
  if (ref_logp != nullptr && !aligned(ref_logp, 4)) return GRPO_ERR_INVALID_ARG;
  const int64_t rows = logits->B * logits->L;
  if (rows == 0) return GRPO_OK;
  FwdParams p{};
  p.x = view_of(logits);
  p.idx = idx;
  p.old_logp = old_logp;
  p.ref_logp = ref_logp;
  p.adv = adv;
  p.mask = mask;
  p.c = static_cast<float>(kLog2eD / static_cast<double>(T));
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
  const int mode = entropy ? grpo::kFwdGrpoH : grpo::kFwdGrpo;
  return from_cuda(grpo::launch_fwd(mode, logits->dtype, p, rows, device_sms(), reinterpret_cast<cudaStream_t>(stream)));
}

grpo_status grpo_loss_bwd(const grpo_rows* logits, const int64_t* idx, const float* old_logp,
                          const float* ref_logp, const float* adv, const uint8_t* mask,
                          const float* dloss, const float* logp, const float* lse, float T,
                          float beta, float eps_low, float eps_high, const grpo_rows* dlogits,
                          int32_t* dev_err, grpo_stream_t stream) {
  grpo_status st = check_rows(logits);
  if (st != GRPO_OK) return st;
  if ((st = check_scalars_grpo(T, beta, eps_low, eps_high)) != GRPO_OK) return st;
  bool same_phase = false;
  if ((st = check_dlogits(logits, dlogits, &same_phase)) != GRPO_OK) return st;
  if (rows_of(logits) == 0) return GRPO_OK;
  if (!ok_i64(idx) || !ok_opt_f32(old_logp) || !ok_f32(adv) || !ok_f32(dloss) || !ok_f32(logp) ||
      !ok_f32(lse) || !ok_opt_i32(dev_err))
    return GRPO_ERR_INVALID_ARG;
  if (beta != 0.f && !ok_f32(ref_logp)) return GRPO_ERR_INVALID_ARG;
  if (ref_logp != nullptr && !aligned(ref_logp, 4)) return GRPO_ERR_INVALID_ARG;
  const int64_t rows = logits->B * logits->L;
  if (rows == 0) return GRPO_OK;
  BwdParams p{};
  p.x = view_of(logits);
  p.dx = grpo::OutView{dlogits->ptr, dlogits->L, dlogits->stride_b, dlogits->stride_l,
                       static_cast<int>(dlogits->V)};
  p.idx = idx;
  p.lse = lse;
  p.old_logp = old_logp;
  p.ref_logp = ref_logp;
  p.adv = adv;
  p.mask = mask;
  p.dloss = dloss;
  p.logp = logp;
  p.c = static_cast<float>(kLog2eD / static_cast<double>(T));
  p.T = T;
  p.beta = beta;
  p.lo = static_cast<float>(1.0 - static_cast<double>(eps_low));
  p.hi = static_cast<float>(1.0 + static_cast<double>(eps_high));
  p.dev_err = dev_err;
  return from_cuda(grpo::launch_bwd(true, logits->dtype, same_phase, p, rows, device_sms(),
                                    reinterpret_cast<cudaStream_t>(stream)));
}

grpo_status grpo_loss_fused(const grpo_rows* logits, const int64_t* idx, const float* old_logp,
                            const float* ref_logp, const float* adv, const uint8_t* mask, const float* dloss,
                            float T, float beta, float eps_low, float eps_high, float* loss, float* logp,
                            float* lse, float* kl, uint8_t* is_clipped, float* entropy,
                            const grpo_rows* dlogits, int32_t* dev_err, grpo_stream_t stream) {
  grpo_status st = check_rows(logits);
  if (st != GRPO_OK) return st;
  if ((st = check_scalars_grpo(T, beta, eps_low, eps_high)) != GRPO_OK) return st;
  bool same_phase = false;
  if ((st = check_dlogits(logits, dlogits, &same_phase)) != GRPO_OK) return st;
  if (rows_of(logits) == 0) return GRPO_OK;
  if (!ok_i64(idx) || !ok_opt_f32(old_logp) || !ok_f32(adv) || !ok_f32(dloss) || !ok_f32(loss) ||
      !ok_f32(logp) || !ok_f32(lse) || !ok_opt_f32(kl) || !ok_opt_f32(entropy) || !ok_opt_i32(dev_err))
    return GRPO_ERR_INVALID_ARG;
  if (beta != 0.f && !ok_f32(ref_logp)) return GRPO_ERR_INVALID_ARG;
  if (ref_logp != nullptr && !aligned(ref_logp, 4)) return GRPO_ERR_INVALID_ARG;
  const int64_t rows = logits->B * logits->L;
  grpo::FusedParams q{};
  FwdParams& p = q.f;
  p.x = view_of(logits);
  p.idx = idx;
  p.old_logp = old_logp;
  p.ref_logp = ref_logp;
  p.adv = adv;
  p.mask = mask;
  p.c = static_cast<float>(kLog2eD / static_cast<double>(T));
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
  q.dx = grpo::OutView{dlogits->ptr, dlogits->L, dlogits->stride_b, dlogits->stride_l, static_cast<int>(dlogits->V)};
  q.dloss = dloss;
  q.T = T;
  return from_cuda(grpo::launch_fused(logits->dtype, q, rows, same_phase, device_sms(),
                                      reinterpret_cast<cudaStream_t>(stream)));
}

grpo_status entropy_from_logits(const grpo_rows* logits, float T, float* entropy, float* lse,
                                grpo_stream_t stream) {
  grpo_status st = check_rows(logits);
  if (st != GRPO_OK) return st;
  if (!finite_pos(T)) return GRPO_ERR_INVALID_ARG;
  if (rows_of(logits) == 0) return GRPO_OK;
  if (!ok_f32(entropy) || !ok_opt_f32(lse)) return GRPO_ERR_INVALID_ARG;
  const int64_t rows = logits->B * logits->L;
  if (rows == 0) return GRPO_OK;
  FwdParams p{};
  p.x = view_of(logits);
  p.c = static_cast<float>(kLog2eD / static_cast<double>(T));
  p.invT = static_cast<float>(1.0 / static_cast<double>(T));
  p.entropy = entropy;
  p.lse = lse;
  return from_cuda(grpo::launch_fwd(grpo::kFwdEntropy, logits->dtype, p, rows, device_sms(), reinterpret_cast<cudaStream_t>(stream)));
}

grpo_status entropy_from_logits_bwd(const grpo_rows* logits, const float* dentropy, const float* lse,
                                    const float* entropy, float T, const grpo_rows* dlogits,
                                    grpo_stream_t stream) {
  grpo_status st = check_rows(logits);
  if (st != GRPO_OK) return st;
  if (!finite_pos(T)) return GRPO_ERR_INVALID_ARG;
  bool same_phase = false;
  if ((st = check_dlogits(logits, dlogits, &same_phase)) != GRPO_OK) return st;
  if (rows_of(logits) == 0) return GRPO_OK;
  if (!ok_f32(dentropy) || !ok_f32(lse) || !ok_f32(entropy)) return GRPO_ERR_INVALID_ARG;
  const int64_t rows = logits->B * logits->L;
  BwdParams p{};
  p.x = view_of(logits);
  p.dx = grpo::OutView{dlogits->ptr, dlogits->L, dlogits->stride_b, dlogits->stride_l,
                       static_cast<int>(dlogits->V)};
  p.lse = lse;
  p.dentropy = dentropy;
  p.entropy = entropy;
  p.c = static_cast<float>(kLog2eD / static_cast<double>(T));
  p.T = T;
  return from_cuda(grpo::launch_entgrad(logits->dtype, same_phase, p, rows, device_sms(),
                                        reinterpret_cast<cudaStream_t>(stream)));
}

grpo_status selective_log_softmax_fwd(const grpo_rows* logits, const int64_t* idx, float T,
                                      float* logp, float* lse, int32_t* dev_err,
                                      grpo_stream_t stream) {
  grpo_status st = check_rows(logits);
  if (st != GRPO_OK) return st;
  if (!finite_pos(T)) return GRPO_ERR_INVALID_ARG;
  if (rows_of(logits) == 0) return GRPO_OK;
  if (!ok_i64(idx) || !ok_f32(logp) || !ok_f32(lse) || !ok_opt_i32(dev_err)) return GRPO_ERR_INVALID_ARG;
  const int64_t rows = logits->B * logits->L;
  if (rows == 0) return GRPO_OK;
  FwdParams p{};
  p.x = view_of(logits);
  p.idx = idx;
  p.c = static_cast<float>(kLog2eD / static_cast<double>(T));
  p.invT = static_cast<float>(1.0 / static_cast<double>(T));
  p.logp = logp;
  p.lse = lse;
  p.dev_err = dev_err;
  return from_cuda(grpo::launch_fwd(grpo::kFwdSlsm, logits->dtype, p, rows, device_sms(), reinterpret_cast<cudaStream_t>(stream)));
}

grpo_status selective_log_softmax_bwd(const grpo_rows* logits, const int64_t* idx,
                                      const float* dlogp, const float* lse, float T,
                                      const grpo_rows* dlogits, int32_t* dev_err,
                                      grpo_stream_t stream) {
  grpo_status st = check_rows(logits);
  if (st != GRPO_OK) return st;
  if (!finite_pos(T)) return GRPO_ERR_INVALID_ARG;
  bool same_phase = false;
  if ((st = check_dlogits(logits, dlogits, &same_phase)) != GRPO_OK) return st;
  if (rows_of(logits) == 0) return GRPO_OK;
  if (!ok_i64(idx) || !ok_f32(dlogp) || !ok_f32(lse) || !ok_opt_i32(dev_err))
    return GRPO_ERR_INVALID_ARG;
  const int64_t rows = logits->B * logits->L;
  if (rows == 0) return GRPO_OK;
  BwdParams p{};
  p.x = view_of(logits);
  p.dx = grpo::OutView{dlogits->ptr, dlogits->L, dlogits->stride_b, dlogits->stride_l,
                       static_cast<int>(dlogits->V)};
  p.idx = idx;
  p.lse = lse;
  p.dlogp_up = dlogp;
  p.c = static_cast<float>(kLog2eD / static_cast<double>(T));
  p.T = T;
  p.dev_err = dev_err;
  return from_cuda(grpo::launch_bwd(false, logits->dtype, same_phase, p, rows, device_sms(),
                                    reinterpret_cast<cudaStream_t>(stream)));
}

grpo_status grpo_seq_terms(int64_t B, int64_t L, const float* logp, const float* old_logp,
                           const float* ref_logp, const float* adv, const uint8_t* mask, const float* dloss,
                           float beta, float eps_low, float eps_high, float* loss, float* kl, float* dlogp,
                           float* seq_ratio, uint8_t* seq_is_clipped, grpo_stream_t stream) {
  if (B < 0 || L < 0) return GRPO_ERR_INVALID_ARG;
  if (static_cast<long double>(B) * L > kMaxRows) return GRPO_ERR_UNSUPPORTED;
  if (!std::isfinite(beta) || beta < 0.f) return GRPO_ERR_INVALID_ARG;
  if (!std::isfinite(eps_low) || eps_low < 0.f || eps_low > 1.f) return GRPO_ERR_INVALID_ARG;
  if (!std::isfinite(eps_high) || eps_high < 0.f) return GRPO_ERR_INVALID_ARG;
  if (B == 0 || L == 0) return GRPO_OK;
  if (!ok_f32(logp) || !ok_opt_f32(old_logp) || !ok_f32(adv) || !ok_f32(dloss) || !ok_f32(loss) ||
      !ok_opt_f32(kl) || !ok_f32(dlogp) || !ok_opt_f32(seq_ratio))
    return GRPO_ERR_INVALID_ARG;
  if (beta != 0.f && !ok_f32(ref_logp)) return GRPO_ERR_INVALID_ARG;
  if (ref_logp != nullptr && !aligned(ref_logp, 4)) return GRPO_ERR_INVALID_ARG;
  grpo::SeqParams p{};
  p.B = B;
  p.L = L;
  p.logp = logp;
  p.old_logp = old_logp;
  p.ref_logp = ref_logp;
  p.adv = adv;
  p.mask = mask;
  p.dloss = dloss;
  p.beta = beta;
  p.lo = static_cast<float>(1.0 - static_cast<double>(eps_low));
  p.hi = static_cast<float>(1.0 + static_cast<double>(eps_high));
  p.loss = loss;
  p.kl = kl;
  p.dlogp = dlogp;
  p.seq_ratio = seq_ratio;
  p.seq_is_clipped = seq_is_clipped;
  return from_cuda(grpo::launch_seq(p, reinterpret_cast<cudaStream_t>(stream)));
}

grpo_status grpo_vocab_shard_stats(const grpo_rows* logits_shard, int64_t vocab_start, const int64_t* idx,
                                   const uint8_t* mask, float T, float* stats, grpo_stream_t stream) {
  grpo_status st = check_rows(logits_shard);
  if (st != GRPO_OK) return st;
  if (!finite_pos(T) || vocab_start < 0) return GRPO_ERR_INVALID_ARG;
  const int64_t rows = rows_of(logits_shard);
  if (rows == 0) return GRPO_OK;
  if (stats == nullptr || !aligned(stats, 16) || (idx != nullptr && !aligned(idx, 8)))
    return GRPO_ERR_INVALID_ARG;
  FwdParams p{};
  p.x = view_of(logits_shard);
  p.idx = idx;
  p.mask = mask;
  p.c = static_cast<float>(kLog2eD / static_cast<double>(T));
  p.invT = static_cast<float>(1.0 / static_cast<double>(T));
  p.vocab_start = vocab_start;
  p.stats = stats;
  return from_cuda(grpo::launch_fwd(grpo::kFwdShard, logits_shard->dtype, p, rows, device_sms(),
                                    reinterpret_cast<cudaStream_t>(stream)));
}

grpo_status grpo_vocab_combine(int32_t world, const float* stats_all, const int64_t* vocab_starts, int64_t B,
                               int64_t L, const int64_t* idx, const float* old_logp, const float* ref_logp,
                               const float* adv, const uint8_t* mask, float T, float beta, float eps_low,
                               float eps_high, float* loss, float* logp, float* lse, float* kl,
                               uint8_t* is_clipped, float* entropy, float* p_rest, int32_t* dev_err,
                               grpo_stream_t stream) {
  if (world < 1 || world > grpo::kVocabMaxWorld || vocab_starts == nullptr) return GRPO_ERR_INVALID_ARG;
  if (vocab_starts[0] != 0) return GRPO_ERR_INVALID_ARG;
  for (int k = 0; k < world; ++k)
    if (vocab_starts[k + 1] <= vocab_starts[k]) return GRPO_ERR_INVALID_ARG;
  if (vocab_starts[world] > kMaxV) return GRPO_ERR_UNSUPPORTED;
  if (B < 0 || L < 0) return GRPO_ERR_INVALID_ARG;
  if (static_cast<long double>(B) * L > kMaxRows) return GRPO_ERR_UNSUPPORTED;
  const bool grpo = loss != nullptr;
  if (!finite_pos(T)) return GRPO_ERR_INVALID_ARG;
  if (grpo) {
    grpo_status st = check_scalars_grpo(T, beta, eps_low, eps_high);
    if (st != GRPO_OK) return st;
  }
  const int64_t rows = B * L;
  if (rows == 0) return GRPO_OK;
  if (stats_all == nullptr || !aligned(stats_all, 16) || !ok_f32(lse) || !ok_opt_f32(entropy) ||
      !ok_opt_f32(p_rest) || !ok_opt_i32(dev_err))
    return GRPO_ERR_INVALID_ARG;
  if (idx == nullptr) {
    if (logp != nullptr || loss != nullptr || p_rest != nullptr) return GRPO_ERR_INVALID_ARG;
  } else if (!ok_i64(idx) || !ok_f32(logp)) {
    return GRPO_ERR_INVALID_ARG;
  }
  if (grpo) {
    if (!ok_f32(loss) || !ok_opt_f32(old_logp) || !ok_f32(adv) || !ok_opt_f32(kl)) return GRPO_ERR_INVALID_ARG;
    if (beta != 0.f && !ok_f32(ref_logp)) return GRPO_ERR_INVALID_ARG;
    if (ref_logp != nullptr && !aligned(ref_logp, 4)) return GRPO_ERR_INVALID_ARG;
  } else if (kl != nullptr || is_clipped != nullptr) {
    return GRPO_ERR_INVALID_ARG;
  }
  grpo::VocabCombineParams q{};
  q.world = world;
  for (int k = 0; k <= world; ++k) q.starts[k] = vocab_starts[k];
  q.stats = stats_all;
  q.rows = rows;
  q.p_rest = p_rest;
  FwdParams& p = q.f;
  p.x = grpo::RowsView{nullptr, L, 0, 0, static_cast<int>(vocab_starts[world])};
  p.idx = idx;
  p.old_logp = old_logp;
  p.ref_logp = ref_logp;
  p.adv = adv;
  p.mask = mask;
  p.c = static_cast<float>(kLog2eD / static_cast<double>(T));
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
  return from_cuda(grpo::launch_vocab_combine(q, grpo, reinterpret_cast<cudaStream_t>(stream)));
}

grpo_status grpo_loss_bwd_vocab_shard(const grpo_rows* logits_shard, int64_t vocab_start, int64_t vocab_total,
                                      const int64_t* idx, const float* old_logp, const float* ref_logp,
                                      const float* adv, const uint8_t* mask, const float* dloss,
                                      const float* logp, const float* lse, const float* p_rest, float T,
                                      float beta, float eps_low, float eps_high, const grpo_rows* dlogits_shard,
                                      int32_t* dev_err, grpo_stream_t stream) {
  grpo_status st = check_rows(logits_shard);
  if (st != GRPO_OK) return st;
  if ((st = check_scalars_grpo(T, beta, eps_low, eps_high)) != GRPO_OK) return st;
  if (vocab_start < 0 || vocab_total < vocab_start + logits_shard->V || vocab_total > kMaxV)
    return GRPO_ERR_INVALID_ARG;
  bool same_phase = false;
  if ((st = check_dlogits(logits_shard, dlogits_shard, &same_phase)) != GRPO_OK) return st;
  const int64_t rows = rows_of(logits_shard);
  if (rows == 0) return GRPO_OK;
  if (!ok_i64(idx) || !ok_opt_f32(old_logp) || !ok_f32(adv) || !ok_f32(dloss) || !ok_f32(logp) ||
      !ok_f32(lse) || !ok_f32(p_rest) || !ok_opt_i32(dev_err))
    return GRPO_ERR_INVALID_ARG;
  if (beta != 0.f && !ok_f32(ref_logp)) return GRPO_ERR_INVALID_ARG;
  if (ref_logp != nullptr && !aligned(ref_logp, 4)) return GRPO_ERR_INVALID_ARG;
  BwdParams p{};
  p.x = view_of(logits_shard);
  p.dx = grpo::OutView{dlogits_shard->ptr, dlogits_shard->L, dlogits_shard->stride_b, dlogits_shard->stride_l,
                       static_cast<int>(dlogits_shard->V)};
  p.idx = idx;
  p.lse = lse;
  p.old_logp = old_logp;
  p.ref_logp = ref_logp;
  p.adv = adv;
  p.mask = mask;
  p.dloss = dloss;
  p.logp = logp;
  p.c = static_cast<float>(kLog2eD / static_cast<double>(T));
  p.T = T;
  p.beta = beta;
  p.lo = static_cast<float>(1.0 - static_cast<double>(eps_low));
  p.hi = static_cast<float>(1.0 + static_cast<double>(eps_high));
  p.dev_err = dev_err;
  p.vocab_start = vocab_start;
  p.vocab_total = vocab_total;
  p.p_rest = p_rest;
  return from_cuda(grpo::launch_bwd_shard(true, logits_shard->dtype, same_phase, p, rows, device_sms(),
                                          reinterpret_cast<cudaStream_t>(stream)));
}

grpo_status selective_log_softmax_bwd_vocab_shard(const grpo_rows* logits_shard, int64_t vocab_start,
                                                  int64_t vocab_total, const int64_t* idx, const float* dlogp,
                                                  const float* lse, const float* p_rest, float T,
                                                  const grpo_rows* dlogits_shard, int32_t* dev_err,
                                                  grpo_stream_t stream) {
  grpo_status st = check_rows(logits_shard);
  if (st != GRPO_OK) return st;
  if (!finite_pos(T)) return GRPO_ERR_INVALID_ARG;
  if (vocab_start < 0 || vocab_total < vocab_start + logits_shard->V || vocab_total > kMaxV)
    return GRPO_ERR_INVALID_ARG;
  bool same_phase = false;
  if ((st = check_dlogits(logits_shard, dlogits_shard, &same_phase)) != GRPO_OK) return st;
  const int64_t rows = rows_of(logits_shard);
  if (rows == 0) return GRPO_OK;
  if (!ok_i64(idx) || !ok_f32(dlogp) || !ok_f32(lse) || !ok_f32(p_rest) || !ok_opt_i32(dev_err))
    return GRPO_ERR_INVALID_ARG;
  BwdParams p{};
  p.x = view_of(logits_shard);
  p.dx = grpo::OutView{dlogits_shard->ptr, dlogits_shard->L, dlogits_shard->stride_b, dlogits_shard->stride_l,
                       static_cast<int>(dlogits_shard->V)};
  p.idx = idx;
  p.lse = lse;
  p.dlogp_up = dlogp;
  p.c = static_cast<float>(kLog2eD / static_cast<double>(T));
  p.T = T;
  p.dev_err = dev_err;
  p.vocab_start = vocab_start;
  p.vocab_total = vocab_total;
  p.p_rest = p_rest;
  return from_cuda(grpo::launch_bwd_shard(false, logits_shard->dtype, same_phase, p, rows, device_sms(),
                                          reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {
// Room for the K splits of grad_hidden's GEMM: 16 splits of a 2048-row chunk at H = 1024,
// and never less than one split.
constexpr uint64_t kLinearSplitWs = uint64_t(128) << 20;
}  // namespace

extern "C" {

grpo_status grpo_fused_linear_workspace_size(int64_t H, int64_t V, int64_t chunk_rows, uint64_t* bytes) {
  if (bytes == nullptr || H < 8 || H % 8 != 0 || H > (int64_t(1) << 24) || V < 1 || V > kMaxV || chunk_rows < 1 ||
      chunk_rows > kMaxRows)
    return GRPO_ERR_INVALID_ARG;
  const uint64_t one_split = grpo::linear_round256(static_cast<uint64_t>(chunk_rows) * H * 4);
  *bytes = grpo::linear_chunk_bytes(H, V, chunk_rows) + std::max(kLinearSplitWs, one_split);
  return GRPO_OK;
}

grpo_status grpo_fused_linear(const void* hidden, const void* weight, int64_t B, int64_t L, int64_t H, int64_t V,
                              const int64_t* idx, const float* old_logp, const float* ref_logp, const float* adv,
                              const uint8_t* mask, const float* dloss, float T, float beta, float eps_low,
                              float eps_high, int64_t chunk_rows, void* workspace, uint64_t workspace_bytes,
                              float* loss, float* logp, float* lse, float* kl, uint8_t* is_clipped, float* entropy,
                              float* grad_hidden, float* grad_weight, int32_t* dev_err, grpo_stream_t stream) {
  grpo_status st = check_scalars_grpo(T, beta, eps_low, eps_high);
  if (st != GRPO_OK) return st;
  if (B < 0 || L < 0 || H < 8 || H % 8 != 0 || V < 1 || chunk_rows < 1) return GRPO_ERR_INVALID_ARG;
  if (V > kMaxV || static_cast<long double>(B) * L > kMaxRows || H > (int64_t(1) << 24)) return GRPO_ERR_UNSUPPORTED;
  const int64_t rows = B * L;
  if (rows == 0) return GRPO_OK;
  uint64_t need = 0;
  const int64_t chunk = chunk_rows < rows ? chunk_rows : rows;
  grpo_fused_linear_workspace_size(H, V, chunk, &need);
  if (hidden == nullptr || !aligned(hidden, 16) || weight == nullptr || !aligned(weight, 16) ||
      workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < need)
    return GRPO_ERR_INVALID_ARG;
  if (!ok_i64(idx) || !ok_opt_f32(old_logp) || !ok_f32(adv) || !ok_f32(dloss) || !ok_f32(loss) || !ok_f32(logp) ||
      !ok_f32(lse) || !ok_opt_f32(kl) || !ok_opt_f32(entropy) || !ok_opt_i32(dev_err))
    return GRPO_ERR_INVALID_ARG;
  if ((grad_hidden != nullptr && !aligned(grad_hidden, 16)) || (grad_weight != nullptr && !aligned(grad_weight, 16)))
    return GRPO_ERR_INVALID_ARG;
  if (beta != 0.f && !ok_f32(ref_logp)) return GRPO_ERR_INVALID_ARG;
  if (ref_logp != nullptr && !aligned(ref_logp, 4)) return GRPO_ERR_INVALID_ARG;
  grpo::FusedLinearParams q{};
  q.hidden = static_cast<const uint16_t*>(hidden);
  q.weight = static_cast<const uint16_t*>(weight);
  q.rows = rows;
  q.H = H;
  q.V = V;
  q.chunk = chunk;
  q.ld = grpo::linear_ld(V);
  grpo::linear_carve(q, static_cast<char*>(workspace), need);
  q.grad_hidden = grad_hidden;
  q.grad_weight = grad_weight;
  grpo::LinearChunkParams& cp = q.chunk_params;
  FwdParams& p = cp.f;
  p.x = grpo::RowsView{nullptr, L, 0, 0, static_cast<int>(V)};
  p.idx = idx;
  p.old_logp = old_logp;
  p.ref_logp = ref_logp;
  p.adv = adv;
  p.mask = mask;
  p.c = static_cast<float>(kLog2eD / static_cast<double>(T));
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
  return from_cuda(grpo::launch_fused_linear(q, reinterpret_cast<cudaStream_t>(stream)));
}

const char* grpo_status_string(grpo_status status) {
  switch (status) {
    case GRPO_OK: return "GRPO_OK";
    case GRPO_ERR_INVALID_ARG: return "GRPO_ERR_INVALID_ARG: invalid pointer, size, stride, scalar or aliasing";
    case GRPO_ERR_UNSUPPORTED: return "GRPO_ERR_UNSUPPORTED: valid arguments outside what the library handles";
    case GRPO_ERR_CUDA: return "GRPO_ERR_CUDA: the kernel launch failed";
    default: return "unknown grpo_status";
  }
}

}  // extern "C"
