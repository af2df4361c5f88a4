// Backward row kernels instantiated for F32 logits (see rowpass_bwd.cuh).
#include "rowpass_bwd.cuh"

namespace grpo {
cudaError_t launch_bwd_f32(bool grpo, bool same_phase, const BwdParams& p, int64_t rows, int sms,
                            cudaStream_t stream) {
  return launch2<F32>(grpo, same_phase, p, rows, sms, stream);
}
cudaError_t launch_bwd_shard_f32(bool grpo, bool same_phase, const BwdParams& p, int64_t rows, int sms,
                                  cudaStream_t stream) {
  return launch2<F32, true>(grpo, same_phase, p, rows, sms, stream);
}
cudaError_t launch_entgrad_f32(bool same_phase, const BwdParams& p, int64_t rows, int sms, cudaStream_t stream) {
  return launch_entgrad_dtype<F32>(same_phase, p, rows, sms, stream);
}
}  // namespace grpo
