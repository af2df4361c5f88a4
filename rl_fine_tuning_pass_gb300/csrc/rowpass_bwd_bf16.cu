// Backward row kernels instantiated for BF16 logits (see rowpass_bwd.cuh).
#include "rowpass_bwd.cuh"

namespace grpo {
cudaError_t launch_bwd_bf16(bool grpo, bool same_phase, const BwdParams& p, int64_t rows, int sms,
                            cudaStream_t stream) {
  return launch2<BF16>(grpo, same_phase, p, rows, sms, stream);
}
cudaError_t launch_bwd_shard_bf16(bool grpo, bool same_phase, const BwdParams& p, int64_t rows, int sms,
                                  cudaStream_t stream) {
  return launch2<BF16, true>(grpo, same_phase, p, rows, sms, stream);
}
cudaError_t launch_entgrad_bf16(bool same_phase, const BwdParams& p, int64_t rows, int sms, cudaStream_t stream) {
  return launch_entgrad_dtype<BF16>(same_phase, p, rows, sms, stream);
}
}  // namespace grpo
