// Fused GRPO forward + backward instantiated for BF16 logits (see rowpass_fused.cuh).
#include "rowpass_fused.cuh"

namespace grpo {
cudaError_t launch_fused_bf16(const FusedParams& q, int64_t rows, bool same_phase, int sms, cudaStream_t stream) {
  return launch_fused_dtype<BF16>(q, rows, same_phase, sms, stream);
}
}  // namespace grpo
