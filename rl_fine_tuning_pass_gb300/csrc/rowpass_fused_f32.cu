// Fused GRPO forward + backward instantiated for F32 logits (see rowpass_fused.cuh).
#include "rowpass_fused.cuh"

namespace grpo {
cudaError_t launch_fused_f32(const FusedParams& q, int64_t rows, bool same_phase, int sms, cudaStream_t stream) {
  return launch_fused_dtype<F32>(q, rows, same_phase, sms, stream);
}
}  // namespace grpo
