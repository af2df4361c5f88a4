// Forward row kernels instantiated for F32 logits (see rowpass_fwd.cuh).
#include "rowpass_fwd.cuh"

namespace grpo {
cudaError_t launch_fwd_f32(int mode, const FwdParams& p, int64_t rows, int sms, cudaStream_t stream) {
  return launch_dtype<F32>(mode, p, rows, sms, stream);
}
}  // namespace grpo
