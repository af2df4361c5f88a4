// Forward row kernels instantiated for BF16 logits (see rowpass_fwd.cuh).
#include "rowpass_fwd.cuh"

namespace grpo {
cudaError_t launch_fwd_bf16(int mode, const FwdParams& p, int64_t rows, int sms, cudaStream_t stream) {
  return launch_dtype<BF16>(mode, p, rows, sms, stream);
}
}  // namespace grpo
