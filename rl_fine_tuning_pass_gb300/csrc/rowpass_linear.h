// Internal interface of the GRPO loss on top of the LM head (rowpass_linear.cu) for the
// C-ABI layer: the chunk parameter blocks, the workspace layout and the launcher.  Kept
// apart from rowpass_internal.h so that the row-pass kernels do not depend on it.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "rowpass_internal.h"

namespace grpo {

// The GRPO loss on top of the LM head, in chunks of rows (rowpass_linear.cu).
struct LinearChunkParams {
  FwdParams f;            // per-row inputs and outputs of the whole batch; f.x.L = tokens per
                          // sequence, f.x.V = vocabulary
  const float4* stats;    // the chunk's per-128-column statistics [rows][n_stat]
  uint16_t* dlogits;      // [rows][ld]: the logits GEMM's fp16 exponentials in, bf16 dlogits out
  const uint16_t* hidden_rows;  // the chunk's gathered hidden states [rows][H] bf16
  const uint16_t* weight;       // the head weight [V][H] bf16
  int64_t H;
  int64_t ld;             // elements between rows, a multiple of 8
  int n_stat;             // statistics slots per row (two per 256-column tile)
  const int32_t* list;    // the chunk's rows: row i of the chunk is batch row list[i]
  const int32_t* state;   // state[0]: how many rows the chunk holds (set on the device)
  int64_t chunk;          // rows of the chunk buffers
  const float* dloss;     // [batch rows]
  float T;
};
// One chunk's buffers: 16-bit [chunk][ld] (the logits GEMM's fp16 exponentials, then the row
// pass's bf16 dlogits in their place), the statistics of the logits GEMM [chunk][2 ceil(V / 256)], its
// hidden states gathered into consecutive rows [chunk][H] bf16, the batch rows they come from
// [chunk] and the chunk's state: [0] its number of rows, [1] the batch row after its last one.
struct LinearChunkBufs {
  uint16_t* dlogits;
  float4* stats;
  uint16_t* hidden;
  int32_t* list;
  int32_t* state;
};
struct FusedLinearParams {
  const uint16_t* hidden;  // [rows][H] bf16
  const uint16_t* weight;  // [V][H] bf16
  int64_t rows, H, V;
  int64_t chunk;           // rows per chunk
  int64_t ld;              // row stride of the chunk buffers (V rounded up to 8)
  LinearChunkBufs bufs;    // workspace: one chunk's buffers
  float* part;             // workspace: the K splits of grad_hidden [splits][chunk][H] fp32
  uint64_t part_bytes;     // its size (sets the number of splits)
  float* grad_hidden;      // [rows][H] fp32, or null
  float* grad_weight;      // [V][H] fp32, accumulated into, or null
  LinearChunkParams chunk_params;
};
// Sizes of the workspace parts for H, V and a chunk of rows (each rounded up to 256 bytes).
inline uint64_t linear_round256(uint64_t v) { return (v + 255) & ~uint64_t(255); }
inline int64_t linear_ld(int64_t V) { return (V + 7) / 8 * 8; }
inline int64_t linear_n_stat(int64_t V) { return 2 * ((V + 255) / 256); }
struct LinearChunkLayout {
  uint64_t dlogits, stats, hidden, list, state;  // bytes of each part
  uint64_t total() const { return dlogits + stats + hidden + list + state; }
};
inline LinearChunkLayout linear_chunk_layout(int64_t H, int64_t V, int64_t chunk) {
  const uint64_t ld = static_cast<uint64_t>(linear_ld(V)), c = static_cast<uint64_t>(chunk);
  return LinearChunkLayout{linear_round256(ld * c * 2),
                           linear_round256(static_cast<uint64_t>(linear_n_stat(V)) * c * 16),
                           linear_round256(static_cast<uint64_t>(H) * c * 2),
                           linear_round256(c * 4),
                           256};
}
inline uint64_t linear_chunk_bytes(int64_t H, int64_t V, int64_t chunk) {
  return linear_chunk_layout(H, V, chunk).total();
}
// Carve the chunk buffers out of `base`; the rest of total_bytes holds grad_hidden's K splits.
inline void linear_carve(FusedLinearParams& q, char* base, uint64_t total_bytes) {
  const LinearChunkLayout l = linear_chunk_layout(q.H, q.V, q.chunk);
  char* p = base;
  q.bufs.dlogits = reinterpret_cast<uint16_t*>(p);
  p += l.dlogits;
  q.bufs.stats = reinterpret_cast<float4*>(p);
  p += l.stats;
  q.bufs.hidden = reinterpret_cast<uint16_t*>(p);
  p += l.hidden;
  q.bufs.list = reinterpret_cast<int32_t*>(p);
  p += l.list;
  q.bufs.state = reinterpret_cast<int32_t*>(p);
  p += l.state;
  q.part = reinterpret_cast<float*>(p);
  q.part_bytes = total_bytes - l.total();
}
cudaError_t launch_fused_linear(const FusedLinearParams& q, cudaStream_t stream);

}  // namespace grpo
