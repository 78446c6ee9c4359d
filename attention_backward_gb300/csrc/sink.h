// Gradient of per-query-head attention-sink logits from the LSE2 and delta
// rows that the preprocess leaves in the workspace (kernel in preprocess.cu).
#pragma once
#include <cuda_runtime.h>

namespace ab {

struct SinkGradParams {
  const float* sink;   // [H] logits (natural-log units)
  const float* lse2;   // [B,H,S] workspace, LSE * log2(e) of the sink-aware forward
  const float* delta;  // [B,H,S] workspace
  int B, S, H;
  const int* cu_seqlens;  // packed rows [cu[0], cu[num_seqs]) (B == 1), or null: all rows
  int num_seqs;
  float* dsink;  // [H]
};

cudaError_t launch_sink_grad(const SinkGradParams& p, cudaStream_t st);

}  // namespace ab
