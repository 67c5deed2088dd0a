// Parameters and launcher of the row softmax of the materialising baseline
// (scores written to HBM, read for the softmax, probabilities written, read
// for the value product).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace fa {

struct MaterializedParams {
  void* s;           // bf16 [rows, Nk]: scale * Q K^T in, probabilities out (in place)
  float* lse;        // fp32 [rows] (natural log) or nullptr
  long long rows;    // B * H * Nq
  int Nq, Nk;
  int causal;        // key j visible to query i iff j <= i + Nk - Nq
};

cudaError_t launch_materialized_softmax(const MaterializedParams& p, cudaStream_t stream);
cudaError_t materialized_set_attributes();
// largest Nk one CTA's shared memory holds (one fp32 row)
constexpr int MATERIALIZED_MAX_NK = (227 * 1024) / 4 - 64;

}  // namespace fa
