// Parameters and launcher of the split-KV decode for grouped K/V heads, several
// query tokens per sequence and per-sequence KV lengths (tensor-core kernels,
// and a CUDA-core kernel for groups of at most four query rows).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa_common.cuh"

namespace fa {

struct DecodeGroupedParams {
  const void* q;             // bf16 [B, H, Nq, d]       (read by the CUDA-core kernel; the others use tensor maps)
  const void* k;             // bf16 [B, Hkv, Nk, d]
  const void* v;             // bf16 [B, Hkv, Nk, d]
  const int* seqlens;        // int32 [B] keys per sequence (device), or nullptr: every sequence has Nk
  float* ws_o;               // fp32 [B*H*Nq, S, d]  unnormalised partial outputs
  float* ws_ml;              // fp32 [B*H*Nq, S, 2]  partial (reference max in log2 units, sum)
  int B, H, Hkv, G, Nq, R;   // G = H / Hkv query heads per K/V head; R = G * Nq rows per tile
  int Nk;                    // keys in the cache per (b, kv head)
  int S, chunk;              // splits; keys per split (a multiple of 128)
  float scale_log2;          // |scale| * log2(e)
  int negate_s;              // scale < 0: the score MMA computes -(Q K^T)
  uint64_t wait_limit_ns;
  unsigned int* status;      // device status word
};

cudaError_t launch_decode_grouped(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                  const DecodeGroupedParams& p, cudaStream_t stream);
cudaError_t decode_grouped_set_attributes(int d);
// Rows of the Q tensor map's box the kernel chosen for (d, R = G * Nq query
// rows per K/V head) loads: the launcher picks the kernel by the same rule.
int decode_grouped_q_box_rows(int d, int R);
// The split-KV decode's merge pass alone (defined with the split-KV decode).
cudaError_t launch_decode_merge(int d, const DecodeParams& p, cudaStream_t stream);

}  // namespace fa
