// Row softmax of the materialising baseline ("Explain FlashAttention ...",
// section "What the byte arithmetic does and does not say": a baseline that
// writes the scores, reads them for the softmax, writes the probabilities and
// reads them for the value product). The two products are library GEMMs; this
// kernel is the middle pass: one CTA per score row reads the row once from
// HBM into shared memory, forms the max and the sum of the exponentials over
// the visible keys in fp32, and writes P = exp(s - max) / sum (bf16) over the
// row in place, with lse = max + ln(sum) (-inf and P = 0 for a row that sees
// no key).
#include <cuda_bf16.h>

#include <cmath>

#include "materialized.cuh"

namespace fa {

namespace {

constexpr int MS_THREADS = 256;
constexpr float MS_LOG2E = 1.4426950408889634f;

__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// block-wide reduction over 256 threads (max when IS_MAX, else sum)
template <bool IS_MAX>
__device__ __forceinline__ float block_reduce(float x, float* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float y = __shfl_xor_sync(0xffffffffu, x, off);
    x = IS_MAX ? fmaxf(x, y) : x + y;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();  // red[] may still hold the previous reduction's values
  if (lane == 0) red[warp] = x;
  __syncthreads();
  x = red[0];
#pragma unroll
  for (int w = 1; w < MS_THREADS / 32; ++w) x = IS_MAX ? fmaxf(x, red[w]) : x + red[w];
  return x;
}

}  // namespace

__global__ void __launch_bounds__(MS_THREADS) fa_materialized_softmax_kernel(const MaterializedParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ float red[MS_THREADS / 32];
  uint4* srow = reinterpret_cast<uint4*>(smem);
  const long long row = blockIdx.x;
  const int i = static_cast<int>(row % p.Nq);
  const int limit = p.causal ? max(0, min(p.Nk, i + p.Nk - p.Nq + 1)) : p.Nk;  // keys below are visible
  uint4* g = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.s) + row * p.Nk);
  const int nv = p.Nk / 8;  // 16-byte vectors per row (Nk is a multiple of 8)

  float mx = -INFINITY;
  for (int c = threadIdx.x; c < nv; c += MS_THREADS) {
    const uint4 u = g[c];
    srow[c] = u;
    float f[8];
    unpack8(u, f);
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if (8 * c + e < limit) mx = fmaxf(mx, f[e]);
  }
  mx = block_reduce<true>(mx, red);
  float sum = 0.f;
  if (limit > 0) {
    for (int c = threadIdx.x; c < nv; c += MS_THREADS) {
      float f[8];
      unpack8(srow[c], f);
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (8 * c + e < limit) sum += exp2f((f[e] - mx) * MS_LOG2E);
    }
  }
  sum = block_reduce<false>(sum, red);
  const float inv = limit > 0 ? 1.f / sum : 0.f;
  for (int c = threadIdx.x; c < nv; c += MS_THREADS) {
    float f[8];
    unpack8(srow[c], f);
    float pr[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) pr[e] = (8 * c + e < limit) ? exp2f((f[e] - mx) * MS_LOG2E) * inv : 0.f;
    g[c] = make_uint4(pack2(pr[0], pr[1]), pack2(pr[2], pr[3]), pack2(pr[4], pr[5]), pack2(pr[6], pr[7]));
  }
  if (threadIdx.x == 0 && p.lse != nullptr) p.lse[row] = limit > 0 ? mx + logf(sum) : -INFINITY;
}

cudaError_t materialized_set_attributes() {
  return cudaFuncSetAttribute(fa_materialized_softmax_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              MATERIALIZED_MAX_NK * 2);
}

cudaError_t launch_materialized_softmax(const MaterializedParams& p, cudaStream_t stream) {
  fa_materialized_softmax_kernel<<<static_cast<unsigned>(p.rows), MS_THREADS, static_cast<size_t>(p.Nk) * 2, stream>>>(
      p);
  return cudaGetLastError();
}

}  // namespace fa
