// Row softmax of the materialising baseline ("Explain FlashAttention ...",
// section "What the byte arithmetic does and does not say": a baseline that
// writes the scores, reads them for the softmax, writes the probabilities and
// reads them for the value product). The two products are library GEMMs; this
// kernel is the middle pass: one CTA per score row reads the row once from
// HBM into shared memory (fp32), forms the max, the exponentials (the MUFU
// base-2 exponential, once per element) and their sum, and writes
// P = exp(s - max) / sum (bf16) over the row in place, with
// lse = max + ln(sum) (-inf and P = 0 for a row that sees no key).
#include <cuda_bf16.h>

#include <cmath>

#include "fa_ptx.cuh"
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
  float4* srow = reinterpret_cast<float4*>(smem);  // the row in fp32: scores, then exponentials
  const long long row = blockIdx.x;
  const int i = static_cast<int>(row % p.Nq);
  const int limit = p.causal ? max(0, min(p.Nk, i + p.Nk - p.Nq + 1)) : p.Nk;  // keys below are visible
  uint4* g = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.s) + row * p.Nk);
  const int nv = p.Nk / 8;  // 16-byte vectors per row (Nk is a multiple of 8)
  if (limit == 0) {  // no visible key: P = 0, lse = -inf
    for (int c = threadIdx.x; c < nv; c += MS_THREADS) g[c] = make_uint4(0u, 0u, 0u, 0u);
    if (threadIdx.x == 0 && p.lse != nullptr) p.lse[row] = -INFINITY;
    return;
  }
  // pass 1: the row into shared memory (masked keys -inf) and its max; only a
  // vector that crosses the limit needs per-element tests
  float mx = -INFINITY;
  for (int c = threadIdx.x; c < nv; c += MS_THREADS) {
    float f[8];
    unpack8(g[c], f);
    if (8 * c + 8 > limit) {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (8 * c + e >= limit) f[e] = -INFINITY;
    }
    srow[2 * c] = make_float4(f[0], f[1], f[2], f[3]);
    srow[2 * c + 1] = make_float4(f[4], f[5], f[6], f[7]);
    mx = fmaxf(mx, fmaxf(fmaxf(fmaxf(f[0], f[1]), fmaxf(f[2], f[3])), fmaxf(fmaxf(f[4], f[5]), fmaxf(f[6], f[7]))));
  }
  mx = block_reduce<true>(mx, red);
  // pass 2: the exponentials (in place) and their sum; -inf -> 0
  const float nm = -mx * MS_LOG2E;
  float sum = 0.f;
  for (int c = threadIdx.x; c < 2 * nv; c += MS_THREADS) {
    float4 x = srow[c];
    x.x = ex2_approx(fmaf(x.x, MS_LOG2E, nm));
    x.y = ex2_approx(fmaf(x.y, MS_LOG2E, nm));
    x.z = ex2_approx(fmaf(x.z, MS_LOG2E, nm));
    x.w = ex2_approx(fmaf(x.w, MS_LOG2E, nm));
    srow[c] = x;
    sum += (x.x + x.y) + (x.z + x.w);
  }
  sum = block_reduce<false>(sum, red);
  const float inv = 1.f / sum;
  // pass 3: P = exponential / sum, bf16, over the scores
  for (int c = threadIdx.x; c < nv; c += MS_THREADS) {
    const float4 a = srow[2 * c], b = srow[2 * c + 1];
    g[c] = make_uint4(pack2(a.x * inv, a.y * inv), pack2(a.z * inv, a.w * inv), pack2(b.x * inv, b.y * inv),
                      pack2(b.z * inv, b.w * inv));
  }
  if (threadIdx.x == 0 && p.lse != nullptr) p.lse[row] = mx + logf(sum);
}

// The same three passes with one warp per row and MS_WARP_ROWS rows per CTA
// (warp-shuffle reductions, no CTA barrier), for rows that fit eight to a CTA.
constexpr int MS_WARP_ROWS = 8;

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

__global__ void __launch_bounds__(32 * MS_WARP_ROWS) fa_materialized_softmax_warp_kernel(const MaterializedParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * MS_WARP_ROWS + warp;
  if (row >= p.rows) return;  // warp-uniform
  float4* srow = reinterpret_cast<float4*>(smem) + static_cast<size_t>(warp) * (p.Nk / 4);
  const int i = static_cast<int>(row % p.Nq);
  const int limit = p.causal ? max(0, min(p.Nk, i + p.Nk - p.Nq + 1)) : p.Nk;
  uint4* g = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.s) + row * p.Nk);
  const int nv = p.Nk / 8;
  if (limit == 0) {
    for (int c = lane; c < nv; c += 32) g[c] = make_uint4(0u, 0u, 0u, 0u);
    if (lane == 0 && p.lse != nullptr) p.lse[row] = -INFINITY;
    return;
  }
  float mx = -INFINITY;
  // eight 16-byte loads per lane in flight before any is used
  for (int c0 = lane; c0 < nv; c0 += 32 * 8) {
    uint4 u[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) u[k] = (c0 + 32 * k < nv) ? g[c0 + 32 * k] : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int c = c0 + 32 * k;
      if (c >= nv) break;
      float f[8];
      unpack8(u[k], f);
      if (8 * c + 8 > limit) {
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (8 * c + e >= limit) f[e] = -INFINITY;
      }
      srow[2 * c] = make_float4(f[0], f[1], f[2], f[3]);
      srow[2 * c + 1] = make_float4(f[4], f[5], f[6], f[7]);
      mx = fmaxf(mx,
                 fmaxf(fmaxf(fmaxf(f[0], f[1]), fmaxf(f[2], f[3])), fmaxf(fmaxf(f[4], f[5]), fmaxf(f[6], f[7]))));
    }
  }
  mx = warp_max(mx);
  __syncwarp();  // the next pass reads entries other lanes wrote
  const float nm = -mx * MS_LOG2E;
  float sum = 0.f;
  for (int c = lane; c < 2 * nv; c += 32) {
    float4 x = srow[c];
    x.x = ex2_approx(fmaf(x.x, MS_LOG2E, nm));
    x.y = ex2_approx(fmaf(x.y, MS_LOG2E, nm));
    x.z = ex2_approx(fmaf(x.z, MS_LOG2E, nm));
    x.w = ex2_approx(fmaf(x.w, MS_LOG2E, nm));
    srow[c] = x;
    sum += (x.x + x.y) + (x.z + x.w);
  }
  sum = warp_sum(sum);
  __syncwarp();
  const float inv = 1.f / sum;
  for (int c = lane; c < nv; c += 32) {
    const float4 a = srow[2 * c], b = srow[2 * c + 1];
    g[c] = make_uint4(pack2(a.x * inv, a.y * inv), pack2(a.z * inv, a.w * inv), pack2(b.x * inv, b.y * inv),
                      pack2(b.z * inv, b.w * inv));
  }
  if (lane == 0 && p.lse != nullptr) p.lse[row] = mx + logf(sum);
}

cudaError_t materialized_set_attributes() {
  cudaError_t e = cudaFuncSetAttribute(fa_materialized_softmax_warp_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, MATERIALIZED_MAX_NK * 4);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(fa_materialized_softmax_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              MATERIALIZED_MAX_NK * 4);
}

cudaError_t launch_materialized_softmax(const MaterializedParams& p, cudaStream_t stream) {
  const size_t warp_smem = static_cast<size_t>(MS_WARP_ROWS) * p.Nk * 4;
  if (warp_smem <= static_cast<size_t>(MATERIALIZED_MAX_NK) * 4) {
    const long long ctas = (p.rows + MS_WARP_ROWS - 1) / MS_WARP_ROWS;
    fa_materialized_softmax_warp_kernel<<<static_cast<unsigned>(ctas), 32 * MS_WARP_ROWS, warp_smem, stream>>>(p);
    return cudaGetLastError();
  }
  fa_materialized_softmax_kernel<<<static_cast<unsigned>(p.rows), MS_THREADS, static_cast<size_t>(p.Nk) * 4, stream>>>(
      p);
  return cudaGetLastError();
}

}  // namespace fa
