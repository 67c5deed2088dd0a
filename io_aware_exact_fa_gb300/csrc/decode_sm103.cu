// Split-KV decode for one query token per (b, h), and the merge of the
// per-split partial states.
//
// Decode is a matrix-vector product against the whole KV cache, bound by
// streaming K and V from HBM; Flash-Decoding splits the K/V sequence and
// merges the partial results ("FlashAttention: Attention Is Limited by
// Memory, Not Math", section "Where it helps, and where it does not").
// The merge re-bases each split to the global max with one scalar per split
// ("Handwritten Notes on Flash Attention", section "Merging two blocks").
//
// Split kernel: one CTA (4 warps) per (split, b*h). A key row of d bf16 is
// read by d/8 lanes with one 16-byte load each, so a warp-wide load covers
// 32*16 = 512 contiguous bytes (2 keys at d = 128, 4 at d = 64). Each lane
// group keeps its own online state (m, l, o-slice) in log2 units; groups and
// warps are combined at the end and the split writes its unnormalised
// partial (o_s, m_s, l_s) to the caller's workspace.
// Merge kernel: one CTA per (b, h), one thread per output element.
#include <cuda_bf16.h>

#include <cstdio>
#include <mutex>

#include "fa.h"
#include "fa_ptx.cuh"

namespace fa {

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// exp2(m - M) with the empty-state convention: a part that saw no key (m = -inf)
// contributes nothing.
__device__ __forceinline__ float rebase(float m, float M) {
  return (m == -INFINITY) ? 0.f : ex2_approx(m - M);
}

template <int D>
__global__ void __launch_bounds__(128) fa_decode_split_kernel(const DecodeParams p) {
  constexpr int LPK = D / 8;        // lanes per key row
  constexpr int KPW = 32 / LPK;     // keys per warp-wide load
  constexpr int ROUND = 4 * KPW;    // keys per CTA-wide load round
  constexpr int U = 4;              // rounds in flight per iteration
  const int s = blockIdx.x % p.S;
  const int bh = blockIdx.x / p.S;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPK;
  const int li = lane % LPK;
  const int k0 = s * p.chunk;
  const int k1 = min(p.Nk, k0 + p.chunk);

  const __nv_bfloat16* kbase = reinterpret_cast<const __nv_bfloat16*>(p.k) + static_cast<size_t>(bh) * p.Nk * D;
  const __nv_bfloat16* vbase = reinterpret_cast<const __nv_bfloat16*>(p.v) + static_cast<size_t>(bh) * p.Nk * D;

  float q[8];
  bf16x8_to_f32(*reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(p.q) + static_cast<size_t>(bh) * D + li * 8), q);
#pragma unroll
  for (int e = 0; e < 8; ++e) q[e] *= p.scale_log2;  // scores come out in log2 units

  float m = -INFINITY, l = 0.f;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;

  // the trip count is warp-uniform (every lane runs the same shuffles)
  for (int base0 = k0 + warp * KPW; base0 < k1; base0 += ROUND * U) {
    const int base = base0 + sub;
    uint4 kr[U], vr[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int key = base + u * ROUND;
      if (key < k1) {
        kr[u] = ldg_stream(kbase + static_cast<size_t>(key) * D + li * 8);
        vr[u] = ldg_stream(vbase + static_cast<size_t>(key) * D + li * 8);
      } else {
        kr[u] = make_uint4(0, 0, 0, 0);
        vr[u] = make_uint4(0, 0, 0, 0);
      }
    }
    float sc[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float kf[8];
      bf16x8_to_f32(kr[u], kf);
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) dot = fmaf(q[e], kf[e], dot);
#pragma unroll
      for (int off = LPK / 2; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
      sc[u] = (base + u * ROUND < k1) ? dot : -INFINITY;
    }
    float mx = sc[0];
#pragma unroll
    for (int u = 1; u < U; ++u) mx = fmaxf(mx, sc[u]);
    if (mx == -INFINITY) continue;  // group-uniform: no key of this group in range
    const float m_new = fmaxf(m, mx);
    const float alpha = rebase(m, m_new);
    l *= alpha;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] *= alpha;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const float pu = ex2_approx(sc[u] - m_new);  // -inf -> 0
      l += pu;
      float vf[8];
      bf16x8_to_f32(vr[u], vf);
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = fmaf(pu, vf[e], acc[e]);
    }
    m = m_new;
  }

  // combine the KPW lane groups of this warp (same output slice li)
#pragma unroll
  for (int off = LPK; off < 32; off <<= 1) {
    const float mo = __shfl_xor_sync(0xffffffffu, m, off);
    const float lo = __shfl_xor_sync(0xffffffffu, l, off);
    const float M = fmaxf(m, mo);
    const float a = rebase(m, M), b = rebase(mo, M);
    l = l * a + lo * b;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float ao = __shfl_xor_sync(0xffffffffu, acc[e], off);
      acc[e] = acc[e] * a + ao * b;
    }
    m = M;
  }

  // combine the 4 warps
  __shared__ float sm_m[4], sm_l[4];
  __shared__ float sm_acc[4][D];
  if (sub == 0) {
#pragma unroll
    for (int e = 0; e < 8; ++e) sm_acc[warp][li * 8 + e] = acc[e];
    if (li == 0) {
      sm_m[warp] = m;
      sm_l[warp] = l;
    }
  }
  __syncthreads();
  const size_t part = static_cast<size_t>(bh) * p.S + s;
  if (threadIdx.x < D) {
    const int c = threadIdx.x;
    float M = fmaxf(fmaxf(sm_m[0], sm_m[1]), fmaxf(sm_m[2], sm_m[3]));
    float L = 0.f, o = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float f = rebase(sm_m[w], M);
      L += sm_l[w] * f;
      o += sm_acc[w][c] * f;
    }
    p.ws_o[part * D + c] = o;
    if (c == 0) {
      p.ws_ml[part * 2 + 0] = M;
      p.ws_ml[part * 2 + 1] = L;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(D) fa_decode_merge_kernel(const DecodeParams p) {
  const int bh = blockIdx.x;
  const int c = threadIdx.x;
  const float* ml = p.ws_ml + static_cast<size_t>(bh) * p.S * 2;
  const float* po = p.ws_o + static_cast<size_t>(bh) * p.S * D;
  float M = -INFINITY;
  for (int s = 0; s < p.S; ++s)
    if (ml[2 * s + 1] > 0.f) M = fmaxf(M, ml[2 * s]);
  float L = 0.f, o = 0.f;
  for (int s = 0; s < p.S; ++s) {
    const float ls = ml[2 * s + 1];
    if (ls > 0.f) {  // empty splits contribute nothing
      const float f = ex2_approx(ml[2 * s] - M);
      L += ls * f;
      o = fmaf(po[static_cast<size_t>(s) * D + c], f, o);
    }
  }
  const float out = (L > 0.f) ? o / L : 0.f;
  reinterpret_cast<__nv_bfloat16*>(p.o)[static_cast<size_t>(bh) * D + c] = __float2bfloat16_rn(out);
  if (c == 0 && p.lse != nullptr)
    p.lse[bh] = (L > 0.f) ? (M + lg2_approx(L)) * 0.69314718055994530942f : -INFINITY;
}

template <int D>
static cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>(static_cast<long long>(p.S) * p.BH);
  fa_decode_split_kernel<D><<<grid, 128, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  fa_decode_merge_kernel<D><<<p.BH, D, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_decode(int d, const DecodeParams& p, cudaStream_t stream) {
  return d == 64 ? launch_decode_t<64>(p, stream) : launch_decode_t<128>(p, stream);
}

// The merge pass alone, over p.BH rows of p.S partial states each (used by the
// grouped decode, whose rows are the B * H * Nq query tokens).
cudaError_t launch_decode_merge(int d, const DecodeParams& p, cudaStream_t stream) {
  if (d == 64)
    fa_decode_merge_kernel<64><<<p.BH, 64, 0, stream>>>(p);
  else
    fa_decode_merge_kernel<128><<<p.BH, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

// Self-test of the bounded wait: one warp waits on an mbarrier that nothing
// ever arrives on; the wait gives up after limit_ns and records FA_DEV_TIMEOUT.
__global__ void fa_wait_selftest_kernel(uint64_t limit_ns, unsigned int* status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, limit_ns, status, &abort_flag);
  __syncthreads();
}

// Evaluates the FMA-pipe exponential used by the prefill softmax on n inputs.
__global__ void fa_exp2_selftest_kernel(const float* x, float* y, int n) {
  const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
  if (i >= n) return;
  const float x0 = x[i];
  const float x1 = (i + 1 < n) ? x[i + 1] : 0.f;
  float y0, y1;
  f2unpack(exp2_fma2(f2pack(x0, x1)), y0, y1);
  y[i] = y0;
  if (i + 1 < n) y[i + 1] = y1;
}

cudaError_t launch_exp2_selftest(const float* x, float* y, int n, cudaStream_t stream) {
  const int pairs = (n + 1) / 2;
  fa_exp2_selftest_kernel<<<(pairs + 255) / 256, 256, 0, stream>>>(x, y, n);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(uint64_t limit_ns, unsigned int* status, cudaStream_t stream) {
  fa_wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns, status);
  return cudaGetLastError();
}

}  // namespace fa

// ---------------------------------------------------------------------------
// Split-KV decode without any allocation by the caller or the library.
//
// Some callers of this library cannot allocate device memory: a plugin or
// kernel interface that hands over only the input and output buffers, a
// serving loop that must not call cudaMalloc/cudaFree (they can synchronise
// the device) or whose device memory is entirely owned by another allocator.
// For them the decode scratch (the per-split partial (o, m, l) states) lives
// in one file-scope device array, allocated once when the library's device
// code is loaded and held by every GPU that loads it until the process exits.
namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[FA_DECODE_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void* g_scratch_ptr[fa::kMaxDevices] = {nullptr};

// Per-device set-up, done by the first call on each device (with that device
// current): the array's name is only a host-side stand-in, so its device
// address is looked up and cached. Like the rest of the library's per-device
// state, the cached address belongs to the device's primary context as it
// was at that first call; it is not valid after cudaDeviceReset.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= fa::kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" fa_status fa_decode_splitkv_noalloc(const void* q, const void* k_cache, const void* v_cache, void* o,
                                               float* lse, int B, int H, int Nk, int d, float scale,
                                               int num_splits, void* stream) {
  const size_t need = fa_decode_workspace_size(B, H, d, num_splits);
  if (need == 0)  // invalid sizes: let the regular entry point report them
    return fa_decode_splitkv(q, k_cache, v_cache, o, lse, B, H, Nk, d, scale, num_splits, nullptr, 0, stream);
  if (need > FA_DECODE_NOALLOC_SCRATCH_BYTES) {
    fa_set_error_detail("decode needs %zu bytes of scratch; the static scratch holds %zu (use fa_decode_splitkv "
                        "with a caller-provided workspace)",
                        need, static_cast<size_t>(FA_DECODE_NOALLOC_SCRATCH_BYTES));
    return FA_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  const cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) {
    fa_set_error_detail("cudaGetSymbolAddress(decode scratch): %s", cudaGetErrorString(e));
    return FA_ERR_CUDA;
  }
  // every partial is written by the split kernel before the merge reads it,
  // so the shared scratch needs no clearing between calls
  return fa_decode_splitkv(q, k_cache, v_cache, o, lse, B, H, Nk, d, scale, num_splits, scratch,
                           FA_DECODE_NOALLOC_SCRATCH_BYTES, stream);
}
