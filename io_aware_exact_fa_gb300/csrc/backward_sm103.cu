// Exact-attention backward pass for sm_103a: dQ, dK, dV of a loss through
// O = softmax(scale * Q K^T + causal mask) V, recomputing the probability
// tiles from the forward's per-row log-sum-exp instead of storing P ("Flash
// Attention Optimization", section "Sizing a tile, and why the backward pass
// recomputes instead of storing"; "Explain FlashAttention ...", section
// "Exact attention, finite precision and backward"). With
// P_ij = exp(scale q_i.k_j - lse_i) and D_i = sum_c dO_ic O_ic:
//   dV = P^T dO,   dS = P * (dO V^T - D),   dQ = scale dS K,   dK = scale dS^T Q.
//
// Three launches:
//   fa_bwd_prep_kernel      D and lse (log2 units) per query row; zero the
//                           fp32 dQ accumulator.
//   fa_bwd_kernel<D>        one CTA per 128-key tile of one (b, h): K and V stay
//                           in shared memory while the 128-row Q / dO tiles
//                           the causal mask leaves visible stream past; dK and
//                           dV accumulate in TMEM; each Q tile's dQ
//                           contribution is added to the accumulator with
//                           vector atomics.
//   fa_bwd_finish_kernel    dQ = bf16(scale * accumulator).
//
// fa_bwd_kernel, 512 threads:
//   warp 0       TMA producer: K and V once, then Q_i / dO_i into two stages.
//   warp 1       TMEM allocator and MMA issuer.
//   warps 4-11   "softmax-grad": a thread owns one key row (TMEM lane) and one
//                half of the 128 query columns of S^T = K Q_i^T and
//                dP^T = V dO_i^T, forms P^T and dS^T, writes P^T (bf16) into
//                the S^T columns and dS^T (bf16) into shared memory; at the
//                end one half writes dV, the other dK.
//   warps 12-15  dQ drain: a thread owns one query row of dQ_i = dS K.
// Per step the MMAs run dQ_i, dV_i, S^T_{i+1}, dP^T_{i+1}, dK_i, so the next
// step's softmax-grad overlaps dK_i and the drain overlaps the rest.
// TMEM columns: S^T [0,128) (P^T bf16 in [0,32) and [64,96)), dP^T
// [128,256) (later dQ_i), dV [256,256+D), dK [256+D,256+2D).
#include <cuda_bf16.h>

#include "fa_ptx.cuh"

namespace fa {

#ifndef FA_BWD_ELECT_ISSUE
#define FA_BWD_ELECT_ISSUE 1
#endif
#ifndef FA_BWD_EARLY_S
#define FA_BWD_EARLY_S 1
#endif

namespace {

constexpr int BWD_THREADS = 512;
constexpr int BWD_TMA_WARP = 0;
constexpr int BWD_MMA_WARP = 1;
constexpr int BWD_SG_WARP0 = 4;  // warps 4-11
constexpr int BWD_SG_THREADS = 256;
constexpr int BWD_DQ_WARP0 = 12;  // warps 12-15

template <int D>
struct BwdCfg {
  static_assert(D == 64 || D == 128, "head dim 64 or 128");
  static constexpr int TILE_BYTES = 128 * D * 2;  // one K, V, Q or dO tile (128 rows x D bf16)
  static constexpr int BOX_BYTES = 128 * 128;     // one TMA box: 128 rows x 64 bf16
  static constexpr int NBOX = D / 64;
  static constexpr int DS_BYTES = 128 * 128 * 2;  // dS^T tile: 128 keys x 128 queries bf16
  // At d = 64, P^T and dQ_i get TMEM columns of their own and dS^T two shared
  // buffers, so the next step's S^T and dP^T need not wait for this step's
  // products; at d = 128 neither fits.
  static constexpr bool SEP = (D == 64);
  static constexpr int NDS = SEP ? 2 : 1;
  // The MMA warp walks the issue loop converged, and the lane elect.sync
  // picks issues every MMA and commit: one thread then keeps the tensor pipe
  // fed with the N = 64 products, which a loop run by lane 0 alone issues at
  // about half the pipe's rate. (Otherwise, at d = 64, lane 0 walks the loop
  // alone: its waits need no warp vote.)
  static constexpr bool ELECT_ISSUE = FA_BWD_ELECT_ISSUE;
  static constexpr bool SOLO_ISSUE = !ELECT_ISSUE && (D == 64);
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + TILE_BYTES;
  static constexpr int Q_OFF = V_OFF + TILE_BYTES;                 // 2 stages of (Q, dO)
  static constexpr int DS_OFF = Q_OFF + 2 * 2 * TILE_BYTES;        // NDS dS^T buffers
  // At d = 64 the next step's S^T and dP^T are issued as soon as the
  // softmax-grad has loaded this step's (EARLY_S), so two steps' statistics
  // can be live at once: they alternate between two buffers.
  static constexpr bool EARLY_S = SEP && FA_BWD_EARLY_S;
  static constexpr int NSTAT = EARLY_S ? 2 : 1;
  static constexpr int STAT_OFF = DS_OFF + NDS * DS_BYTES;         // [NSTAT] of lse2[128], Dv[128]
  static constexpr int BAR_OFF = STAT_OFF + NSTAT * 2 * 128 * 4;
  static constexpr int NBAR = 16;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int SMEM = MISC_OFF + 16 + 1024;
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  static constexpr uint32_t ST_COL = 0, DPT_COL = 128, DV_COL = 256, DK_COL = 256 + D;
  // P^T (bf16, 64 columns): inside S^T at d = 128 (half h at 64 h), its own columns at d = 64 (half h at 32 h);
  // dQ_i: in the dP^T columns at d = 128, its own columns at d = 64
  static constexpr uint32_t PT_COL = SEP ? 384 : ST_COL, PT_HALF = SEP ? 32 : 64;
  static constexpr uint32_t DQ_COL = SEP ? 448 : DPT_COL;
  static constexpr uint32_t IDESC_T = idesc_bf16_f32(128, 128, false);        // K-major A and B
  static constexpr uint32_t IDESC_B_MN = idesc_bf16_f32(128, D, true);        // B MN-major
  static constexpr uint32_t IDESC_AB_MN = idesc_bf16_f32(128, D, true, true); // A and B MN-major
};

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(a, parity)) return;
    if ((i & 31u) == 31u && globaltimer_ns() - t0 > limit_ns) return;
  }
}

// First 128-row Q tile a key tile starting at key k0 needs under the causal
// mask: query i sees key j iff j <= i + delta.
__device__ __forceinline__ int first_qtile(int k0, int delta, bool causal) {
  if (!causal) return 0;
  const int first_q = k0 - delta;  // the smallest query that sees key k0
  return first_q <= 0 ? 0 : first_q / 128;
}

}  // namespace

// ------------------------------------------------------------------ prepare
// One thread per query row of the 128-row-padded Q tiles: the row's entries of
// the tiled fp32 dQ accumulator set to 0 and, for a row below Nq,
// D_i = sum_c dO_ic O_ic (fp32) and lse2_i = lse_i * log2(e) (+inf for an
// empty row, so its recomputed weights are 0).
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_prep_kernel(const __nv_bfloat16* __restrict__ o,
                                                          const __nv_bfloat16* __restrict__ dout,
                                                          const float* __restrict__ lse, float* __restrict__ dq_acc,
                                                          float* __restrict__ lse2, float* __restrict__ drow,
                                                          long long bh_count, int Nq) {
  const long long nqt = (Nq + 127) / 128;
  const long long r = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (r >= bh_count * nqt * 128) return;
  const long long bh = r / (nqt * 128);
  const int qq = static_cast<int>(r - bh * nqt * 128);
  float4* acc = reinterpret_cast<float4*>(dq_acc) + ((bh * nqt + (qq >> 7)) * (D / 4)) * 128 + (qq & 127);
#pragma unroll
  for (int c = 0; c < D / 4; ++c) acc[c * 128] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (qq >= Nq) return;
  const long long gr = bh * Nq + qq;
  const uint4* po = reinterpret_cast<const uint4*>(o + gr * D);
  const uint4* pd = reinterpret_cast<const uint4*>(dout + gr * D);
  float a = 0.f;
#pragma unroll
  for (int c = 0; c < D / 8; ++c) {
    const uint4 x = __ldg(po + c), y = __ldg(pd + c);
    const uint32_t wa[4] = {x.x, x.y, x.z, x.w}, wb[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wa[e]));
      const float2 fb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wb[e]));
      a = fmaf(fa.x, fb.x, a);
      a = fmaf(fa.y, fb.y, a);
    }
  }
  drow[gr] = a;
  const float l = lse[gr];
  lse2[gr] = (l == -INFINITY) ? INFINITY : l * 1.4426950408889634f;
}

// ------------------------------------------------------------------- finish
// One thread per 8 columns of a dQ row: dQ = bf16(scale * accumulator), read
// from the tiled accumulator layout.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_finish_kernel(const float* __restrict__ dq_acc,
                                                            __nv_bfloat16* __restrict__ dq, float scale,
                                                            long long n8, int Nq) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n8) return;
  const long long row = i / (D / 8);
  const int g = static_cast<int>(i - row * (D / 8));
  const long long bh = row / Nq;
  const int q = static_cast<int>(row - bh * Nq);
  const long long nqt = (Nq + 127) / 128;
  const float4* a4 =
      reinterpret_cast<const float4*>(dq_acc) + ((bh * nqt + (q >> 7)) * (D / 4) + 2 * g) * 128 + (q & 127);
  const float4 a = a4[0], b = a4[128];
  uint4 w;
  w.x = pack_bf16x2(a.x * scale, a.y * scale);
  w.y = pack_bf16x2(a.z * scale, a.w * scale);
  w.z = pack_bf16x2(b.x * scale, b.y * scale);
  w.w = pack_bf16x2(b.z * scale, b.w * scale);
  reinterpret_cast<uint4*>(dq)[i] = w;
}

// ----------------------------------------------------- softmax-grad half tile
// One thread, one key row, one half (64 query columns, chunks 2h and 2h + 1) of
// a 128 x 128 step: P^T = exp2(S^T * scale * log2(e) - lse2) and
// dS^T = P^T * (dP^T - D). P^T (bf16) goes to the P^T columns of half h,
// dS^T (bf16) into the 128-byte-swizzled shared tile (box h). nlse2 and ndrow
// hold -lse2 and -D per query column. With MASK, columns below c_lo are
// masked. One exponential pair in four runs on the FMA pipe (exp2_fma2) to
// offload the MUFU unit. before_math() is called once, after the first TMEM
// loads are issued and before the statistics are read; before_pstore() once,
// before the first P^T store; before_store() once, before the first
// shared-memory store. If any returns false the step stops there. A non-null
// loaded_bar is arrived on once this thread has loaded all its S^T and dP^T
// columns.
template <int D, bool MASK, typename F, typename G, typename E>
__device__ __forceinline__ bool sg_half(uint32_t tST, uint32_t tDPT, uint32_t tPT, uint32_t ds_row, int row, int h,
                                        int c_lo, const float* nlse2, const float* ndrow, float sl2, G&& before_math,
                                        E&& before_pstore, F&& before_store, uint64_t* loaded_bar) {
  using C = BwdCfg<D>;
  const uint64_t sl2x2 = f2pack(sl2, sl2);
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    const int ch = 2 * h + cc;
    uint32_t sv[32], dp[32];
    tmem_ld32(tST + ch * 32, sv);
    tmem_ld32(tDPT + ch * 32, dp);
    if (cc == 0 && !before_math()) {
      tmem_ld_wait32(sv);
      reg_fence32(dp);
      return false;
    }
    tmem_ld_wait32(sv);
    reg_fence32(dp);
    if (cc == 1 && loaded_bar != nullptr) {
      // this thread's S^T and dP^T columns are in registers: the next step's
      // products may overwrite them
      tc_fence_before();
      mbar_arrive(loaded_bar);
    }
    uint32_t pk[16], dk[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int c = ch * 32 + 4 * j;
      const float4 nl = *reinterpret_cast<const float4*>(nlse2 + c);
      const float4 nd = *reinterpret_cast<const float4*>(ndrow + c);
      const uint64_t a01 = ffma2(f2pack(u2f(sv[4 * j]), u2f(sv[4 * j + 1])), sl2x2, f2pack(nl.x, nl.y));
      const uint64_t a23 = ffma2(f2pack(u2f(sv[4 * j + 2]), u2f(sv[4 * j + 3])), sl2x2, f2pack(nl.z, nl.w));
      float x0, x1, p0, p1, p2, p3;
      f2unpack(a01, x0, x1);
      p0 = ex2_approx(x0);
      p1 = ex2_approx(x1);
      if (j & 1) {
        f2unpack(exp2_fma2(a23), p2, p3);
      } else {
        float x2, x3;
        f2unpack(a23, x2, x3);
        p2 = ex2_approx(x2);
        p3 = ex2_approx(x3);
      }
      if (MASK) {
        p0 = c >= c_lo ? p0 : 0.f;
        p1 = c + 1 >= c_lo ? p1 : 0.f;
        p2 = c + 2 >= c_lo ? p2 : 0.f;
        p3 = c + 3 >= c_lo ? p3 : 0.f;
      }
      const uint64_t g01 = fadd2(f2pack(u2f(dp[4 * j]), u2f(dp[4 * j + 1])), f2pack(nd.x, nd.y));
      const uint64_t g23 = fadd2(f2pack(u2f(dp[4 * j + 2]), u2f(dp[4 * j + 3])), f2pack(nd.z, nd.w));
      float d0, d1, d2, d3;
      f2unpack(fmul2(f2pack(p0, p1), g01), d0, d1);
      f2unpack(fmul2(f2pack(p2, p3), g23), d2, d3);
      pk[2 * j] = pack_bf16x2(p0, p1);
      pk[2 * j + 1] = pack_bf16x2(p2, p3);
      dk[2 * j] = pack_bf16x2(d0, d1);
      dk[2 * j + 1] = pack_bf16x2(d2, d3);
    }
    // P^T: half h keeps its 64 queries (32 bf16x2 columns) at tPT + PT_HALF h;
    // at d = 128 that is inside the S^T columns this thread already read
    if (cc == 0 && !before_pstore()) return false;
    tmem_st16(tPT + h * C::PT_HALF + cc * 16, pk);
    if (cc == 0 && !before_store()) return false;
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      // 16-byte chunk (ch % 2) * 4 + v of the row's 128-byte line in box h
      const uint32_t a = ds_row + static_cast<uint32_t>(h * C::BOX_BYTES) +
                         (static_cast<uint32_t>(((cc * 4 + v) ^ (row & 7))) << 4);
      st_shared_v4(a, dk[4 * v], dk[4 * v + 1], dk[4 * v + 2], dk[4 * v + 3]);
    }
  }
  return true;
}

// --------------------------------------------------------------------- main
template <int D>
__global__ void __launch_bounds__(BWD_THREADS, 1)
    fa_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                  const BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = smem + C::K_OFF;
  uint8_t* sV = smem + C::V_OFF;
  uint8_t* sQ0 = smem + C::Q_OFF;  // stage s: Q at Q_OFF + s*2*TILE, dO right after
  uint8_t* sDS = smem + C::DS_OFF;
  // -lse2 and -D per query of a step (buffer it % NSTAT)
  auto s_nlse2 = [&](int it) { return reinterpret_cast<float*>(smem + C::STAT_OFF) + (it % C::NSTAT) * 256; };
  auto s_ndrow = [&](int it) { return s_nlse2(it) + 128; };
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* kv_full = bars + 0;
  uint64_t* q_full = bars + 1;     // [2]
  uint64_t* q_empty = bars + 3;    // [2]
  uint64_t* s_full = bars + 5;     // S^T and dP^T of a step computed
  uint64_t* p_full = bars + 6;     // P^T stored in TMEM and dS^T in shared memory (all softmax-grad threads)
  uint64_t* dv_done = bars + 7;    // the step's dV MMA (reading P^T from the S^T columns) completed
  uint64_t* step_done = bars + 8;  // the step's last MMA (dK) completed: dS^T may be rewritten
  uint64_t* dq_full = bars + 9;    // dQ_i in the dP^T columns
  uint64_t* dq_free = bars + 10;   // dQ_i read out
  uint64_t* acc_done = bars + 11;  // every MMA completed: dK, dV final
  uint64_t* stat_full = bars + 12; // the step's lse / D staged in shared memory
  uint64_t* st_free = bars + 13;   // S^T and dP^T of a step loaded by every softmax-grad thread (EARLY_S)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t lim = p.wait_limit_ns;
  const int nkt = (p.Nk + 127) / 128;
  const int bh = static_cast<int>(blockIdx.x) / nkt;
  const int kt = static_cast<int>(blockIdx.x) % nkt;
  const int k0 = kt * 128;
  const int delta = p.Nk - p.Nq;
  const int nqt = (p.Nq + 127) / 128;
  const int qt0 = first_qtile(k0, delta, p.causal != 0);
  const int n_it = max(0, nqt - qt0);  // Q tiles this key tile visits

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(q_full + s, 1);
      mbar_init(q_empty + s, 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_full, BWD_SG_THREADS);
    mbar_init(dv_done, 1);
    mbar_init(step_done, 1);
    mbar_init(dq_full, 1);
    mbar_init(dq_free, 128);
    mbar_init(acc_done, 1);
    mbar_init(stat_full, BWD_SG_THREADS);
    mbar_init(st_free, BWD_SG_THREADS);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == BWD_MMA_WARP) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == BWD_TMA_WARP) {
    // ---------------------------------------------------------- TMA producer
    const bool leader = lane == 0;
    bool ok = true;
    int issued = 0;
    if (leader) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
      mbar_arrive_expect_tx(kv_full, 2 * C::TILE_BYTES);
      for (int b = 0; b < C::NBOX; ++b) {
        tma_load_3d(sK + b * C::BOX_BYTES, &tmK, kv_full, 64 * b, k0, bh);
        tma_load_3d(sV + b * C::BOX_BYTES, &tmV, kv_full, 64 * b, k0, bh);
      }
    }
    for (int it = 0; ok && it < n_it; ++it) {
      const int s = it & 1;
      if (it >= 2) {
        ok = mbar_wait(q_empty + s, ((it - 2) >> 1) & 1, lim, p.status, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
      if (leader) {
        uint8_t* dq_ = sQ0 + s * 2 * C::TILE_BYTES;
        const int q0 = (qt0 + it) * 128;
        mbar_arrive_expect_tx(q_full + s, 2 * C::TILE_BYTES);
        for (int b = 0; b < C::NBOX; ++b) {
          tma_load_3d(dq_ + b * C::BOX_BYTES, &tmQ, q_full + s, 64 * b, q0, bh);
          tma_load_3d(dq_ + C::TILE_BYTES + b * C::BOX_BYTES, &tmDO, q_full + s, 64 * b, q0, bh);
        }
      }
      ++issued;
    }
    if (leader) {
      // every copy issued lands before the CTA exits
      mbar_drain(kv_full, 0, lim);
      for (int n = max(0, issued - 2); n < issued; ++n) mbar_drain(q_full + (n & 1), (n >> 1) & 1, lim);
    }
    __syncwarp();
  } else if (warp == BWD_MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    // Per step i at d = 128: dQ_i, dV_i, then (for step i + 1) S^T and dP^T,
    // then dK_i, so the next step's softmax-grad starts while dK_i runs. At
    // d = 64 (separate P^T and dQ columns, two dS^T buffers): the next step's
    // S^T and dP^T first, then dV_i, dQ_i and dK_i, so the next softmax-grad
    // overlaps all three.
    const bool leader = lane == 0;
    // the thread that issues the MMAs and commits
    auto issuer = [&]() -> bool {
      if constexpr (C::ELECT_ISSUE) return elect_one();
      else return leader;
    };
    bool ok = true;
    auto wait_bar = [&](uint64_t* bar, uint32_t parity) {
      ok = mbar_wait(bar, parity, lim, p.status, abort_flag);
      if (!C::SOLO_ISSUE) ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
      return ok;
    };
    constexpr uint32_t DHI = sdesc_sw128_hi(1024);
    const uint32_t k_lo = sdesc_sw128_lo(smem_u32(sK), 16), kmn_lo = sdesc_sw128_lo(smem_u32(sK), C::BOX_BYTES);
    const uint32_t v_lo = sdesc_sw128_lo(smem_u32(sV), 16);
    const uint32_t tST = tmem + C::ST_COL, tDPT = tmem + C::DPT_COL, tDV = tmem + C::DV_COL,
                   tDK = tmem + C::DK_COL, tPT = tmem + C::PT_COL, tDQ = tmem + C::DQ_COL;
    auto ds_base = [&](int it) { return smem_u32(sDS) + (C::NDS > 1 ? (it & 1) * C::DS_BYTES : 0); };
    // K-major K-step kk of a tile: (kk / 4) boxes plus (kk % 4) x 32 bytes in;
    // MN-major K-step kk: 16 rows = 2048 bytes in (64-column boxes LBO apart)
    auto kmaj = [](int kk) { return static_cast<uint32_t>(((kk >> 2) * C::BOX_BYTES + (kk & 3) * 32) >> 4); };
    auto mnmaj = [](int kk) { return static_cast<uint32_t>((kk * 2048) >> 4); };
    auto stage = [&](int it) { return smem_u32(sQ0) + (it & 1) * 2 * C::TILE_BYTES; };
    // S^T = K Q_i^T and dP^T = V dO_i^T of step it (both operands K-major)
    auto issue_s_dp = [&](int it) {
      const uint32_t qb = stage(it);
      const uint32_t q_lo = sdesc_sw128_lo(qb, 16), do_lo = sdesc_sw128_lo(qb + C::TILE_BYTES, 16);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        if (issuer()) mma_ss_w(tST, k_lo + kmaj(kk), DHI, q_lo + kmaj(kk), DHI, C::IDESC_T, kk > 0 ? 1u : 0u);
      // at d = 128, dP^T (the dP^T columns) only after the previous dQ_i was read out
      if (!C::SEP && it > 0 && !wait_bar(dq_free, (it - 1) & 1)) return false;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        if (issuer()) mma_ss_w(tDPT, v_lo + kmaj(kk), DHI, do_lo + kmaj(kk), DHI, C::IDESC_T, kk > 0 ? 1u : 0u);
      if (issuer()) mma_commit(s_full);
      return true;
    };
    const bool walks = !C::SOLO_ISSUE || leader;  // this lane runs the issue loop
    if (n_it > 0 && walks) {
      if (wait_bar(kv_full, 0) && wait_bar(q_full, 0)) issue_s_dp(0);
    }
    for (int it = 0; ok && walks && it < n_it; ++it) {
      const uint32_t qb = stage(it);
      const uint32_t qmn_lo = sdesc_sw128_lo(qb, C::BOX_BYTES), domn_lo = sdesc_sw128_lo(qb + C::TILE_BYTES, C::BOX_BYTES);
      const uint32_t ds_lo = sdesc_sw128_lo(ds_base(it), 16), dsmn_lo = sdesc_sw128_lo(ds_base(it), C::BOX_BYTES);
      // dQ_i = dS K (A = dS, the MN-major view of dS^T; B = K MN-major)
      auto issue_dq = [&]() {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          if (issuer())
            mma_ss_w(tDQ, dsmn_lo + mnmaj(kk), DHI, kmn_lo + mnmaj(kk), DHI, C::IDESC_AB_MN, kk > 0 ? 1u : 0u);
        if (issuer()) mma_commit(dq_full);
      };
      // dV += P^T dO_i (A = P^T from TMEM: queries 16 kk.. of half kk / 4 at
      // tPT + PT_HALF (kk / 4) + 8 (kk % 4); B = dO_i MN-major)
      auto issue_dv = [&]() {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          if (issuer())
            mma_ts_w(tDV, tPT + (kk >> 2) * C::PT_HALF + (kk & 3) * 8, domn_lo + mnmaj(kk), DHI, C::IDESC_B_MN,
                     (it > 0 || kk > 0) ? 1u : 0u);
        if (issuer()) mma_commit(dv_done);
      };
      // dK += dS^T Q_i (A = dS^T K-major, B = Q_i MN-major)
      auto issue_dk = [&]() {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          if (issuer())
            mma_ss_w(tDK, ds_lo + kmaj(kk), DHI, qmn_lo + mnmaj(kk), DHI, C::IDESC_B_MN, (it > 0 || kk > 0) ? 1u : 0u);
        if (issuer()) {
          mma_commit(step_done);
          mma_commit(q_empty + (it & 1));
        }
      };
      if (!wait_bar(C::EARLY_S ? st_free : p_full, it & 1)) break;
      if constexpr (C::SEP) {
        // the softmax-grad has read S^T_i and dP^T_i: the next step's products may overwrite them
        // (with EARLY_S as soon as every thread has loaded them, while the softmax-grad still runs)
        if (it + 1 < n_it) {
          if (!wait_bar(q_full + ((it + 1) & 1), ((it + 1) >> 1) & 1)) break;
          if (!issue_s_dp(it + 1)) break;
        }
        if (C::EARLY_S && !wait_bar(p_full, it & 1)) break;
        issue_dv();
        // dQ_i into the dQ columns once the drain has read dQ_{i-1}
        if (it > 0 && !wait_bar(dq_free, (it - 1) & 1)) break;
        issue_dq();
        issue_dk();
      } else {
        issue_dq();  // into the dP^T columns, so its drain overlaps dV and dK
        issue_dv();
        if (it + 1 < n_it) {
          // the next S^T overwrites P^T_i: only after dV_i read it
          if (!wait_bar(q_full + ((it + 1) & 1), ((it + 1) >> 1) & 1)) break;
          if (!wait_bar(dv_done, it & 1)) break;
          if (!issue_s_dp(it + 1)) break;
        }
        issue_dk();
      }
    }
    if (!C::SOLO_ISSUE) __syncwarp();
    if (n_it > 0) {
      if (issuer()) mma_commit(acc_done);
    } else if (leader) {
      mbar_arrive(acc_done);
    }
    if (leader) mbar_drain(acc_done, 0, lim);  // every MMA completed before TMEM is released
    __syncwarp();
  } else if (warp >= BWD_SG_WARP0 && warp < BWD_DQ_WARP0) {
    // ---------------------------------------------------------- softmax-grad
    // warp w: key rows 32 * (w % 4) .. + 31 (its TMEM lane quarter), query
    // columns 64 * h .. + 63 with h = (w - 4) / 4
    const int wq = warp & 3;
    const int h = (warp - BWD_SG_WARP0) >> 2;
    const int row = wq * 32 + lane;  // key row within the tile
    const int kabs = k0 + row;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tST = tmem + lane_base + C::ST_COL, tDPT = tmem + lane_base + C::DPT_COL;
    bool ok = true;
    const uint32_t tPT = tmem + lane_base + C::PT_COL;
    // this thread's key row in dS^T buffer b
    auto ds_row = [&](int it) {
      return smem_u32(sDS) + (C::NDS > 1 ? (it & 1) * C::DS_BYTES : 0) + static_cast<uint32_t>(row) * 128u;
    };
    // one entry of the per-row statistics (h = 0: lse2, h = 1: D) of query
    // row `row` of the Q tile, loaded one step ahead
    const float* stat_src = h ? p.drow : p.lse2;
    auto stat_dst = [&](int it) { return (h ? s_ndrow(it) : s_nlse2(it)) + row; };
    float nx = 0.f;
    auto fetch = [&](int it) {
      const int qi = (qt0 + it) * 128 + row;
      nx = h ? 0.f : INFINITY;
      if (it < n_it && qi < p.Nq) nx = stat_src[static_cast<size_t>(bh) * p.Nq + qi];
    };
    fetch(0);
    for (int it = 0; ok && it < n_it; ++it) {
      const int q0 = (qt0 + it) * 128;
      ok = mbar_wait(s_full, it & 1, lim, p.status, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      // stage this Q tile's statistics, negated; every thread has finished
      // with the buffer's previous contents (s_full of this step needed all of
      // p_full of the previous one, or with EARLY_S and two buffers st_free
      // of the previous step, which every thread reaches after step it - 2)
      *stat_dst(it) = -nx;
      fetch(it + 1);
      mbar_arrive(stat_full);  // release: this thread's value is visible to the waiters
      // the statistics are waited for once the first TMEM loads are in flight
      auto before_math = [&]() {
        const bool w = mbar_wait(stat_full, it & 1, lim, p.status, abort_flag);
        return __all_sync(0xffffffffu, w) != 0;
      };
      // dS^T in shared memory is rewritten only after the previous step's dK
      // (its last reader) completed
      // At d = 128 dS^T is rewritten only after the previous step's dK (its
      // last reader) completed. At d = 64 this step's buffer was last read by
      // step i-2's dQ and dK, which completed before S^T_i (their commit order
      // covers them), so no wait.
      auto before_store = [&]() {
        if (C::SEP || it == 0) return true;
        bool w = mbar_wait(step_done, (it - 1) & 1, lim, p.status, abort_flag);
        return __all_sync(0xffffffffu, w) != 0;
      };
      // At d = 64 P^T has columns of its own, which dV_{i-1} reads: wait for it.
      // At d = 128 P^T goes over S^T_i, which was written after dV_{i-1} completed.
      auto before_pstore = [&]() {
        if (!C::SEP || it == 0) return true;
        bool w = mbar_wait(dv_done, (it - 1) & 1, lim, p.status, abort_flag);
        w = __all_sync(0xffffffffu, w) != 0;
        tc_fence_after();
        return w;
      };
      // Only a Q tile that crosses the causal diagonal (query q sees this key
      // iff q >= kabs - delta) or a key tile past Nk needs a per-element test.
      // Key rows >= Nk hold zero K and V (TMA fill) but exp2(0 - lse2) may
      // overflow there, so they are masked whole; query rows >= Nq carry
      // lse = +inf, so their weights are 0 without a test.
      if ((p.causal && k0 + 127 - delta > q0) || k0 + 128 > p.Nk) {
        const int c_lo = kabs >= p.Nk ? INT_MAX : (p.causal ? kabs - delta - q0 : INT_MIN);
        ok = sg_half<D, true>(tST, tDPT, tPT, ds_row(it), row, h, c_lo, s_nlse2(it), s_ndrow(it), p.scale_log2,
                              before_math, before_pstore, before_store, C::EARLY_S ? st_free : nullptr);
      } else {
        ok = sg_half<D, false>(tST, tDPT, tPT, ds_row(it), row, h, 0, s_nlse2(it), s_ndrow(it), p.scale_log2,
                               before_math, before_pstore, before_store, C::EARLY_S ? st_free : nullptr);
      }
      if (!ok) break;
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    // ---- epilogue: h = 0 writes dV = acc, h = 1 writes dK = scale * acc (bf16), rows below Nk
    if (ok) {
      ok = mbar_wait(acc_done, 0, lim, p.status, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
    }
    // tcgen05.ld is warp-collective: every lane loads, only rows below Nk store
    if (ok) {
      const bool row_ok = kabs < p.Nk;
      const size_t kr = static_cast<size_t>(bh) * p.Nk + (row_ok ? kabs : 0);
      const uint32_t src = tmem + lane_base + (h ? C::DK_COL : C::DV_COL);
      const float f = h ? p.scale : 1.f;
      __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(h ? p.dk : p.dv) + kr * D;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t a[32];
        if (n_it > 0) {
          tmem_ld32(src + ch * 32, a);
          tmem_ld_wait32(a);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) a[i] = 0u;
        }
        uint4* d4 = reinterpret_cast<uint4*>(dst + ch * 32);
#pragma unroll
        for (int v = 0; v < 4; ++v)
          if (row_ok)
            d4[v] = make_uint4(pack_bf16x2(u2f(a[8 * v]) * f, u2f(a[8 * v + 1]) * f),
                               pack_bf16x2(u2f(a[8 * v + 2]) * f, u2f(a[8 * v + 3]) * f),
                               pack_bf16x2(u2f(a[8 * v + 4]) * f, u2f(a[8 * v + 5]) * f),
                               pack_bf16x2(u2f(a[8 * v + 6]) * f, u2f(a[8 * v + 7]) * f));
      }
    }
  } else if (warp >= BWD_DQ_WARP0) {
    // -------------------------------------------------------------- dQ drain
    const int wq = warp & 3;
    const int row = wq * 32 + lane;  // query row within the Q tile
    const uint32_t src = tmem + (static_cast<uint32_t>(wq * 32) << 16) + C::DQ_COL;
    bool ok = true;
    for (int it = 0; ok && it < n_it; ++it) {
      ok = mbar_wait(dq_full, it & 1, lim, p.status, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      // Tiled accumulator: one warp's 32 rows of a 4-column chunk are 512
      // contiguous bytes. Rows past Nq add zeros to the padding.
      float* dst = p.dq_acc + ((static_cast<size_t>(bh) * nqt + qt0 + it) * (D / 4) * 128 + row) * 4;
#pragma unroll
      for (int hh = 0; hh < D / 32; ++hh) {
        uint32_t a[32];
        tmem_ld32(src + hh * 32, a);
        tmem_ld_wait32(a);
        if (hh == D / 32 - 1) {
          // the dP^T columns may take the next step's dP^T once the loads completed
          tc_fence_before();
          mbar_arrive(dq_free);
        }
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4)
          red_add_v4_f32(dst + (hh * 8 + c4) * 512, u2f(a[4 * c4]), u2f(a[4 * c4 + 1]), u2f(a[4 * c4 + 2]),
                         u2f(a[4 * c4 + 3]));
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == BWD_MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
static cudaError_t launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const CUtensorMap& tdo, const BwdParams& p, const void* o, const void* dout,
                                const float* lse, void* dq, cudaStream_t stream) {
  const long long bhc = static_cast<long long>(p.B) * p.H;
  const long long rows = bhc * p.Nq;
  const long long rows_pad = bhc * ((p.Nq + 127) / 128) * 128;
  fa_bwd_prep_kernel<D><<<static_cast<unsigned>((rows_pad + 255) / 256), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), lse, p.dq_acc, p.lse2,
      p.drow, bhc, p.Nq);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const long long ctas = static_cast<long long>(p.B) * p.H * ((p.Nk + 127) / 128);
  fa_bwd_kernel<D><<<static_cast<unsigned>(ctas), BWD_THREADS, BwdCfg<D>::SMEM, stream>>>(tq, tk, tv, tdo, p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const long long n8 = rows * D / 8;
  fa_bwd_finish_kernel<D><<<static_cast<unsigned>((n8 + 255) / 256), 256, 0, stream>>>(
      p.dq_acc, static_cast<__nv_bfloat16*>(dq), p.scale, n8, p.Nq);
  return cudaGetLastError();
}

cudaError_t bwd_set_attributes(int d) {
  if (d == 64)
    return cudaFuncSetAttribute(fa_bwd_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdCfg<64>::SMEM);
  return cudaFuncSetAttribute(fa_bwd_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdCfg<128>::SMEM);
}

cudaError_t launch_bwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const BwdParams& p, const void* o, const void* dout, const float* lse,
                       void* dq, cudaStream_t stream) {
  return d == 64 ? launch_bwd_t<64>(tq, tk, tv, tdo, p, o, dout, lse, dq, stream)
                 : launch_bwd_t<128>(tq, tk, tv, tdo, p, o, dout, lse, dq, stream);
}

}  // namespace fa
