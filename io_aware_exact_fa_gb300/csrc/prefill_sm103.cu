// Fused exact-attention forward pass (prefill) for sm_103a.
//
// What it computes: O = softmax(scale * Q K^T + mask) V and the per-row
// log-sum-exp, without ever writing the score matrix to HBM ("Flash Attention
// Optimization", sections "Attention is not slow because of arithmetic" and
// "The fix: tile the computation, never materialize the full matrix").
// The row recurrence is the new-max form with one rescale factor
// alpha = exp(m_old - m_new) per tile and a single division at the end
// ("Explain FlashAttention. Why is it called IO-aware ...", section "Keep only
// the state needed for the final weighted average"); Q tiles stay resident
// and K/V tiles stream past them (the loop order the FlashAttention-2 section
// of "FlashAttention: Attention Is Limited by Memory, Not Math" describes as
// parallel over sequence length).
//
// One CTA per SM handles a work unit of two 128-row Q tiles of one (b, h).
// 384 threads = 3 warpgroups; after set-up the softmax warpgroups take more
// registers and the producer warpgroup fewer (setmaxnreg).
//   warp 8      TMA producer: Q once, then K_j / V_j into a ring of slots.
//   warps 10-11 idle after set-up.
//   warp 9      TMEM allocator and MMA issuer (one thread):
//               S_t = Q_t K_j^T into TMEM, later O_t += P_t V_j.
//   warps 0-3   softmax for Q tile 0, warps 4-7 for Q tile 1: each thread
//               owns one query row (TMEM lane), reads its 128 scores with
//               tcgen05.ld, applies the mask from absolute positions, folds
//               the tile into (m, l), writes P (bf16) over S in TMEM and
//               rescales its O row when the running max rose; at the end it
//               divides by l and writes O (bf16) and lse (fp32).
// TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256,256+D), O_1 [256+D,256+2D).
// The two Q tiles ping-pong: while one softmax warpgroup works, the tensor
// core runs the other tile's MMAs.
#include <cuda_bf16.h>

#include "fa_ptx.cuh"

namespace fa {

template <int D>
struct PrefillCfg {
  static_assert(D == 64 || D == 128, "head dim 64 or 128");
  static constexpr int TILE_BYTES = BLOCK_N * D * 2;  // one Q, K or V tile (128 rows x D bf16)
  static constexpr int BOX_BYTES = 128 * 128;         // one TMA box: 128 rows x 64 bf16
  static constexpr int NBOX = D / 64;
  static constexpr int NSLOT = (D == 128) ? 4 : 8;    // K/V ring slots (K and V alternate)
  static constexpr int Q_OFF = 0;
  static constexpr int KV_OFF = Q_TILES * TILE_BYTES;
  static constexpr int BAR_OFF = KV_OFF + NSLOT * TILE_BYTES;
  static constexpr int NBAR = 1 + 2 * NSLOT + 3 * Q_TILES + 1;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int SMEM = MISC_OFF + 16 + 1024;   // + slack to align the base to 1024
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t IDESC_S = idesc_bf16_f32(128, 128, false);  // Q, K both K-major
  static constexpr uint32_t IDESC_O = idesc_bf16_f32(128, D, true);     // V is MN-major
};

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

// Drain wait used only on the error path: ignores the abort flag.
__device__ __forceinline__ void mbar_wait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(a, parity)) return;
    if ((i & 31u) == 31u && globaltimer_ns() - t0 > limit_ns) return;
  }
}

template <int D>
__global__ void __launch_bounds__(PREFILL_THREADS, 1)
    fa_prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
  using C = PrefillCfg<D>;
  constexpr int NSLOT = C::NSLOT;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::Q_OFF;
  uint8_t* sKV = smem + C::KV_OFF;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* q_full = bars;
  uint64_t* full = bars + 1;
  uint64_t* empty = full + NSLOT;
  uint64_t* s_full = empty + NSLOT;
  uint64_t* p_full = s_full + Q_TILES;
  uint64_t* o_done = p_full + Q_TILES;
  uint64_t* drain = o_done + Q_TILES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t lim = p.wait_limit_ns;

  // ---- work unit: Q-tile pair `pair` of head `bh`; causal runs the longest pairs first
  const int BH = p.B * p.H;
  const int unit = blockIdx.x;
  const int pair = p.causal ? (p.n_qpairs - 1 - unit / BH) : (unit / BH);
  const int bh = unit % BH;
  const int nkv_total = (p.Nk + BLOCK_N - 1) / BLOCK_N;
  int n_t[Q_TILES];
#pragma unroll
  for (int t = 0; t < Q_TILES; ++t) {
    const int r0 = pair * (Q_TILES * BLOCK_M) + t * BLOCK_M;
    int n = 0;
    if (r0 < p.Nq) {
      if (p.causal) {
        // bottom-right alignment: row i sees keys j <= i + (Nk - Nq)
        const int last_key = min(r0 + BLOCK_M - 1, p.Nq - 1) + (p.Nk - p.Nq);
        n = last_key < 0 ? 0 : min(nkv_total, last_key / BLOCK_N + 1);
      } else {
        n = nkv_total;
      }
    }
    n_t[t] = n;
  }
  const int n_max = max(n_t[0], n_t[1]);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < NSLOT; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, 1);
    }
    for (int t = 0; t < Q_TILES; ++t) {
      mbar_init(s_full + t, 1);
      mbar_init(p_full + t, 128);
      mbar_init(o_done + t, 1);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 8) {
    setmaxnreg_dec<PREFILL_PRODUCER_REGS>();
    if (warp == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      const int rq = pair * (Q_TILES * BLOCK_M);
      mbar_arrive_expect_tx(q_full, Q_TILES * C::TILE_BYTES);
      for (int t = 0; t < Q_TILES; ++t)
        for (int b = 0; b < C::NBOX; ++b)
          tma_load_3d(sQ + t * C::TILE_BYTES + b * C::BOX_BYTES, &tmQ, q_full, 64 * b, rq + t * BLOCK_M, bh);
      int last = -1;
      bool ok = true;
      for (int j = 0; ok && j < n_max; ++j) {
        for (int w = 0; w < 2; ++w) {
          const int n = 2 * j + w;
          const int slot = n % NSLOT;
          if (!mbar_wait(empty + slot, ((n / NSLOT) & 1) ^ 1, lim, p.status, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full + slot, C::TILE_BYTES);
          for (int b = 0; b < C::NBOX; ++b)
            tma_load_3d(sKV + slot * C::TILE_BYTES + b * C::BOX_BYTES, w ? &tmV : &tmK, full + slot, 64 * b,
                        j * BLOCK_N, bh);
          last = n;
        }
      }
      if (!ok) {
        // error path: let the copies already issued land before the CTA exits
        mbar_wait_drain(q_full, 0, lim);
        for (int n = max(0, last - NSLOT + 1); n <= last; ++n)
          mbar_wait_drain(full + (n % NSLOT), (n / NSLOT) & 1, lim);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait(q_full, 0, lim, p.status, abort_flag);
      tc_fence_after();
      const uint32_t sQa = smem_u32(sQ);
      const uint32_t sKVa = smem_u32(sKV);
      for (int j = 0; ok && j < n_max; ++j) {
        const int nk = 2 * j;
        const int ks = nk % NSLOT;
        if (!(ok = mbar_wait(full + ks, (nk / NSLOT) & 1, lim, p.status, abort_flag))) break;
        tc_fence_after();
        for (int t = 0; t < Q_TILES && ok; ++t) {
          if (j >= n_t[t]) continue;
          if (j > 0) {
            // S_t is overwritten: the PV MMA that read P_t from it must be complete
            if (!(ok = mbar_wait(o_done + t, (j - 1) & 1, lim, p.status, abort_flag))) break;
            tc_fence_after();
          }
          const uint32_t dS = tmem + BLOCK_N * t;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::BOX_BYTES + (kk & 3) * 32;
            mma_ss(dS, sdesc_sw128(sQa + t * C::TILE_BYTES + off, 16, 1024),
                   sdesc_sw128(sKVa + ks * C::TILE_BYTES + off, 16, 1024), C::IDESC_S, kk > 0 ? 1u : 0u);
          }
          mma_commit(s_full + t);
        }
        if (!ok) break;
        mma_commit(empty + ks);  // K_j slot is free once these MMAs are done
        const int nv = 2 * j + 1;
        const int vs = nv % NSLOT;
        if (!(ok = mbar_wait(full + vs, (nv / NSLOT) & 1, lim, p.status, abort_flag))) break;
        tc_fence_after();
        for (int t = 0; t < Q_TILES && ok; ++t) {
          if (j >= n_t[t]) continue;
          if (!(ok = mbar_wait(p_full + t, j & 1, lim, p.status, abort_flag))) break;
          tc_fence_after();
          const uint32_t dO = tmem + 2 * BLOCK_N + D * t;
          const uint32_t aP = tmem + BLOCK_N * t;
#pragma unroll
          for (int kk = 0; kk < BLOCK_N / 16; ++kk) {
            mma_ts(dO, aP + kk * 8, sdesc_sw128(sKVa + vs * C::TILE_BYTES + kk * 2048, C::BOX_BYTES, 1024),
                   C::IDESC_O, (j > 0 || kk > 0) ? 1u : 0u);
          }
          mma_commit(o_done + t);
        }
        if (!ok) break;
        mma_commit(empty + vs);  // V_j slot is free once these MMAs are done
      }
      // every MMA this thread issued must finish before TMEM is released
      mma_commit(drain);
      mbar_wait_drain(drain, 0, lim);
    }
    __syncwarp();
    }
  } else {
    setmaxnreg_inc<PREFILL_SOFTMAX_REGS>();
    // ------------------------------------------------- softmax / correction
    const int t = warp >> 2;
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const int r0 = pair * (Q_TILES * BLOCK_M) + t * BLOCK_M;
    const int qi = r0 + row;
    const int n = n_t[t];
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + BLOCK_N * t;
    const uint32_t tO = tmem + lane_base + 2 * BLOCK_N + D * t;
    const float sl2 = p.scale_log2;
    const int delta = p.Nk - p.Nq;
    const int diag = qi + delta;          // last key this row may see (causal)
    const int tile_lim = r0 + delta;      // last key the first row of the tile may see
    const int nwords = (p.Nk + 31) >> 5;
    const uint32_t* krow = nullptr;
    if (p.keep != nullptr && qi < p.Nq) {
      const int b = bh / p.H, h = bh % p.H;
      krow = p.keep + b * p.msb + h * p.msh + static_cast<int64_t>(qi) * p.msq;
    }
    float m = -INFINITY;  // running max, in log2 units of the scaled score
    float l = 0.f;        // running sum of exponentials
    bool ok = true;

    for (int j = 0; j < n; ++j) {
      ok = mbar_wait(s_full + t, j & 1, lim, p.status, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      uint32_t s[BLOCK_N];
      tmem_ld32(tS + 0, s);
      tmem_ld32(tS + 32, s + 32);
      tmem_ld32(tS + 64, s + 64);
      tmem_ld32(tS + 96, s + 96);
      tmem_ld_wait32(s);
      reg_fence32(s + 32);
      reg_fence32(s + 64);
      reg_fence32(s + 96);

      const int kbase = j * BLOCK_N;
      const bool need_mask =
          (kbase + BLOCK_N > p.Nk) || (p.causal && kbase + BLOCK_N - 1 > tile_lim) || (p.keep != nullptr);
      if (need_mask) {
        uint32_t kw[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
        if (krow != nullptr) {
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const int wi = (kbase >> 5) + w;
            kw[w] = wi < nwords ? __ldg(krow + wi) : 0u;
          }
        }
#pragma unroll
        for (int c = 0; c < BLOCK_N; ++c) {
          const int key = kbase + c;
          bool vis = key < p.Nk;
          if (p.causal) vis = vis && key <= diag;
          vis = vis && ((kw[c >> 5] >> (c & 31)) & 1u);
          if (!vis) s[c] = f2u(-INFINITY);
        }
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < BLOCK_N; ++c) mx = fmaxf(mx, u2f(s[c]));
      const float m_tile = (mx == -INFINITY) ? -INFINITY : mx * sl2;
      const float m_new = fmaxf(m, m_tile);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2_approx(m - m_use);  // 0 while nothing was accumulated
      const float nm = -m_use;
      float sum = 0.f;
#pragma unroll
      for (int ch = 0; ch < BLOCK_N / 32; ++ch) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float x0 = u2f(s[ch * 32 + 2 * i]);
          const float x1 = u2f(s[ch * 32 + 2 * i + 1]);
          float p0 = ex2_approx(fmaf(x0, sl2, nm));
          float p1 = ex2_approx(fmaf(x1, sl2, nm));
          if (need_mask) {  // masked scores are -inf; keep them at 0 even for scale 0
            p0 = (x0 == -INFINITY) ? 0.f : p0;
            p1 = (x1 == -INFINITY) ? 0.f : p1;
          }
          sum += p0 + p1;
          pk[i] = pack_bf16x2(p0, p1);
        }
        tmem_st16(tS + ch * 16, pk);  // P (bf16 pairs) over the first 64 columns of S_t
      }
      l = l * alpha + sum;
      // O_t is quiescent here: S_t,j was issued only after PV_t,j-1 completed.
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t o[32];
          tmem_ld32(tO + ch * 32, o);
          tmem_ld_wait32(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = f2u(u2f(o[i]) * alpha);
          tmem_st32(tO + ch * 32, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(p_full + t);
      m = m_new;
    }

    // ---- epilogue: O = o / l (0 for an empty row), lse = m + ln l (-inf for an empty row)
    if (ok && n > 0) {
      ok = mbar_wait(o_done + t, (n - 1) & 1, lim, p.status, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
    }
    if (ok) {
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(p.o) + (static_cast<size_t>(bh) * p.Nq + qi) * D;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t o[32];
        if (n > 0) {
          tmem_ld32(tO + ch * 32, o);
          tmem_ld_wait32(o);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(u2f(o[2 * i]) * inv, u2f(o[2 * i + 1]) * inv);
        if (qi < p.Nq) {
          uint4* dst = reinterpret_cast<uint4*>(orow + ch * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
      if (p.lse != nullptr && qi < p.Nq)
        p.lse[static_cast<size_t>(bh) * p.Nq + qi] =
            (l > 0.f) ? (m + lg2_approx(l)) * 0.69314718055994530942f : -INFINITY;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D>
static cudaError_t launch_prefill_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                    const PrefillParams& p, cudaStream_t stream) {
  const long long units = static_cast<long long>(p.n_qpairs) * p.B * p.H;
  fa_prefill_kernel<D><<<static_cast<unsigned>(units), PREFILL_THREADS, PrefillCfg<D>::SMEM, stream>>>(tq, tk, tv,
                                                                                                      p);
  return cudaGetLastError();
}

int prefill_num_regs(int d) {
  cudaFuncAttributes a{};
  const cudaError_t e = (d == 64) ? cudaFuncGetAttributes(&a, fa_prefill_kernel<64>)
                                  : cudaFuncGetAttributes(&a, fa_prefill_kernel<128>);
  return e == cudaSuccess ? a.numRegs : -1;
}

size_t prefill_smem_bytes(int d) {
  return d == 64 ? PrefillCfg<64>::SMEM : PrefillCfg<128>::SMEM;
}

cudaError_t prefill_set_attributes(int d) {
  if (d == 64)
    return cudaFuncSetAttribute(fa_prefill_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                PrefillCfg<64>::SMEM);
  return cudaFuncSetAttribute(fa_prefill_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              PrefillCfg<128>::SMEM);
}

cudaError_t launch_prefill(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const PrefillParams& p, cudaStream_t stream) {
  return d == 64 ? launch_prefill_t<64>(tq, tk, tv, p, stream) : launch_prefill_t<128>(tq, tk, tv, p, stream);
}

}  // namespace fa
