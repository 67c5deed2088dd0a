// Split-KV decode on the tensor cores for grouped K/V heads, several query
// tokens per sequence and per-sequence KV lengths.
//
// Decode streams the KV cache from HBM; the sequence is split and the partial
// results merged ("FlashAttention: Attention Is Limited by Memory, Not Math",
// section "Where it helps, and where it does not"; the merge re-bases each
// part to the common max, "Handwritten Notes on Flash Attention", section
// "Merging two blocks"). With grouped K/V heads (H query heads share Hkv K/V
// heads, G = H / Hkv) and Nq new tokens per sequence, the G * Nq query rows of
// one (b, kv head) read the same K/V stream. They form one 128-row query tile
// here, so every K/V byte is read once per group and both products run on
// tcgen05: S = Q K^T and O += P V, fp32 accumulators in TMEM.
//
// Visibility: sequence b holds L_b keys (seqlens_k[b], or Nk when none is
// given), the Nq new tokens are its last Nq positions, and token t sees key j
// iff j < L_b and j <= L_b - Nq + t (bottom-right causal alignment within the
// sequence). A token that sees no key gets O = 0 and lse = -inf.
//
// fa_decode_grouped_kernel<D>: one CTA per (split, b, kv head), 256 threads.
//   warp 0     TMA producer: the Q tile once, then K and V tiles of the split
//              into a ring of NS stages.
//   warp 1     TMEM allocator and MMA issuer: S_j into one of two S buffers
//              (the next tile's S is issued before the current PV), PV_j
//              after the softmax of tile j stored P.
//   warps 4-7  softmax: one query row per thread, online state in log2
//              units with a lazily moved reference max; P (bf16) is written
//              over the first 64 columns of its S buffer; at the end the
//              unnormalised partial (o, m, l) goes to the caller's workspace.
// The merge of the splits is the split-KV decode's merge kernel, run over
// the B * H * Nq query rows.
#include <cuda_bf16.h>

#include "decode_grouped.cuh"
#include "fa_ptx.cuh"

namespace fa {

namespace {

constexpr int DG_THREADS = 256;
constexpr int DG_TMA_WARP = 0;
constexpr int DG_MMA_WARP = 1;
constexpr int DG_SM_WARP0 = 4;  // warps 4-7
// The reference max moves only when a row's max exceeds it by more than this
// (log2 units), so the weights stay below 2^8 and O is rescaled rarely.
constexpr float DG_RESCALE_THRESHOLD = 8.0f;

// Wait used only to drain: returns when the phase completed or the limit ran out.
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(a, parity)) return;
    if ((i & 31u) == 31u && globaltimer_ns() - t0 > limit_ns) return;
  }
}

template <int D>
struct DgCfg {
  static_assert(D == 64 || D == 128, "head dim 64 or 128");
  static constexpr int TILE = 128 * D * 2;  // one 128-row tile of bf16
  static constexpr int BOX = 128 * 128;     // one TMA box: 128 rows x 64 bf16
  static constexpr int NBOX = D / 64;
  static constexpr int NS = (D == 64) ? 6 : 3;  // K/V stages (one key tile's K and V each)
  static constexpr int Q_OFF = 0;
  static constexpr int KV_OFF = TILE;  // stage s: K at KV_OFF + 2 s TILE, V right after
  static constexpr int BAR_OFF = KV_OFF + NS * 2 * TILE;
  static constexpr int NBAR = 1 + 2 * NS + 2 + 2 + 1 + 1;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int SMEM = MISC_OFF + 16 + 1024;  // + slack to align the base to 1024
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  static constexpr uint32_t S_COL = 0;    // S_0 [0, 128), S_1 [128, 256)
  static constexpr uint32_t O_COL = 256;  // O [256, 256 + D)
  static constexpr uint32_t IDESC_S = idesc_bf16_f32(128, 128, false);  // Q and K K-major
  static constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, D, true);    // V MN-major
};

}  // namespace

template <int D>
__global__ void __launch_bounds__(DG_THREADS, 1)
    fa_decode_grouped_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                             const __grid_constant__ CUtensorMap tmV, const DecodeGroupedParams p) {
  using C = DgCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::Q_OFF;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* q_full = bars;                  // the Q tile landed
  uint64_t* kv_full = bars + 1;             // [NS] K and V of a key tile landed
  uint64_t* kv_empty = bars + 1 + C::NS;    // [NS] PV of that tile completed
  uint64_t* s_full = bars + 1 + 2 * C::NS;  // [2] S_j computed
  uint64_t* p_full = s_full + 2;            // [2] P_j stored (all 128 softmax threads)
  uint64_t* o_done = p_full + 2;            // PV_j completed (one phase per key tile)
  // The last PV completed. The epilogue gets a barrier of its own: the softmax
  // may finish the last tile while o_done is still short of the last two PVs,
  // and a parity wait cannot tell a phase two ahead.
  uint64_t* o_last = o_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t lim = p.wait_limit_ns;
  const int s = static_cast<int>(blockIdx.x) % p.S;
  const int bg = static_cast<int>(blockIdx.x) / p.S;  // b * Hkv + g
  const int b = bg / p.Hkv;
  const int L = p.seqlens ? min(max(p.seqlens[b], 0), p.Nk) : p.Nk;
  const int k0 = s * p.chunk;
  const int k1 = min(L, k0 + p.chunk);
  const int n = k1 > k0 ? (k1 - k0 + 127) / 128 : 0;  // key tiles of this split

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(kv_full + i, 1);
      mbar_init(kv_empty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full + i, 1);
      mbar_init(p_full + i, 128);
    }
    mbar_init(o_done, 1);
    mbar_init(o_last, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == DG_MMA_WARP) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == DG_TMA_WARP) {
    // ---------------------------------------------------------- TMA producer
    const bool leader = lane == 0;
    bool ok = true;
    int issued = 0;
    if (leader && n > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(q_full, C::TILE);
      for (int bx = 0; bx < C::NBOX; ++bx) tma_load_3d(sQ + bx * C::BOX, &tmQ, q_full, 64 * bx, 0, bg);
    }
    for (int j = 0; ok && j < n; ++j) {
      const int st = j % C::NS;
      if (j >= C::NS) {
        ok = mbar_wait(kv_empty + st, ((j / C::NS) - 1) & 1, lim, p.status, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
      if (leader) {
        uint8_t* sK = smem + C::KV_OFF + st * 2 * C::TILE;
        const int kt0 = k0 + j * 128;
        mbar_arrive_expect_tx(kv_full + st, 2 * C::TILE);
        for (int bx = 0; bx < C::NBOX; ++bx) {
          tma_load_3d(sK + bx * C::BOX, &tmK, kv_full + st, 64 * bx, kt0, bg);
          tma_load_3d(sK + C::TILE + bx * C::BOX, &tmV, kv_full + st, 64 * bx, kt0, bg);
        }
      }
      ++issued;
    }
    if (leader && n > 0) {
      // every copy issued lands before the CTA exits
      mbar_drain(q_full, 0, lim);
      for (int j = max(0, issued - C::NS); j < issued; ++j) mbar_drain(kv_full + j % C::NS, (j / C::NS) & 1, lim);
    }
    __syncwarp();
  } else if (warp == DG_MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    const bool leader = lane == 0;
    bool ok = true;
    auto wait_bar = [&](uint64_t* bar, uint32_t parity) {
      ok = mbar_wait(bar, parity, lim, p.status, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
      return ok;
    };
    constexpr uint32_t DHI = sdesc_sw128_hi(1024);
    const uint32_t q_lo = sdesc_sw128_lo(smem_u32(sQ), 16);
    const uint32_t idesc_s = C::IDESC_S | (p.negate_s ? IDESC_NEGATE_A : 0u);
    // K-major K-step kk of a tile: (kk / 4) boxes plus (kk % 4) x 32 bytes in;
    // MN-major K-step kk: 16 rows = 2048 bytes in (64-column boxes BOX apart)
    auto kmaj = [](int kk) { return static_cast<uint32_t>(((kk >> 2) * C::BOX + (kk & 3) * 32) >> 4); };
    auto mnmaj = [](int kk) { return static_cast<uint32_t>((kk * 2048) >> 4); };
    auto issue_s = [&](int j) {  // S_{j&1} = Q K_j^T
      const uint32_t kb = smem_u32(smem + C::KV_OFF + (j % C::NS) * 2 * C::TILE);
      const uint32_t k_lo = sdesc_sw128_lo(kb, 16);
      const uint32_t tS = tmem + C::S_COL + (j & 1) * 128;
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss_w(tS, q_lo + kmaj(kk), DHI, k_lo + kmaj(kk), DHI, idesc_s, kk > 0 ? 1u : 0u);
        mma_commit(s_full + (j & 1));
      }
    };
    if (n > 0 && wait_bar(q_full, 0) && wait_bar(kv_full, 0)) issue_s(0);
    for (int j = 0; ok && j < n; ++j) {
      if (j + 1 < n) {
        // S_{j+1} goes to the buffer PV_{j-1} read P from
        if (!wait_bar(kv_full + (j + 1) % C::NS, ((j + 1) / C::NS) & 1)) break;
        if (j >= 1 && !wait_bar(o_done, (j - 1) & 1)) break;
        issue_s(j + 1);
      }
      if (!wait_bar(p_full + (j & 1), (j >> 1) & 1)) break;
      if (leader) {
        // O += P_j V_j (A = P from the first 64 columns of S_{j&1}, B = V_j MN-major)
        const uint32_t vb = smem_u32(smem + C::KV_OFF + (j % C::NS) * 2 * C::TILE + C::TILE);
        const uint32_t v_lo = sdesc_sw128_lo(vb, C::BOX);
        const uint32_t tP = tmem + C::S_COL + (j & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts_w(tmem + C::O_COL, tP + kk * 8, v_lo + mnmaj(kk), DHI, C::IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(o_done);
        mma_commit(kv_empty + j % C::NS);
        if (j == n - 1) mma_commit(o_last);
      }
    }
    if (leader && n > 0) mbar_drain(o_done, (n - 1) & 1, lim);  // every MMA completed before TMEM is released
    __syncwarp();
  } else if (warp >= DG_SM_WARP0 && warp < DG_SM_WARP0 + 4) {
    // --------------------------------------------------------------- softmax
    const int wq = warp - DG_SM_WARP0;
    const int r = wq * 32 + lane;  // query row of the tile: head (r / Nq) of the group, token (r % Nq)
    const bool row_ok = r < p.R;
    const int t = r % p.Nq;
    // keys below vis are visible to this row; rows past the group see none
    const int vis = row_ok ? max(0, L - p.Nq + t + 1) : 0;
    const int vis_all = max(0, L - p.Nq + 1);  // visible to every row of the group
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const float sl2 = p.scale_log2;
    bool ok = true;
    float m_ref = -INFINITY;  // reference max (log2 units) of P and O
    float l = 0.f;
    for (int j = 0; ok && j < n; ++j) {
      const int kt0 = k0 + j * 128;
      ok = mbar_wait(s_full + (j & 1), (j >> 1) & 1, lim, p.status, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tS = tmem + lane_base + C::S_COL + (j & 1) * 128;
      uint32_t sv[128];
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) tmem_ld32(tS + ch * 32, sv + ch * 32);
      tmem_ld_wait32(sv);
#pragma unroll
      for (int ch = 1; ch < 4; ++ch) reg_fence32(sv + ch * 32);
      // mask (only a tile that reaches past the keys every row sees) and row max
      const int c_end = vis - kt0;  // columns below c_end are visible
      const bool full = kt0 + 128 <= vis_all;
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 128; ++c) {
        float x = __uint_as_float(sv[c]);
        if (!full && c >= c_end) x = -INFINITY;
        sv[c] = __float_as_uint(x);
        mx = fmaxf(mx, x);
      }
      const float mx2 = mx * sl2;  // log2 units (-inf stays -inf: scale_log2 > 0, the sign is in the MMA)
      // move the reference max only when this tile's max exceeds it by more than the threshold
      const bool move = mx2 > m_ref + DG_RESCALE_THRESHOLD;
      float alpha = 1.f;
      if (move) {
        alpha = (m_ref == -INFINITY) ? 0.f : ex2_approx(m_ref - mx2);
        m_ref = mx2;
        l *= alpha;
      }
      uint32_t pk[64];
      float sum = 0.f;
      if (m_ref == -INFINITY) {
#pragma unroll
        for (int i = 0; i < 64; ++i) pk[i] = 0u;
      } else {
        const float nm = -m_ref;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          const float p0 = ex2_approx(fmaf(__uint_as_float(sv[2 * i]), sl2, nm));  // -inf -> 0
          const float p1 = ex2_approx(fmaf(__uint_as_float(sv[2 * i + 1]), sl2, nm));
          sum += p0 + p1;
          pk[i] = pack_bf16x2(p0, p1);
        }
      }
      l += sum;
      tmem_st32(tS, pk);  // P over the S columns already read
      tmem_st32(tS + 32, pk + 32);
      // O holds PV_0 .. PV_{j-1}, taken relative to the old reference: rescale
      // it (whole warp, tcgen05 is warp-collective) once PV_{j-1} completed
      if (__any_sync(0xffffffffu, move && alpha != 1.f && j > 0)) {
        ok = mbar_wait(o_done, (j - 1) & 1, lim, p.status, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
        tc_fence_after();
        const uint32_t tO = tmem + lane_base + C::O_COL;
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t ov[32];
          tmem_ld32(tO + ch * 32, ov);
          tmem_ld_wait32(ov);
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = __float_as_uint(__uint_as_float(ov[i]) * alpha);
          tmem_st32(tO + ch * 32, ov);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(p_full + (j & 1));
    }
    // ---- epilogue: the unnormalised partial (o, m, l) of this split
    if (ok && n > 0) {
      ok = mbar_wait(o_last, 0, lim, p.status, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      tc_fence_after();
    }
    if (ok) {
      const int g = bg % p.Hkv;
      const int hh = r / p.Nq;
      // query row (b, g * G + hh, t) of [B, H, Nq]
      const size_t qrow = (static_cast<size_t>(b) * p.H + g * p.G + hh) * p.Nq + t;
      const size_t part = qrow * p.S + s;
      float* wo = p.ws_o + part * D;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t ov[32];
        if (n > 0) {  // warp-uniform: every lane loads, only rows of the group store
          tmem_ld32(tmem + lane_base + C::O_COL + ch * 32, ov);
          tmem_ld_wait32(ov);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) ov[i] = 0u;
        }
        if (row_ok) {
          float4* w4 = reinterpret_cast<float4*>(wo + ch * 32);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            w4[v] = make_float4(__uint_as_float(ov[4 * v]), __uint_as_float(ov[4 * v + 1]),
                                __uint_as_float(ov[4 * v + 2]), __uint_as_float(ov[4 * v + 3]));
        }
      }
      if (row_ok) {
        p.ws_ml[part * 2 + 0] = m_ref;
        p.ws_ml[part * 2 + 1] = l;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == DG_MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D>
static cudaError_t launch_decode_grouped_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                           const DecodeGroupedParams& p, cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>(static_cast<long long>(p.B) * p.Hkv * p.S);
  fa_decode_grouped_kernel<D><<<grid, DG_THREADS, DgCfg<D>::SMEM, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

cudaError_t decode_grouped_set_attributes(int d) {
  if (d == 64)
    return cudaFuncSetAttribute(fa_decode_grouped_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                DgCfg<64>::SMEM);
  return cudaFuncSetAttribute(fa_decode_grouped_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              DgCfg<128>::SMEM);
}

cudaError_t launch_decode_grouped(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                  const DecodeGroupedParams& p, cudaStream_t stream) {
  return d == 64 ? launch_decode_grouped_t<64>(tq, tk, tv, p, stream)
                 : launch_decode_grouped_t<128>(tq, tk, tv, p, stream);
}

}  // namespace fa
