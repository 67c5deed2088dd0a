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

// Wait used only to drain: returns true when the phase completed, false when
// the limit ran out first.
__device__ __forceinline__ bool mbar_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(a, parity)) return true;
    if ((i & 31u) == 31u && globaltimer_ns() - t0 > limit_ns) return false;
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

// ---------------------------------------------------------------------------
// Keys on the TMEM lanes (d = 128, at most 16 query rows per K/V head).
//
// With G * Nq <= 16 real rows, the 128-row query tile above is mostly padding:
// it pins 32 KB of Q, two 128-column S buffers and a 128-row O accumulator, so
// one CTA fills an SM and its set-up is never overlapped. Here the products
// run transposed, S^T = K Q^T (M = 128 keys, N = 16 rows) and
// O^T += V^T P^T (M = d, N = 16 rows): TMEM holds two 16-column S^T buffers
// and a 16-column O^T, P^T goes to shared memory, and with one K and one V
// stage a CTA needs 74 KB of shared memory: three CTAs share an SM, and one
// streams while another sets up. (Measured on the GQA decode workloads: three
// CTAs with one stage each 6.45 / 6.18 TB/s, two with two V stages or two P^T
// buffers 6.29-6.44 / 5.96-6.13, one with three stages 4.77 / 4.48, the
// 128-row kernel above 6.02 / 5.78.) The softmax runs one thread per key:
// the row max and sum over the 128 keys of a tile are warp reductions plus a
// four-warp exchange.
//
// At d = 64 the value product keeps M = 128: a V stage holds two 64-column
// boxes as at d = 128, the second zeroed once at the start and never loaded,
// so O^T lanes 64-127 stay zero and only lanes 0-63 are written out.
//
// fa_decode_grouped_kt_kernel<D, NK, NV, NPB, MINB>: one CTA per (split, b,
// kv head), 192 threads, registers sized for MINB CTAs per SM.
//   warp 0     TMA producer: Q (16 rows) once, K tiles into a ring of NK
//              stages, V tiles into a ring of NV stages.
//   warp 1     TMEM allocator and MMA issuer (converged warp, elected lane):
//              S^T_j into one of two buffers, the next one issued before PV_j.
//   warps 2-5  softmax, one key per thread (TMEM lane = key); P^T_j (bf16)
//              into one of NPB shared buffers in the 128-byte-swizzled
//              K-major layout the PV product reads.
namespace {

constexpr int DGT_NP = 16;        // query rows per tile (MMA N)
constexpr uint32_t DGT_BAR_ID = 1;  // named barrier of the four softmax warps

constexpr int DGT_THREADS = 192;   // warp 0 TMA, warp 1 MMA, warps 2-5 softmax
constexpr int DGT_SM_WARP0 = 2;

template <int D, int NK, int NV, int NPB>
struct DgtCfg {
  static_assert(D == 64 || D == 128, "head dim 64 or 128");
  static constexpr int NP = DGT_NP;
  static constexpr int NBX = D / 64;             // 64-column boxes of a K/V row or a Q row
  static constexpr int KV_BYTES = 128 * D * 2;   // one K or V tile: 128 keys x D bf16
  static constexpr int V_STAGE = 128 * 128 * 2;  // a V stage: two boxes (the second zero at d = 64)
  static constexpr int BOX = 128 * 128;          // one TMA box of a K/V tile: 128 rows x 64 bf16
  static constexpr int QBOX = NP * 128;          // one box of Q or P^T: NP rows x 64 bf16
  static constexpr int Q_OFF = 0;                // Q: NBX boxes
  static constexpr int P_OFF = Q_OFF + NBX * QBOX;  // P^T buffer b (of NPB): 2 boxes (keys 0-63, 64-127)
  static constexpr int K_OFF = P_OFF + NPB * 2 * QBOX;
  static constexpr int V_OFF = K_OFF + NK * KV_BYTES;
  static constexpr int RED_OFF = V_OFF + NV * V_STAGE;  // float [2][NP][4] row maxima per warp, [NP][4] row sums
  static constexpr int BAR_OFF = RED_OFF + 3 * NP * 4 * 4;
  static constexpr int NBAR = 1 + 2 * NK + 2 * NV + 2 + 2 + 2 + NPB + 1 + 1;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int SMEM = MISC_OFF + 16 + 1024;  // + slack to align the base to 1024
  static_assert(QBOX % 1024 == 0 && K_OFF % 1024 == 0 && V_OFF % 1024 == 0, "swizzle atoms are 1024-byte aligned");
  static constexpr uint32_t S_COL = 0;        // S^T_0 [0, NP), S^T_1 [NP, 2 NP)
  static constexpr uint32_t O_COL = 2 * NP;   // O^T [2 NP, 3 NP)
  static constexpr uint32_t TMEM_COLS = 64;
  static constexpr uint32_t IDESC_S = idesc_bf16_f32(128, NP, false);          // K and Q K-major
  static constexpr uint32_t IDESC_PV = idesc_bf16_f32(128, NP, false, true);   // A = V^T MN-major, B = P^T K-major
};

// 16 consecutive 32-bit TMEM columns of the thread's lane.
__device__ __forceinline__ void tmem_ld16_dg(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait16_dg(uint32_t* r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15])::"memory");
}
__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
// Named barrier over `count` threads that also returns the AND of `v` over them.
__device__ __forceinline__ bool bar_and(uint32_t id, uint32_t count, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.and.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(v ? 1u : 0u), "r"(id), "r"(count)
      : "memory");
  return r != 0u;
}
// Reduction of 16 values per lane over the 32 lanes of a warp, by halving: at
// each step a lane keeps half of its values and takes the other half from its
// partner. On return v[0] of lane l holds the result for value index
// (l >> 1) & 15. MAX: maximum, else sum.
template <bool MAX>
__device__ __forceinline__ void warp_reduce16(float* v, int lane) {
  auto op = [](float a, float b) { return MAX ? fmaxf(a, b) : a + b; };
#pragma unroll
  for (int half = 8, bit = 16; half >= 1; half >>= 1, bit >>= 1) {
    const bool hi = (lane & bit) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = hi ? v[i] : v[i + half];
      const float keep = hi ? v[i + half] : v[i];
      v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, bit));
    }
  }
  v[0] = op(v[0], __shfl_xor_sync(0xffffffffu, v[0], 1));
}

}  // namespace

template <int D, int NK, int NV, int NPB, int MINB>
__global__ void __launch_bounds__(DGT_THREADS, MINB)
    fa_decode_grouped_kt_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                                const __grid_constant__ CUtensorMap tmV, const DecodeGroupedParams p) {
  using C = DgtCfg<D, NK, NV, NPB>;
  constexpr int NP = C::NP;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* q_full = bars;                 // Q landed
  uint64_t* k_full = q_full + 1;           // [NK] K tile landed
  uint64_t* k_empty = k_full + NK;         // [NK] S^T of that tile completed
  uint64_t* v_full = k_empty + NK;         // [NV] V tile landed
  uint64_t* v_empty = v_full + NV;         // [NV] PV of that tile completed
  uint64_t* s_full = v_empty + NV;         // [2] S^T_j computed (buffer j & 1)
  uint64_t* s_free = s_full + 2;           // [2] S^T_j read by the softmax
  uint64_t* p_full = s_free + 2;           // [2] P^T_j stored (all 128 softmax threads)
  uint64_t* pv_done = p_full + 2;          // [NPB] PV_j completed (P^T buffer j % NPB, phase j / NPB)
  uint64_t* o_last = pv_done + NPB;        // the last PV completed
  uint64_t* drain = o_last + 1;            // every MMA completed (end of the issuer)
  float* red = reinterpret_cast<float*>(smem + C::RED_OFF);  // [2][NP][4] maxima, then [NP][4] sums
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
    for (int i = 0; i < NK; ++i) {
      mbar_init(k_full + i, 1);
      mbar_init(k_empty + i, 1);
    }
    for (int i = 0; i < NV; ++i) {
      mbar_init(v_full + i, 1);
      mbar_init(v_empty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(s_full + i, 1);
      mbar_init(s_free + i, 128);
      mbar_init(p_full + i, 128);
    }
    for (int i = 0; i < NPB; ++i) mbar_init(pv_done + i, 1);
    mbar_init(o_last, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == DG_MMA_WARP) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  if constexpr (D == 64) {
    // the second box of every V stage: zeros, read by the value product
    for (int i = threadIdx.x; i < NV * C::BOX / 16; i += DGT_THREADS) {
      const int st = i / (C::BOX / 16), w = i % (C::BOX / 16);
      st_shared_v4(smem_u32(smem + C::V_OFF + st * C::V_STAGE + C::BOX) + w * 16, 0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();  // the tensor core reads it through the async proxy
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == DG_TMA_WARP) {
    // ---------------------------------------------------------- TMA producer
    // K_j goes to slot j % NK once S^T_{j-NK} (its last reader) completed; V_j
    // to slot j % NV once PV_{j-NV} completed.
    const bool leader = lane == 0;
    bool ok = true;
    int nk = 0, nv = 0;
    if (leader && n > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(q_full, C::NBX * C::QBOX);
      for (int bx = 0; bx < C::NBX; ++bx) tma_load_3d(smem + C::Q_OFF + bx * C::QBOX, &tmQ, q_full, 64 * bx, 0, bg);
    }
    for (int j = 0; ok && j < n; ++j) {
      const int kt0 = k0 + j * 128;
      if (j >= NK) {
        ok = __all_sync(0xffffffffu, mbar_wait(k_empty + j % NK, ((j / NK) - 1) & 1, lim, p.status, abort_flag));
        if (!ok) break;
      }
      if (leader) {
        uint8_t* dst = smem + C::K_OFF + (j % NK) * C::KV_BYTES;
        mbar_arrive_expect_tx(k_full + j % NK, C::KV_BYTES);
        for (int bx = 0; bx < C::NBX; ++bx) tma_load_3d(dst + bx * C::BOX, &tmK, k_full + j % NK, 64 * bx, kt0, bg);
      }
      ++nk;
      if (j >= NV) {
        ok = __all_sync(0xffffffffu, mbar_wait(v_empty + j % NV, ((j / NV) - 1) & 1, lim, p.status, abort_flag));
        if (!ok) break;
      }
      if (leader) {
        uint8_t* dst = smem + C::V_OFF + (j % NV) * C::V_STAGE;
        mbar_arrive_expect_tx(v_full + j % NV, C::KV_BYTES);
        for (int bx = 0; bx < C::NBX; ++bx) tma_load_3d(dst + bx * C::BOX, &tmV, v_full + j % NV, 64 * bx, kt0, bg);
      }
      ++nv;
    }
    if (leader && n > 0) {
      // every copy issued lands before the CTA exits
      mbar_drain(q_full, 0, lim);
      for (int j = max(0, nk - NK); j < nk; ++j) mbar_drain(k_full + j % NK, (j / NK) & 1, lim);
      for (int j = max(0, nv - NV); j < nv; ++j) mbar_drain(v_full + j % NV, (j / NV) & 1, lim);
    }
    __syncwarp();
  } else if (warp == DG_MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    // The converged warp walks the loop; the elected lane issues every MMA and
    // commit.
    bool ok = true;
    auto wait_bar = [&](uint64_t* bar, uint32_t parity) {
      ok = __all_sync(0xffffffffu, mbar_wait(bar, parity, lim, p.status, abort_flag));
      tc_fence_after();
      return ok;
    };
    constexpr uint32_t DHI = sdesc_sw128_hi(1024);
    const uint32_t q_lo = sdesc_sw128_lo(smem_u32(smem + C::Q_OFF), 16);
    const uint32_t idesc_s = C::IDESC_S | (p.negate_s ? IDESC_NEGATE_A : 0u);
    // K-major K-step kk (16 elements = 32 bytes): (kk / 4) boxes plus (kk % 4) x 32 bytes in;
    // MN-major K-step kk (16 keys of V): 16 rows = 2048 bytes in (the two 64-column boxes BOX apart)
    auto kmaj = [](int kk, int box) { return static_cast<uint32_t>(((kk >> 2) * box + (kk & 3) * 32) >> 4); };
    auto issue_s = [&](int j) {  // S^T_j = K_j Q^T into buffer j & 1
      const uint32_t k_lo = sdesc_sw128_lo(smem_u32(smem + C::K_OFF + (j % NK) * C::KV_BYTES), 16);
      const uint32_t tS = tmem + C::S_COL + (j & 1) * NP;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk)
        if (elect_one())
          mma_ss_w(tS, k_lo + kmaj(kk, C::BOX), DHI, q_lo + kmaj(kk, C::QBOX), DHI, idesc_s, kk > 0 ? 1u : 0u);
      if (elect_one()) {
        mma_commit(s_full + (j & 1));
        mma_commit(k_empty + j % NK);
      }
    };
    auto issue_pv = [&](int j) {  // O^T += V_j^T P^T_j
      const uint32_t v_lo = sdesc_sw128_lo(smem_u32(smem + C::V_OFF + (j % NV) * C::V_STAGE), C::BOX);
      const uint32_t p_lo = sdesc_sw128_lo(smem_u32(smem + C::P_OFF + (j % NPB) * 2 * C::QBOX), 16);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        if (elect_one())
          mma_ss_w(tmem + C::O_COL, v_lo + static_cast<uint32_t>((kk * 2048) >> 4), DHI, p_lo + kmaj(kk, C::QBOX), DHI,
                   C::IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
      if (elect_one()) {
        mma_commit(pv_done + j % NPB);
        mma_commit(v_empty + j % NV);
        if (j == n - 1) mma_commit(o_last);
      }
    };
    bool issued_any = false;
    if (n > 0 && wait_bar(q_full, 0) && wait_bar(k_full, 0)) {
      issue_s(0);
      issued_any = true;
    }
    for (int j = 0; ok && j < n; ++j) {
      if (j + 1 < n) {
        // S^T_{j+1} goes to the buffer the softmax read S^T_{j-1} from
        if (!wait_bar(k_full + (j + 1) % NK, ((j + 1) / NK) & 1)) break;
        if (j >= 1 && !wait_bar(s_free + ((j + 1) & 1), ((j - 1) >> 1) & 1)) break;
        issue_s(j + 1);
      }
      if (!wait_bar(p_full + (j & 1), (j >> 1) & 1)) break;
      if (!wait_bar(v_full + j % NV, (j / NV) & 1)) break;
      issue_pv(j);
    }
    __syncwarp();
    // every MMA completed before TMEM is released (a commit tracks the elected
    // lane's MMAs; with none issued a plain arrive completes the phase)
    if (issued_any) {
      if (elect_one()) mma_commit(drain);
    } else if (lane == 0) {
      mbar_arrive(drain);
    }
    mbar_drain(drain, 0, lim);
    __syncwarp();
  } else if (warp >= DGT_SM_WARP0 && warp < DGT_SM_WARP0 + 4) {
    // --------------------------------------------------------------- softmax
    // Thread = key kr of the tile (its TMEM lane); its NP values are the
    // scores of the NP query rows (row r: head r / Nq of the group, token
    // r % Nq, which sees keys below L - Nq + r % Nq + 1; rows past R see none).
    // The four warps stop together: every exit decision passes a barrier
    // that ANDs the warps' states, so none waits at a barrier another left.
    const int wq = warp & 3;  // the TMEM lane quarter this warp may access
    const int kr = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const float sl2 = p.scale_log2;
    const int vis_all = max(0, L - p.Nq + 1);  // keys below this are visible to every row of the group
    float m_ref[NP];  // per row: reference max of P and O (log2 units), moved lazily
    float lp[NP];     // per row: this thread's part of the row sum on the reference m_ref
#pragma unroll
    for (int r = 0; r < NP; ++r) {
      m_ref[r] = -INFINITY;
      lp[r] = 0.f;
    }
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int key = k0 + j * 128 + kr;
      float x[NP];
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(s_full + (j & 1), (j >> 1) & 1, lim, p.status, abort_flag));
      if (ok) {
        tc_fence_after();
        uint32_t sv[NP];
        tmem_ld16_dg(tmem + lane_base + C::S_COL + (j & 1) * NP, sv);
        tmem_ld_wait16_dg(sv);
        tc_fence_before();
        mbar_arrive(s_free + (j & 1));
        const bool all_rows = key < vis_all;
#pragma unroll
        for (int r = 0; r < NP; ++r) {
          const bool vis = r < p.R && (all_rows || key < L - p.Nq + (r % p.Nq) + 1);
          x[r] = vis ? __uint_as_float(sv[r]) : -INFINITY;
        }
      } else {
#pragma unroll
        for (int r = 0; r < NP; ++r) x[r] = -INFINITY;
      }
      // row maxima of the tile: warp reduction, then the four warps' values
      float v[NP];
#pragma unroll
      for (int r = 0; r < NP; ++r) v[r] = x[r];
      warp_reduce16<true>(v, lane);
      float* rm = red + (j & 1) * NP * 4;
      if ((lane & 1) == 0) rm[((lane >> 1) & 15) * 4 + wq] = v[0];
      ok = bar_and(DGT_BAR_ID, 128, ok);
      if (!ok) break;
      float alpha[NP];
      bool rescale = false;
#pragma unroll
      for (int r = 0; r < NP; ++r) {
        const float4 m4 = reinterpret_cast<const float4*>(rm)[r];
        const float mx2 = fmaxf(fmaxf(m4.x, m4.y), fmaxf(m4.z, m4.w)) * sl2;  // -inf stays -inf (sl2 > 0)
        alpha[r] = 1.f;
        if (mx2 > m_ref[r] + DG_RESCALE_THRESHOLD) {
          if (m_ref[r] != -INFINITY) {
            alpha[r] = ex2_approx(m_ref[r] - mx2);
            rescale = true;
          }
          m_ref[r] = mx2;
          lp[r] *= alpha[r];
        }
      }
      // P^T buffer j % NPB is free once PV_{j-NPB} completed; O^T is rescaled
      // (columns of the rows whose reference moved) once PV_{j-1} completed
      if (j >= NPB)
        ok = __all_sync(0xffffffffu,
                        mbar_wait(pv_done + j % NPB, ((j - NPB) / NPB) & 1, lim, p.status, abort_flag));
      if (ok && rescale && j > 0) {
        ok = __all_sync(0xffffffffu,
                        mbar_wait(pv_done + (j - 1) % NPB, ((j - 1) / NPB) & 1, lim, p.status, abort_flag));
        if (ok) {
          tc_fence_after();
          uint32_t ov[NP];
          tmem_ld16_dg(tmem + lane_base + C::O_COL, ov);
          tmem_ld_wait16_dg(ov);
#pragma unroll
          for (int r = 0; r < NP; ++r) ov[r] = __float_as_uint(__uint_as_float(ov[r]) * alpha[r]);
          tmem_st16(tmem + lane_base + C::O_COL, ov);
          tmem_st_wait();
        }
      }
      if (ok) {
        // P^T_j[r][kr] = 2^(x * sl2 - m_ref), bf16, at row r, key kr of the
        // K-major layout: box kr / 64, 16-byte chunk (kr % 64) / 8 swizzled
        // with the row's position in its 8-row group
        const uint32_t pb = smem_u32(smem + C::P_OFF + (j % NPB) * 2 * C::QBOX) + (kr >> 6) * C::QBOX;
        const uint32_t chunk = static_cast<uint32_t>((kr & 63) >> 3), within = static_cast<uint32_t>((kr & 7) * 2);
#pragma unroll
        for (int r = 0; r < NP; ++r) {
          const float pr = (m_ref[r] == -INFINITY) ? 0.f : ex2_approx(fmaf(x[r], sl2, -m_ref[r]));  // -inf -> 0
          lp[r] += pr;
          const uint32_t addr = pb + (r >> 3) * 1024 + (r & 7) * 128 + ((chunk ^ static_cast<uint32_t>(r & 7)) << 4) + within;
          st_shared_u16(addr, __bfloat16_as_ushort(__float2bfloat16_rn(pr)));
        }
        fence_proxy_async_smem();  // the tensor core reads P^T through the async proxy
        tc_fence_before();
        mbar_arrive(p_full + (j & 1));
      }
    }
    // ---- epilogue: the unnormalised partial (o, m, l) of this split
    if (ok && n > 0) ok = __all_sync(0xffffffffu, mbar_wait(o_last, 0, lim, p.status, abort_flag));
    float v[NP];
#pragma unroll
    for (int r = 0; r < NP; ++r) v[r] = lp[r];
    warp_reduce16<false>(v, lane);
    float* rs = red + 2 * NP * 4;
    if ((lane & 1) == 0) rs[((lane >> 1) & 15) * 4 + wq] = v[0];
    ok = bar_and(DGT_BAR_ID, 128, ok);
    if (ok) {
      tc_fence_after();
      uint32_t ov[NP];
      if (n > 0) {
        tmem_ld16_dg(tmem + lane_base + C::O_COL, ov);  // O^T row kr = output column d = kr
        tmem_ld_wait16_dg(ov);
      } else {
#pragma unroll
        for (int r = 0; r < NP; ++r) ov[r] = 0u;
      }
      const int g = bg % p.Hkv;
      float m_mine = -INFINITY;
#pragma unroll
      for (int r = 0; r < NP; ++r) {
        if (r == kr) m_mine = m_ref[r];
        if (r < p.R && kr < D) {
          // query row (b, g * G + r / Nq, r % Nq) of [B, H, Nq]
          const size_t qrow = (static_cast<size_t>(b) * p.H + g * p.G + r / p.Nq) * p.Nq + r % p.Nq;
          p.ws_o[(qrow * p.S + s) * D + kr] = __uint_as_float(ov[r]);
        }
      }
      if (kr < p.R) {
        const float4 l4 = reinterpret_cast<const float4*>(rs)[kr];
        const size_t qrow = (static_cast<size_t>(b) * p.H + g * p.G + kr / p.Nq) * p.Nq + kr % p.Nq;
        const size_t part = qrow * p.S + s;
        p.ws_ml[part * 2 + 0] = m_mine;
        p.ws_ml[part * 2 + 1] = (l4.x + l4.y) + (l4.z + l4.w);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == DG_MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// fa_decode_grouped_cc_kernel<D, RP>: the same split-KV decode for groups of
// R <= RP <= 4 query rows per K/V head (one new token with up to four query
// heads per K/V head). With so few rows each K/V element feeds R multiply-adds
// per product, well below what the CUDA cores sustain at HBM speed, while a
// 128-lane tensor-core tile would be mostly padding; so the products run on
// the CUDA cores in packed fp32x2 and the kernel is a plain stream. The
// launcher takes it at d = 64 (there the keys-on-lanes tensor-core kernel
// streams at about 0.8 of its rate, the 128-row one at 0.6); at d = 128 the
// keys-on-lanes kernel measured faster than this one and is used instead.
//   warp 4     producer: one lane moves KT keys of K and KT keys of V per stage
//              into a ring of NST shared-memory stages with 1-D bulk copies
//              (cp.async.bulk, completion counted on the stage's mbarrier).
//   warps 0-3  consumers: warp w takes U rounds of KPW keys of each stage. A
//              key row (D bf16) is read by LPK = D/8 lanes, 16 bytes each, so
//              one warp-wide shared load covers 512 contiguous bytes. A lane
//              forms the partial dots of its 8 columns with the RP query rows;
//              a halving exchange over the key's lanes leaves each lane the
//              full score of one row (its own row), which it turns into a
//              weight against that row's reference max; the RP weights are
//              then broadcast over the key's lanes and every lane accumulates
//              its 8 columns of o for all rows.
// Online state per lane group (the lanes of one key): per row a reference max
// in log2 units, moved lazily as in the tensor-core kernels, a sum and an
// o-slice. At the end the groups are combined through shared memory and the
// split writes its unnormalised partial (o, m, l) like the other kernels.
namespace {

#ifndef FA_DGC_NW
#define FA_DGC_NW 4    // consumer warps of the CUDA-core kernel
#endif
#ifndef FA_DGC_U
#define FA_DGC_U 4     // key rounds per consumer warp and stage
#endif
#ifndef FA_DGC_NST
#define FA_DGC_NST 4   // shared-memory stages
#endif
#ifndef FA_DGC_MINB
#define FA_DGC_MINB 3  // CTAs per SM the registers and shared memory are sized for
#endif
constexpr int DGC_NW = FA_DGC_NW;
constexpr int DGC_THREADS = 32 * (DGC_NW + 1);  // + the producer warp
constexpr int DGC_U = FA_DGC_U;
constexpr uint32_t DGC_FULL = 0xffffffffu;
constexpr uint32_t DGC_BAR_ID = 1;  // named barrier of all the CTA's warps at the end

template <int D, int RP>
struct DgcCfg {
  static_assert(D == 64 || D == 128, "head dim 64 or 128");
  static_assert(RP == 1 || RP == 2 || RP == 4, "1, 2 or 4 query rows");
  static constexpr int LPK = D / 8;                  // lanes per key row
  static constexpr int KPW = 32 / LPK;               // keys per warp-wide round
  static constexpr int KT = DGC_NW * DGC_U * KPW;    // keys per stage
  static constexpr int ROW = D * 2;                  // bytes of a key row
  static constexpr int STAGE = 2 * KT * ROW;         // K rows, then V rows
  static constexpr int NST = FA_DGC_NST;
  static constexpr int NG = DGC_NW * KPW;            // lane groups of the CTA
  // at the end the stages hold the groups' states: float [NG][RP][D] o-slices, then [NG][RP][2] (m, l)
  static constexpr int ACC_OFF = 0;
  static constexpr int ML_OFF = ACC_OFF + NG * RP * D * 4;
  static_assert(ML_OFF + NG * RP * 2 * 4 <= NST * STAGE, "the final states fit in the stages");
  static constexpr int BAR_OFF = NST * STAGE;        // full[NST], empty[NST]
  static constexpr int MISC_OFF = BAR_OFF + 2 * NST * 8;
  static constexpr int SMEM = MISC_OFF + 16 + 128;   // + slack to align the base to 128
  static_assert(FA_DGC_MINB * (SMEM + 1024) <= 228 * 1024, "shared memory for the CTAs per SM");
};

// Lane (within its key's LPK lanes) that holds the full score of row r after
// dgc_reduce_own.
template <int RP, int LPK>
__device__ __forceinline__ int dgc_owner(int r) {
  if constexpr (RP == 4) return (r >> 1) * (LPK / 2) + (r & 1) * (LPK / 4);
  else if constexpr (RP == 2) return r * (LPK / 2);
  else return 0;
}

// Sum of v[r] over the LPK lanes of a key, returning on lane li the sum for
// its own row (dgc_owner(own) has the same bits as li in the halving
// positions). The first log2(RP) steps halve the values a lane carries (it
// keeps one half and sends the other to its partner); the rest are plain
// butterfly steps, so the LPK / RP lanes of a row end with the same sum.
template <int RP, int LPK>
__device__ __forceinline__ float dgc_reduce_own(const float (&v)[RP], int li) {
  constexpr int REST = RP == 4 ? LPK / 8 : RP == 2 ? LPK / 4 : LPK / 2;  // plain steps after the halving
  float x;
  if constexpr (RP == 4) {
    const bool ha = (li & (LPK / 2)) != 0;
    const float w0 = (ha ? v[2] : v[0]) + __shfl_xor_sync(DGC_FULL, ha ? v[0] : v[2], LPK / 2);
    const float w1 = (ha ? v[3] : v[1]) + __shfl_xor_sync(DGC_FULL, ha ? v[1] : v[3], LPK / 2);
    const bool hb = (li & (LPK / 4)) != 0;
    x = (hb ? w1 : w0) + __shfl_xor_sync(DGC_FULL, hb ? w0 : w1, LPK / 4);
  } else if constexpr (RP == 2) {
    const bool ha = (li & (LPK / 2)) != 0;
    x = (ha ? v[1] : v[0]) + __shfl_xor_sync(DGC_FULL, ha ? v[0] : v[1], LPK / 2);
  } else {
    x = v[0];
  }
#pragma unroll
  for (int off = REST; off >= 1; off >>= 1) x += __shfl_xor_sync(DGC_FULL, x, off);
  return x;
}

template <int RP, int LPK>
__device__ __forceinline__ int dgc_own_row(int li) {
  if constexpr (RP == 4) return ((li & (LPK / 2)) ? 2 : 0) + ((li & (LPK / 4)) ? 1 : 0);
  else if constexpr (RP == 2) return (li & (LPK / 2)) ? 1 : 0;
  else return 0;
}

// Two consecutive bf16 (the low half first) as an fp32 pair.
__device__ __forceinline__ uint64_t dgc_bf16x2_f2(uint32_t w) {
  return f2pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__device__ __forceinline__ uint4 dgc_lds128(uint32_t addr) {
  uint4 r;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(addr));
  return r;
}

// exp2(m - M), 0 for a part that saw no key (m = -inf).
__device__ __forceinline__ float dgc_rebase(float m, float M) { return m == -INFINITY ? 0.f : ex2_approx(m - M); }

}  // namespace

template <int D, int RP>
__global__ void __launch_bounds__(DGC_THREADS, FA_DGC_MINB) fa_decode_grouped_cc_kernel(const DecodeGroupedParams p) {
  using C = DgcCfg<D, RP>;
  constexpr int LPK = C::LPK, KPW = C::KPW, KT = C::KT, NST = C::NST, ROW = C::ROW;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);  // [NST] stage landed
  uint64_t* empty = full + NST;                                      // [NST] stage read by the 4 consumer warps
  float* sacc = reinterpret_cast<float*>(smem + C::ACC_OFF);
  float* sml = reinterpret_cast<float*>(smem + C::ML_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF);
  volatile int* drained = abort_flag + 1;  // every copy the producer issued has landed

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t lim = p.wait_limit_ns;
  const int s = static_cast<int>(blockIdx.x) % p.S;
  const int bg = static_cast<int>(blockIdx.x) / p.S;  // b * Hkv + g
  const int b = bg / p.Hkv;
  const int g = bg % p.Hkv;
  const int L = p.seqlens ? min(max(p.seqlens[b], 0), p.Nk) : p.Nk;
  const int k0 = s * p.chunk;
  const int k1 = min(L, k0 + p.chunk);
  const int n = k1 > k0 ? (k1 - k0 + KT - 1) / KT : 0;  // stages of this split

  if (threadIdx.x == 0) {
    for (int i = 0; i < NST; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, DGC_NW);
    }
    *abort_flag = 0;
    *drained = 1;
    fence_mbar_init();
  }
  __syncthreads();

  const size_t kv_off = static_cast<size_t>(bg) * p.Nk * ROW;  // bytes to this (b, K/V head)'s rows
  const size_t row0 = (static_cast<size_t>(b) * p.H + static_cast<size_t>(g) * p.G) * p.Nq;  // first query row
  const int sub = lane / LPK;  // key of the round within the warp
  const int li = lane % LPK;   // 16-byte slice of the key row
  const int gi = warp * KPW + sub;

  if (warp == DGC_NW) {
    // ---- producer: stage i holds keys [k0 + i KT, min(k1, k0 + (i + 1) KT))
    if (lane == 0) {
      const uint8_t* kg = static_cast<const uint8_t*>(p.k) + kv_off;
      const uint8_t* vg = static_cast<const uint8_t*>(p.v) + kv_off;
      int issued = 0;
      for (int i = 0; i < n; ++i) {
        const int st = i % NST;
        if (i >= NST && !mbar_wait(empty + st, ((i / NST) - 1) & 1, lim, p.status, abort_flag)) break;
        const int key = k0 + i * KT;
        const uint32_t bytes = static_cast<uint32_t>(min(KT, k1 - key) * ROW);
        uint8_t* dst = smem + st * C::STAGE;
        mbar_arrive_expect_tx(full + st, 2 * bytes);
        bulk_load_1d(dst, kg + static_cast<size_t>(key) * ROW, bytes, full + st);
        bulk_load_1d(dst + KT * ROW, vg + static_cast<size_t>(key) * ROW, bytes, full + st);
        issued = i + 1;
      }
      // no copy may still be writing shared memory when it is reused or the CTA exits
      for (int i = max(0, issued - NST); i < issued; ++i)
        if (!mbar_drain(full + i % NST, (i / NST) & 1, lim)) *drained = 0;
    }
    __syncwarp();
    named_bar_sync(DGC_BAR_ID, DGC_THREADS);  // the stages are free
  } else {
    // ---- consumers
    // query rows of this group, columns li*8 .. li*8+7, in log2 units with the scale's sign
    const float qs = p.negate_s ? -p.scale_log2 : p.scale_log2;
    uint64_t q2[RP][4];
#pragma unroll
    for (int r = 0; r < RP; ++r) {
      uint4 w = make_uint4(0, 0, 0, 0);
      if (r < p.R)
        w = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q) + (row0 + r) * D + li * 8);
      const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) q2[r][i] = fmul2(dgc_bf16x2_f2(ww[i]), f2pack(qs, qs));
    }
    // row r (head g G + r / Nq, token r % Nq) sees key j iff j < L - Nq + 1 + r % Nq
    const int own = dgc_own_row<RP, LPK>(li);
    const int lim_own = own < p.R ? min(k1, L - p.Nq + 1 + own % p.Nq) : k0;
    const int base_lane = lane & ~(LPK - 1);
    float m_own = -INFINITY, l_own = 0.f;
    uint64_t acc[RP][4];
#pragma unroll
    for (int r = 0; r < RP; ++r)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[r][i] = 0ull;

    for (int i = 0; i < n; ++i) {
      const int st = i % NST;
      if (!__all_sync(DGC_FULL, mbar_wait(full + st, (i / NST) & 1, lim, p.status, abort_flag))) break;
      const int kl0 = warp * (DGC_U * KPW) + sub;  // stage-local key of round 0
      const int key0 = k0 + i * KT + kl0;
      const uint32_t ks = smem_u32(smem + st * C::STAGE) + kl0 * ROW + li * 16;
      const uint32_t vs = ks + KT * ROW;
      uint4 kr[DGC_U], vr[DGC_U];
#pragma unroll
      for (int u = 0; u < DGC_U; ++u) {
        if (key0 + u * KPW < k1) {  // the rows past the split's end were not copied
          kr[u] = dgc_lds128(ks + u * KPW * ROW);
          vr[u] = dgc_lds128(vs + u * KPW * ROW);
        } else {
          kr[u] = make_uint4(0, 0, 0, 0);
          vr[u] = make_uint4(0, 0, 0, 0);
        }
      }
      float x[DGC_U];
#pragma unroll
      for (int u = 0; u < DGC_U; ++u) {
        const uint64_t k2[4] = {dgc_bf16x2_f2(kr[u].x), dgc_bf16x2_f2(kr[u].y), dgc_bf16x2_f2(kr[u].z),
                                dgc_bf16x2_f2(kr[u].w)};
        float dv[RP];
#pragma unroll
        for (int r = 0; r < RP; ++r) {
          uint64_t d2 = fmul2(q2[r][0], k2[0]);
          d2 = ffma2(q2[r][1], k2[1], d2);
          d2 = ffma2(q2[r][2], k2[2], d2);
          d2 = ffma2(q2[r][3], k2[3], d2);
          float lo, hi;
          f2unpack(d2, lo, hi);
          dv[r] = lo + hi;
        }
        const float sc = dgc_reduce_own<RP, LPK>(dv, li);
        x[u] = (key0 + u * KPW < lim_own) ? sc : -INFINITY;
      }
      // lazy reference max of the own row
      float mx = x[0];
#pragma unroll
      for (int u = 1; u < DGC_U; ++u) mx = fmaxf(mx, x[u]);
      float alpha_own = 1.f;
      bool moved = false;
      if (mx > m_own + DG_RESCALE_THRESHOLD) {
        if (m_own != -INFINITY) {
          alpha_own = ex2_approx(m_own - mx);
          moved = true;
        }
        m_own = mx;
        l_own *= alpha_own;
      }
      if (__any_sync(DGC_FULL, moved)) {
#pragma unroll
        for (int r = 0; r < RP; ++r) {
          const float a = __shfl_sync(DGC_FULL, alpha_own, base_lane + dgc_owner<RP, LPK>(r));
          const uint64_t a2 = f2pack(a, a);
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[r][j] = fmul2(acc[r][j], a2);
        }
      }
#pragma unroll
      for (int u = 0; u < DGC_U; ++u) {
        const float pu = (m_own == -INFINITY) ? 0.f : ex2_approx(x[u] - m_own);  // x = -inf -> 0
        l_own += pu;
        const uint64_t v2[4] = {dgc_bf16x2_f2(vr[u].x), dgc_bf16x2_f2(vr[u].y), dgc_bf16x2_f2(vr[u].z),
                                dgc_bf16x2_f2(vr[u].w)};
#pragma unroll
        for (int r = 0; r < RP; ++r) {
          const float pr = __shfl_sync(DGC_FULL, pu, base_lane + dgc_owner<RP, LPK>(r));
          const uint64_t p2 = f2pack(pr, pr);
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[r][j] = ffma2(p2, v2[j], acc[r][j]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + st);
    }
    // this group's state to shared memory (over the stages, once every copy
    // landed): o-slices from every lane, (m, l) of each row from that row's
    // first owner lane
    named_bar_sync(DGC_BAR_ID, DGC_THREADS);
    if (*drained) {
#pragma unroll
      for (int r = 0; r < RP; ++r) {
        float o[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) f2unpack(acc[r][j], o[2 * j], o[2 * j + 1]);
        float4* dst = reinterpret_cast<float4*>(sacc + (gi * RP + r) * D + li * 8);
        dst[0] = make_float4(o[0], o[1], o[2], o[3]);
        dst[1] = make_float4(o[4], o[5], o[6], o[7]);
      }
      if (li == dgc_owner<RP, LPK>(own)) {
        sml[(gi * RP + own) * 2 + 0] = m_own;
        sml[(gi * RP + own) * 2 + 1] = l_own;
      }
    }
  }
  __syncthreads();
  // ---- combine the NG groups: one thread per (row, column); after a timeout
  // (*drained = 0) the stages may still change, so nothing is combined
  for (int idx = threadIdx.x; *drained && idx < p.R * D; idx += DGC_THREADS) {
    const int r = idx / D, c = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int t = 0; t < C::NG; ++t) M = fmaxf(M, sml[(t * RP + r) * 2]);
    float o = 0.f, l = 0.f;
#pragma unroll
    for (int t = 0; t < C::NG; ++t) {
      const float f = dgc_rebase(sml[(t * RP + r) * 2], M);
      o = fmaf(sacc[(t * RP + r) * D + c], f, o);
      l = fmaf(sml[(t * RP + r) * 2 + 1], f, l);
    }
    const size_t part = (row0 + r) * p.S + s;
    p.ws_o[part * D + c] = o;
    if (c == 0) {
      p.ws_ml[part * 2 + 0] = M;
      p.ws_ml[part * 2 + 1] = l;
    }
  }
}

template <int D>
static cudaError_t launch_decode_grouped_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                           const DecodeGroupedParams& p, cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>(static_cast<long long>(p.B) * p.Hkv * p.S);
  fa_decode_grouped_kernel<D><<<grid, DG_THREADS, DgCfg<D>::SMEM, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

#ifndef FA_DGT_NK
#define FA_DGT_NK 1   // K stages of the keys-on-lanes kernel
#endif
#ifndef FA_DGT_NV
#define FA_DGT_NV 1   // V stages
#endif
#ifndef FA_DGT_NPB
#define FA_DGT_NPB 1  // P^T buffers
#endif
#ifndef FA_DGT_MINB
#define FA_DGT_MINB 3 // CTAs per SM the registers are sized for
#endif
#ifndef FA_DGT_ENABLE
#define FA_DGT_ENABLE 1
#endif
template <int D>
using DgtKernel = DgtCfg<D, FA_DGT_NK, FA_DGT_NV, FA_DGT_NPB>;
#define FA_DGT_KERNEL(D) fa_decode_grouped_kt_kernel<D, FA_DGT_NK, FA_DGT_NV, FA_DGT_NPB, FA_DGT_MINB>

#ifndef FA_DGC_ENABLE
#define FA_DGC_ENABLE 1
#endif
// Groups of at most four query rows stream through the CUDA-core kernel at d = 64.
static bool use_cc(int d, int R) { return FA_DGC_ENABLE && d == 64 && R <= 4; }
// The keys-on-lanes kernel takes the other groups of at most 16 query rows per K/V head
// (at d = 64 with 5-16 rows it measured 4.46 TB/s against 3.53 for the 128-row kernel).
static bool use_kt(int, int R) { return FA_DGT_ENABLE && R <= DGT_NP; }

template <int D>
static cudaError_t launch_kt(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const DecodeGroupedParams& p, cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>(static_cast<long long>(p.B) * p.Hkv * p.S);
  FA_DGT_KERNEL(D)<<<grid, DGT_THREADS, DgtKernel<D>::SMEM, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

template <int D, int RP>
static cudaError_t launch_cc(const DecodeGroupedParams& p, cudaStream_t stream) {
  const unsigned grid = static_cast<unsigned>(static_cast<long long>(p.B) * p.Hkv * p.S);
  fa_decode_grouped_cc_kernel<D, RP><<<grid, DGC_THREADS, DgcCfg<D, RP>::SMEM, stream>>>(p);
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_cc_d(const DecodeGroupedParams& p, cudaStream_t stream) {
  if (p.R == 1) return launch_cc<D, 1>(p, stream);
  if (p.R == 2) return launch_cc<D, 2>(p, stream);
  return launch_cc<D, 4>(p, stream);
}

template <int D, int RP>
static cudaError_t set_cc_attributes() {
  return cudaFuncSetAttribute(fa_decode_grouped_cc_kernel<D, RP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              DgcCfg<D, RP>::SMEM);
}

template <int D>
static cudaError_t set_cc_attributes_d() {
  cudaError_t e = set_cc_attributes<D, 1>();
  if (e == cudaSuccess) e = set_cc_attributes<D, 2>();
  if (e == cudaSuccess) e = set_cc_attributes<D, 4>();
  return e;
}

int decode_grouped_q_box_rows(int d, int R) { return use_kt(d, R) ? DGT_NP : 128; }

cudaError_t decode_grouped_set_attributes(int d) {
  if (d == 64) {
    cudaError_t e = set_cc_attributes_d<64>();
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(FA_DGT_KERNEL(64), cudaFuncAttributeMaxDynamicSharedMemorySize, DgtKernel<64>::SMEM);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(fa_decode_grouped_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                DgCfg<64>::SMEM);
  }
  cudaError_t e = cudaFuncSetAttribute(fa_decode_grouped_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       DgCfg<128>::SMEM);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(FA_DGT_KERNEL(128), cudaFuncAttributeMaxDynamicSharedMemorySize, DgtKernel<128>::SMEM);
}

cudaError_t launch_decode_grouped(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                  const DecodeGroupedParams& p, cudaStream_t stream) {
  if (use_cc(d, p.R)) return launch_cc_d<64>(p, stream);
  if (use_kt(d, p.R)) return d == 64 ? launch_kt<64>(tq, tk, tv, p, stream) : launch_kt<128>(tq, tk, tv, p, stream);
  return d == 64 ? launch_decode_grouped_t<64>(tq, tk, tv, p, stream)
                 : launch_decode_grouped_t<128>(tq, tk, tv, p, stream);
}

}  // namespace fa
