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
// A work unit is two 128-row Q tiles of one (b, h). The launch is persistent:
// one CTA per SM walks its share of the units (round robin; causal units,
// sorted longest first, in snake order), and every barrier phase runs on
// across units, so the next unit's loads and first MMAs overlap the current
// unit's last steps and epilogue.
// 384 threads = 3 warpgroups; after set-up the softmax warpgroups take more
// registers and the producer warpgroup fewer (setmaxnreg). The producer
// warpgroup is warps 8-11; within it:
//   warp 8      TMA producer for K_j / V_j, into separate rings of slots.
//   warp 9      TMEM allocator; with warp 10, MMA issuers (one per Q tile):
//               S_t = Q_t K_j^T into TMEM, later O_t += P_t V_j.
//   warp 11     TMA producer for Q (one tile per buffer per unit).
//   warps 0-3   softmax for Q tile 0, warps 4-7 for Q tile 1 (warp w reads
//               TMEM lanes 32 (w % 4) ..): each thread
//               owns one query row (TMEM lane), reads its 128 scores with
//               tcgen05.ld, applies the mask from absolute positions, folds
//               the tile into (m, l), writes P (bf16) to TMEM and rescales
//               its O row when the running max rose; at the end it divides by
//               l and writes O (bf16, through a TMA store) and lse (fp32).
// TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256,256+D), O_1 [256+D,256+2D).
// The two Q tiles ping-pong: while one softmax warpgroup works, the tensor
// core runs the other tile's MMAs.
#include <cuda_bf16.h>

#include <algorithm>
#include <climits>

#include "fa_debug.cuh"
#include "fa_ptx.cuh"

namespace fa {

// Tuning knobs (compile time): exponential pairs per 16 computed on the FMA
// pipe, and whether the second Q tile starts half a period late.
#ifndef FA_EMU_PAIRS_D64
#define FA_EMU_PAIRS_D64 0
#endif
#ifndef FA_EMU_PAIRS_D128
#define FA_EMU_PAIRS_D128 0
#endif
#ifndef FA_LATE_STORE_WAIT
#define FA_LATE_STORE_WAIT 1   // O staging: wait for the previous store's reads only before rewriting the buffer
#endif
#ifndef FA_QDB_D64
#define FA_QDB_D64 1           // two Q buffers per tile at d = 64
#endif
#ifndef FA_QDB_RING
#define FA_QDB_RING 4          // K and V ring slots beside them (bf16)
#endif
#ifndef FA_STAGGER_D64
#define FA_STAGGER_D64 1
#endif
#ifndef FA_STAGGER_D128
#define FA_STAGGER_D128 0
#endif
#ifndef FA_SORDER
#define FA_SORDER 1              // S_0 and S_1 are issued alternately (see the MMA issuers)
#endif
#ifndef FA_EARLY_POLL
#define FA_EARLY_POLL 1          // poll the next barriers early, use the results late
#endif
#ifndef FA_PERSIST_D64
#define FA_PERSIST_D64 1         // one CTA per SM walking many units (else one CTA per unit)
#endif
#ifndef FA_PERSIST_D128
#define FA_PERSIST_D128 0
#endif
#ifndef FA_UNIT_DONE_EARLY_D64
#define FA_UNIT_DONE_EARLY_D64 0   // an issuer signals unit_done after its last S of a unit (else after its last PV)
#endif
#ifndef FA_UNIT_DONE_EARLY_D128
#define FA_UNIT_DONE_EARLY_D128 1
#endif
#ifndef FA_LEAD_LONGER
#define FA_LEAD_LONGER 1         // the Q tile with more key tiles issues its scores first
#endif
#ifndef FA_O_STAGE
#define FA_O_STAGE 1             // separate O staging buffers where shared memory allows (d = 64)
#endif
#ifndef FA_ELECT_ISSUE_D64
#define FA_ELECT_ISSUE_D64 0     // the converged issuer warp walks the loop; an elected lane issues
#endif
#ifndef FA_ELECT_ISSUE_D128
#define FA_ELECT_ISSUE_D128 1
#endif
#ifndef FA_SOLO_ISSUE_D64
#define FA_SOLO_ISSUE_D64 (!FA_ELECT_ISSUE_D64)  // lane 0 of each issuer warp runs the MMA loop alone (no warp votes)
#endif
#ifndef FA_SOLO_ISSUE_D128
#define FA_SOLO_ISSUE_D128 0
#endif
#ifndef FA_STAGGER_MIN_TILES
#define FA_STAGGER_MIN_TILES 8   // only units this long amortise the delayed start
#endif

// F8: q, k and v are e4m3 codes (kind::f8f6f4 products, P rounded to e4m3);
// otherwise bf16 (kind::f16). O is bf16 either way.
template <int D, bool F8 = false>
struct PrefillCfg {
  static_assert(D == 64 || D == 128, "head dim 64 or 128");
  static constexpr int ESZ = F8 ? 1 : 2;              // bytes per q, k, v element
  static constexpr int TILE_BYTES = BLOCK_N * D * ESZ;  // one Q, K or V tile (128 rows x D elements)
  // Shared-memory rows of a tile are 128 bytes (128-byte swizzle), except the
  // e4m3 tiles at d = 64, whose 64-byte rows use the 64-byte swizzle.
  static constexpr int ROW_BYTES = (D * ESZ < 128) ? D * ESZ : 128;
  static constexpr int BOX_BYTES = 128 * ROW_BYTES;   // one TMA box: 128 rows
  static constexpr int BOX_ELEMS = ROW_BYTES / ESZ;   // elements per box row (64 bf16, 128 or 64 e4m3)
  static constexpr int NBOX = D / BOX_ELEMS;
  // high word of every operand descriptor: 8-row groups of ROW_BYTES rows
  static constexpr uint32_t DESC_HI = (ROW_BYTES == 64) ? sdesc_sw64_hi(512) : sdesc_sw128_hi(1024);
  static constexpr int O_TILE_BYTES = BLOCK_M * D * 2;  // one bf16 O tile
  static constexpr int NBOX_O = D / 64;
  static constexpr int O_BOX_BYTES = 128 * 128;       // one box of the bf16 O tile: 128 rows x 64 bf16
  // products: one K-step takes 32 bytes of every A and B row (16 bf16 or 32
  // e4m3 elements); S = Q K^T has D * ESZ / 32 of them, O += P V has
  // BLOCK_N * ESZ / 32 (each K-step of V is PV_KROWS rows of ROW_BYTES bytes)
  static constexpr int KSTEPS_S = D * ESZ / 32;
  static constexpr int KSTEPS_PV = BLOCK_N * ESZ / 32;
  static constexpr int PV_KROWS = 32 / ESZ;
  // K and V stream through separate rings. K_j is read only by S = Q K_j^T,
  // V_j only by the later O += P V_j, so the K ring runs ahead of the V ring:
  // K_{j+1} can land while P_j is still being computed. Both slots of key
  // tile j are released together, by one release barrier per tile that both
  // issuers signal once their MMAs reading tile j have completed.
  // At d = 64 each Q tile has two buffers (QDB): unit k's Q goes to buffer
  // k % 2, so it loads while unit k - 1 runs instead of after unit k - 1's
  // last score product. (Measured: e4m3 +0.5 % / +2 % non-causal / causal,
  // bf16 flat; with the bf16 K and V rings cut to three slots, causal -3 %.)
  static constexpr bool QDB = (D == 64) && FA_QDB_D64;
  static constexpr int QB = QDB ? 2 : 1;                // Q buffers per tile
  static constexpr int NK = (D == 128 && !F8) ? 3 : ((QDB && !F8) ? FA_QDB_RING : 4);  // K ring slots
  static constexpr int NV = (D == 128 && !F8) ? 2 : ((QDB && !F8) ? FA_QDB_RING : 4);  // V ring slots
  static constexpr int NR = NK > NV ? NK : NV;        // release barriers (tile j uses j % NR)
  static constexpr int Q_OFF = 0;                     // Q of tile t, buffer b at Q_OFF + (b Q_TILES + t) TILE_BYTES
  static constexpr int K_OFF = QB * Q_TILES * TILE_BYTES;
  static constexpr int V_OFF = K_OFF + NK * TILE_BYTES;
  // At d = 64 the epilogue stages O in buffers of its own, so the next unit's
  // Q may be loaded as soon as this unit's score MMAs are done; at d = 128
  // there is no room and O is staged in the Q buffer. An e4m3 Q tile is
  // half the size of the bf16 O tile, so that path always stages O apart.
  static constexpr bool O_STAGE = ((D == 64) && FA_O_STAGE) || F8;
  static constexpr int O_OFF = V_OFF + NV * TILE_BYTES;
  static constexpr int BAR_OFF = O_OFF + (O_STAGE ? Q_TILES * O_TILE_BYTES : 0);
  static_assert(!QDB || O_STAGE, "two Q buffers need O staged apart (the epilogue would stage O in buffer 0)");
  // TMEM columns: S_0 [0,128), S_1 [128,256), O_t at O_COL + D*t; with
  // SEP_P (d = 64) P_t gets its own 64 columns at P_COL + 64*t, otherwise P_t
  // overwrites the first P_WORDS columns of S_t. P is packed 4 / ESZ values
  // per 32-bit column: 64 columns of bf16 pairs or 32 of e4m3 quads.
  static constexpr bool SEP_P = (D == 64);
  static constexpr int P_WORDS = BLOCK_N * ESZ / 4;
  static constexpr uint32_t O_COL = 2 * BLOCK_N;
  static constexpr uint32_t P_COL = SEP_P ? O_COL + Q_TILES * D : 0;
  static constexpr uint32_t P_STRIDE = SEP_P ? P_WORDS : BLOCK_N;
  static_assert(!SEP_P || P_COL + Q_TILES * P_WORDS <= 512, "TMEM budget");
  static constexpr int NBAR = 6 * Q_TILES + 2 * (QB - 1) * Q_TILES + NK + NV + NR + 2;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int SMEM = MISC_OFF + 16 + 1024;   // + slack to align the base to 1024
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t IDESC_S =
      F8 ? idesc_e4m3_f32(128, 128, false) : idesc_bf16_f32(128, 128, false);  // Q, K both K-major
  static constexpr uint32_t IDESC_O = F8 ? idesc_e4m3_f32(128, D, true) : idesc_bf16_f32(128, D, true);  // V MN-major
  // Softmax tuning: exponential pairs (of 16 per 32 columns) computed on the
  // FMA pipe instead of the MUFU unit, and the lazy-rescale threshold.
  static constexpr int EMU_PAIRS = (D == 64) ? FA_EMU_PAIRS_D64 : FA_EMU_PAIRS_D128;
  static constexpr float RESCALE_LOG2 = 8.0f;
  static constexpr bool STAGGER = (D == 64) ? FA_STAGGER_D64 : FA_STAGGER_D128;
  // Persistent launch where it measured faster: at d = 64, where the next
  // unit's Q loads while the current unit finishes (separate O staging). At
  // d = 128 the Q buffer also stages O, so the next Q waits for the epilogue
  // and one CTA per unit is faster.
  static constexpr bool PERSIST = (D == 64) ? FA_PERSIST_D64 : FA_PERSIST_D128;
  static constexpr bool UNIT_DONE_EARLY = (D == 64) ? FA_UNIT_DONE_EARLY_D64 : FA_UNIT_DONE_EARLY_D128;
  // Where it measured faster (d = 64), only lane 0 of each MMA-issuing warp
  // walks the issue loop: its waits then need no warp vote, and lanes 1-31
  // wait once, at the end, for the drain.
  static constexpr bool SOLO_ISSUE = (D == 64) ? FA_SOLO_ISSUE_D64 : FA_SOLO_ISSUE_D128;
  // The MMA-issuing warps run converged and issue each MMA and commit from
  // the lane elect.sync picks. Alone, one such thread keeps the tensor pipe
  // fed, where an MMA loop under `lane == 0` issues at about half the rate.
  // In this kernel it measured 2-5 % faster at d = 128 (bf16 and e4m3); at
  // d = 64 lane 0 walking the loop alone stays faster (no warp votes).
  static constexpr bool ELECT_ISSUE = ((D == 64) ? FA_ELECT_ISSUE_D64 : FA_ELECT_ISSUE_D128) && !SOLO_ISSUE;
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

// One query row's scores s[0..127] (fp32 bit patterns, masked ones -inf) ->
// P = 2^(s * sl2 - m) as 64 bf16 pairs written over s[0..63] (pair i after
// scores 2i and 2i + 1 were read, so no score is overwritten before its
// use), returning the row sum of the fp32 exponentials. EMU pairs of every
// 16 use the FMA-pipe exponential.
// With MASKED, -inf scores give exactly 0 on both exponential paths.
// When poll_bar is nonzero, the barrier at that shared address is polled
// (parity poll_par) halfway through and the result left in *poll_res.
template <bool MASKED, int EMU, bool F8 = false>
__device__ __forceinline__ float softmax_tile_p(uint32_t* s, uint64_t sl2x2, uint64_t nm2, uint32_t poll_bar,
                                                uint32_t poll_par, uint32_t* poll_res) {
  uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
  if constexpr (F8) {
    // e4m3 P: four exponentials per packed word, word w = keys 4w .. 4w + 3
    // written over s[w] (its scores were read first). ex2(-inf) = 0.
#pragma unroll
    for (int w = 0; w < BLOCK_N / 4; ++w) {
      if (FA_EARLY_POLL && w == BLOCK_N / 8 && poll_bar != 0u) *poll_res = mbar_test(poll_bar, poll_par);
      const int c = 4 * w;
      const uint64_t xa = ffma2(f2pack(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), sl2x2, nm2);
      const uint64_t xb = ffma2(f2pack(__uint_as_float(s[c + 2]), __uint_as_float(s[c + 3])), sl2x2, nm2);
      float x0, x1, x2, x3;
      f2unpack(xa, x0, x1);
      f2unpack(xb, x2, x3);
      const float p0 = ex2_approx(x0), p1 = ex2_approx(x1), p2 = ex2_approx(x2), p3 = ex2_approx(x3);
      acc2[w & 3] = fadd2(acc2[w & 3], fadd2(f2pack(p0, p1), f2pack(p2, p3)));
      s[w] = pack_e4m3x4(p0, p1, p2, p3);
    }
    float a0, a1, a2, a3;
    f2unpack(fadd2(acc2[0], acc2[1]), a0, a1);
    f2unpack(fadd2(acc2[2], acc2[3]), a2, a3);
    return (a0 + a1) + (a2 + a3);
  } else {
#pragma unroll
  for (int ch = 0; ch < BLOCK_N / 32; ++ch) {
    if (FA_EARLY_POLL && ch == BLOCK_N / 64 && poll_bar != 0u) *poll_res = mbar_test(poll_bar, poll_par);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int c = ch * 32 + 2 * i;
      const uint64_t x2 = ffma2(f2pack(__uint_as_float(s[c]), __uint_as_float(s[c + 1])), sl2x2, nm2);
      uint64_t p2;
      if (i >= 16 - EMU) {
        p2 = exp2_fma2(x2);
        if (MASKED) {
          float p0, p1;
          f2unpack(p2, p0, p1);
          p0 = (s[c] == 0xff800000u) ? 0.f : p0;
          p1 = (s[c + 1] == 0xff800000u) ? 0.f : p1;
          p2 = f2pack(p0, p1);
        }
      } else {
        float x0, x1;
        f2unpack(x2, x0, x1);
        p2 = f2pack(ex2_approx(x0), ex2_approx(x1));  // ex2(-inf) = 0
      }
      acc2[i & 3] = fadd2(acc2[i & 3], p2);
      float p0, p1;
      f2unpack(p2, p0, p1);
      s[ch * 16 + i] = pack_bf16x2(p0, p1);  // pair index (ch * 32 + 2i) / 2
    }
  }
  float a0, a1, a2, a3;
  f2unpack(fadd2(acc2[0], acc2[1]), a0, a1);
  f2unpack(fadd2(acc2[2], acc2[3]), a2, a3);
  return (a0 + a1) + (a2 + a3);
  }
}

// Waits on two (three) barriers. The first polls are non-blocking and issued
// back to back, so when every phase has already completed the thread pays
// one barrier round trip instead of two (three). A null third barrier is
// skipped.
__device__ __forceinline__ bool mbar_wait2(uint64_t* a, uint32_t pa, uint64_t* b, uint32_t pb, uint64_t lim,
                                           unsigned int* status, volatile int* abort, uint64_t* c = nullptr,
                                           uint32_t pc = 0) {
  const uint32_t ra = mbar_test(smem_u32(a), pa);
  const uint32_t rb = mbar_test(smem_u32(b), pb);
  const uint32_t rc = c == nullptr ? 1u : mbar_test(smem_u32(c), pc);
  if (!ra && !mbar_wait(a, pa, lim, status, abort)) return false;
  if (!rb && !mbar_wait(b, pb, lim, status, abort)) return false;
  if (!rc && !mbar_wait(c, pc, lim, status, abort)) return false;
  return true;
}

// Work unit u: units below p.split_from are Q-tile pair u (pair `pair` of
// head `bh`); the pairs from p.split_from on, which would fill only part of a
// last round of CTAs, are split into two single-tile units each (tile 0, then
// tile 1). Causal runs the longest pairs first.
struct Unit {
  int bh, pair, n0, n1;  // n_t: key tiles Q tile t visits
  bool act0, act1;       // whether this unit computes Q tile t at all
};
__device__ __forceinline__ Unit unit_info(const PrefillParams& p, int u, int kv_keep) {
  const int BH = p.B * p.H;
  Unit w;
  int pu = u, only = -1;
  if (u >= p.split_from) {
    pu = p.split_from + (u - p.split_from) / 2;
    only = (u - p.split_from) & 1;
  }
  if (p.causal && p.band > 0) {
    // Bands of `band` pair lengths, longest band first; inside a band one
    // head's pairs (longest first), then the next head's. The CTAs running at
    // once then read the K/V of about (CTAs / band) heads, which L2 holds,
    // while the last units launched are still the shortest.
    const int per_band = p.band * BH;
    const int bi = pu / per_band;
    const int r = pu - bi * per_band;
    const int bw = min(p.band, p.n_qpairs - bi * p.band);  // pairs in this band (the last may be short)
    const int head = r / bw;
    w.pair = p.n_qpairs - 1 - (bi * p.band + (r - head * bw));
    w.bh = head;
  } else {
    w.pair = p.causal ? (p.n_qpairs - 1 - pu / BH) : (pu / BH);
    w.bh = pu % BH;
  }
  const int nkv_total = (p.Nk + BLOCK_N - 1) / BLOCK_N;
  int n[Q_TILES];
#pragma unroll
  for (int t = 0; t < Q_TILES; ++t) {
    const int r0 = w.pair * (Q_TILES * BLOCK_M) + t * BLOCK_M;
    int nt = 0;
    if (r0 < p.Nq) {
      if (p.causal) {
        // bottom-right alignment: row i sees keys j <= i + (Nk - Nq)
        const int last_key = min(r0 + BLOCK_M - 1, p.Nq - 1) + (p.Nk - p.Nq);
        nt = last_key < 0 ? 0 : min(nkv_total, last_key / BLOCK_N + 1);
      } else {
        nt = nkv_total;
      }
    }
    n[t] = (only < 0 || only == t) ? min(nt, kv_keep) : 0;
  }
  w.n0 = n[0];
  w.n1 = n[1];
  w.act0 = only != 1;
  w.act1 = only != 0;
  return w;
}
// The k-th unit of CTA c of G, or a value >= U when it has no k-th unit.
// Round robin; with `snake` every other round runs in reverse CTA order, so
// with units sorted longest first the per-CTA sums stay balanced.
__device__ __forceinline__ int unit_of(int c, int k, int G, bool snake) {
  return k * G + ((snake && (k & 1)) ? (G - 1 - c) : c);
}

template <int D, bool F8>
__global__ void __launch_bounds__(prefill_threads(D), 1)
    fa_prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                      const PrefillParams p) {
  using C = PrefillCfg<D, F8>;
  constexpr int NK = C::NK, NV = C::NV, NR = C::NR;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem + C::Q_OFF;
  uint8_t* sK = smem + C::K_OFF;
  uint8_t* sV = smem + C::V_OFF;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  // Q barriers of tile t, buffer b at QB t + b; unit k uses buffer k % QB
  // in phase k / QB (qbuf, qpar below)
  uint64_t* q_full = bars;                     // Q_t of unit k landed
  uint64_t* q_free = q_full + C::QB * Q_TILES; // Q_t buffer free again after unit k: its score MMAs are
                                               // done (O_STAGE) or its O store read it
  uint64_t* full_k = q_free + C::QB * Q_TILES; // K of key tile g landed in slot g % NK
  uint64_t* full_v = full_k + NK;          // V of key tile g landed in slot g % NV
  uint64_t* rel = full_v + NV;             // both issuers are done with key tile g (g % NR)
  uint64_t* s_full = rel + NR;             // S_t of step c complete (per-tile step count c)
  uint64_t* p_full = s_full + Q_TILES;     // P_t of step c stored
  uint64_t* o_done = p_full + Q_TILES;     // PV_t of step c complete
  uint64_t* s_free = o_done + Q_TILES;     // S_t of step c read by the softmax
  uint64_t* unit_done = s_free + Q_TILES;  // both tiles' score MMAs of unit k completed (phase k)
  uint64_t* drain = unit_done + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);
  int* kv_keep_slot = reinterpret_cast<int*>(smem + C::MISC_OFF + 8);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Roles by warpgroup: the two softmax warpgroups (warps 0-7) and the
  // producer warpgroup (K/V TMA, MMA issuers, Q TMA); pw is a warp's index
  // within the producer warpgroup. (The producer warpgroup placed first, at
  // warps 0-3, measured 2-3 % slower.)
  const bool producer = warp >= PREFILL_SOFTMAX_WARPS;
  const int pw = warp - PREFILL_SOFTMAX_WARPS;
  const int sw = warp;
  const bool alloc_warp = producer && pw == 1;  // the first MMA issuer allocates and frees TMEM
  const uint64_t lim = p.wait_limit_ns;
  const int U = p.units;
  const int G = static_cast<int>(gridDim.x);
  const int cta = static_cast<int>(blockIdx.x);
  const bool snake = p.causal != 0;
  // With one key mask broadcast over the rows of a head, key tiles after the
  // last one with any key kept are skipped by every role; the host then
  // launches one CTA per unit and warp 11 finds that tile before set-up ends.
  const bool trim = p.keep != nullptr && p.msq == 0;

  if (trim && producer && pw == 3) {
    const int bh = unit_info(p, cta, INT_MAX).bh;  // one unit per CTA here: unit cta
    const int b = bh / p.H, h = bh % p.H;
    const uint32_t* kb = p.keep + b * p.msb + h * p.msh;
    const int nwords = (p.Nk + 31) >> 5;
    int last = -1;
    for (int wi = lane; wi < nwords; wi += 32)
      if (__ldg(kb + wi) != 0u) last = wi;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, off));
    if (lane == 0) *kv_keep_slot = (last < 0) ? 0 : (last * 32) / BLOCK_N + 1;
  }

  if (threadIdx.x == 0) {
    for (int t = 0; t < Q_TILES; ++t) {
      for (int b = 0; b < C::QB; ++b) {
        mbar_init(q_full + C::QB * t + b, 1);
        mbar_init(q_free + C::QB * t + b, 1);
      }
      mbar_init(s_full + t, 1);
      mbar_init(p_full + t, 128);
      mbar_init(o_done + t, 1);
      mbar_init(s_free + t, 128);
    }
    for (int i = 0; i < NK; ++i) mbar_init(full_k + i, 1);
    for (int i = 0; i < NV; ++i) mbar_init(full_v + i, 1);
    for (int i = 0; i < NR; ++i) mbar_init(rel + i, Q_TILES);  // both MMA-issuing warps
    mbar_init(unit_done, Q_TILES);
    mbar_init(drain, Q_TILES);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (alloc_warp) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int kv_keep = trim ? *kv_keep_slot : INT_MAX;
  // Every role walks the same unit sequence; barrier phases run on across
  // units (counts of units, key tiles and per-tile steps done so far).
  auto unit_at = [&](int k) { return unit_of(cta, k, G, snake); };
  auto qbuf = [](int k) { return C::QB == 2 ? (k & 1) : 0; };                              // Q buffer of unit k
  auto qpar = [](int k) { return static_cast<uint32_t>((C::QB == 2 ? (k >> 1) : k) & 1); };  // its phase parity
  int dbg_count0 = 0, dbg_count1 = 0;  // debug build: steps of a tile (softmax) / K and V loads (producer)

  if (producer) {
    setmaxnreg_dec<prefill_producer_regs(D)>();
    const bool leader = lane == 0;
    if (pw == 0) {
      // ------------------------------------------------------ K/V TMA producer
      // The whole warp runs the loop and waits; lane 0 issues the copies.
      // Key tile g (counted over all units of this CTA) goes to K slot g % NK
      // once tile g - NK was released, and to V slot g % NV once tile g - NV
      // was released (release of tile i is phase i / NR of rel[i % NR]).
      if (leader) {
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmO);
      }
      auto wait_rel = [&](int i) -> bool {
        if (i < 0) return true;
        const bool w = mbar_wait(rel + (i % NR), static_cast<uint32_t>((i / NR) & 1), lim, p.status, abort_flag);
        return __all_sync(0xffffffffu, w) != 0;
      };
      int g = 0, nlk = 0, nlv = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int u = unit_at(k);
        if (u >= U) break;
        const Unit w = unit_info(p, u, kv_keep);
        const int n_max = max(w.n0, w.n1);
        for (int jj = 0; jj < n_max; ++jj, ++g) {
          if (!(ok = wait_rel(g - NK))) break;
          if (leader) {
            uint8_t* dst = sK + (g % NK) * C::TILE_BYTES;
            mbar_arrive_expect_tx(full_k + (g % NK), C::TILE_BYTES);
            for (int b = 0; b < C::NBOX; ++b)
              if (dbg_tma_ok(p.dbg, DBG_LOAD_K, C::BOX_ELEMS * b, jj * BLOCK_N, w.bh, D, p.Nk, p.B * p.H, C::ESZ))
                tma_load_3d(dst + b * C::BOX_BYTES, &tmK, full_k + (g % NK), C::BOX_ELEMS * b, jj * BLOCK_N, w.bh);
          }
          ++nlk;
          if (!(ok = wait_rel(g - NV))) break;
          if (leader) {
            uint8_t* dst = sV + (g % NV) * C::TILE_BYTES;
            mbar_arrive_expect_tx(full_v + (g % NV), C::TILE_BYTES);
            for (int b = 0; b < C::NBOX; ++b)
              if (dbg_tma_ok(p.dbg, DBG_LOAD_V, C::BOX_ELEMS * b, jj * BLOCK_N, w.bh, D, p.Nk, p.B * p.H, C::ESZ))
                tma_load_3d(dst + b * C::BOX_BYTES, &tmV, full_v + (g % NV), C::BOX_ELEMS * b, jj * BLOCK_N, w.bh);
          }
          ++nlv;
        }
      }
      if (!ok && leader) {
        // error path: let the copies already issued land before the CTA exits
        for (int n = max(0, nlk - NK); n < nlk; ++n) mbar_wait_drain(full_k + (n % NK), (n / NK) & 1, lim);
        for (int n = max(0, nlv - NV); n < nlv; ++n) mbar_wait_drain(full_v + (n % NV), (n / NV) & 1, lim);
      }
      dbg_count0 = nlk;
      dbg_count1 = nlv;
      __syncwarp();
    } else if (pw == 3) {
      // ------------------------------------------------------- Q TMA producer
      // Q_t of unit k goes into its buffer once unit k-1 is done with it
      // (q_free_t, phase k-1) and Q_t of unit k-1 has landed (q_full_t).
      if (leader) tma_prefetch_desc(&tmQ);
      int issued[Q_TILES] = {0, 0};
      bool ok = true;
      for (int k = 0; ok; ++k) {
        const int u = unit_at(k);
        if (u >= U) break;
        const Unit w = unit_info(p, u, kv_keep);
        for (int t = 0; t < Q_TILES && ok; ++t) {
          uint64_t* qf = q_full + C::QB * t + qbuf(k);
          if (k >= C::QB) {
            // the buffer is free (unit k - QB is done with it), and this
            // warp's previous load into it has landed (nobody else waits for
            // it when that tile had no key tile): a second expect_tx must not
            // join an unfinished phase
            ok = mbar_wait2(q_free + C::QB * t + qbuf(k), qpar(k - C::QB), qf, qpar(k - C::QB), lim, p.status,
                            abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
          }
          if (leader) {
            if (t ? w.act1 : w.act0) {
              mbar_arrive_expect_tx(qf, C::TILE_BYTES);
              // (the second tile of the last pair may start past Nq: it then
              // reads zeros and computes nothing; the pair grid bounds it)
              for (int b = 0; b < C::NBOX; ++b)
                if (dbg_tma_ok(p.dbg, DBG_LOAD_Q, C::BOX_ELEMS * b, w.pair * (Q_TILES * BLOCK_M) + t * BLOCK_M, w.bh,
                               D, p.n_qpairs * Q_TILES * BLOCK_M, p.B * p.H, C::ESZ))
                  tma_load_3d(sQ + (qbuf(k) * Q_TILES + t) * C::TILE_BYTES + b * C::BOX_BYTES, &tmQ, qf,
                              C::BOX_ELEMS * b, w.pair * (Q_TILES * BLOCK_M) + t * BLOCK_M, w.bh);
            } else {
              mbar_arrive(qf);  // a tile this unit does not compute: the phase completes empty
            }
          }
          ++issued[t];
        }
      }
      if (!ok && leader) {
        // error path: the last loads into each buffer land before the CTA exits
        for (int t = 0; t < Q_TILES; ++t)
          for (int k = max(0, issued[t] - C::QB); k < issued[t]; ++k)
            mbar_wait_drain(q_full + C::QB * t + qbuf(k), qpar(k), lim);
      }
      __syncwarp();
    } else {
      // ---------------------------------------------------------- MMA issuers
      // One warp per Q tile (tile 0 first). tcgen05.mma issue only runs about
      // one instruction ahead of the tensor pipe, so every barrier wait or
      // commit of a lone issuing warp would leave the pipe idle; with two
      // issuers each one's waits overlap the other's MMAs. With SOLO_ISSUE
      // (d = 64) lane 0 runs the loop alone and issues; otherwise the whole
      // warp runs it, votes on every wait, and the lane elect.sync picks
      // issues the MMAs and commits (ELECT_ISSUE).
      const int t = pw - 1;
      const uint32_t sQa = smem_u32(sQ) + t * C::TILE_BYTES;  // buffer 0; buffer b is b Q_TILES tiles further
      // Low descriptor words of Q_t, K slot 0 and V slot 0 (every operand
      // shares the high word: 1024-byte 8-row groups, 128-byte swizzle). The
      // K-step kk of Q and K (K-major) starts (kk / 4) boxes plus (kk % 4) x 32
      // bytes in; that of V (MN-major, 64-column boxes LBO apart) 16 rows =
      // 2048 bytes in. Another ring slot adds its offset to the low word.
      constexpr uint32_t DHI = C::DESC_HI;
      const uint32_t q_lo = sdesc_sw128_lo(sQa, 16);
      const uint32_t k_lo = sdesc_sw128_lo(smem_u32(sK), 16);
      const uint32_t v_lo = sdesc_sw128_lo(smem_u32(sV), C::BOX_BYTES);
      const uint32_t dS = tmem + BLOCK_N * t;
      const uint32_t dO = tmem + C::O_COL + D * t;
      const uint32_t aP = tmem + C::P_COL + C::P_STRIDE * t;
      const uint32_t idesc_s = C::IDESC_S | (p.negate_s ? IDESC_NEGATE_A : 0u);
      bool ok = true;
      bool issued_any = false;

      auto wait_bar = [&](uint64_t* bar, uint32_t parity) {
        ok = mbar_wait(bar, parity, lim, p.status, abort_flag);
        if (!C::SOLO_ISSUE) ok = __all_sync(0xffffffffu, ok);
        tc_fence_after();
        return ok;
      };
      // waits for up to three (barrier, parity) pairs; null barriers are skipped
      auto wait_bars = [&](uint64_t* a, uint32_t pa, uint64_t* b, uint32_t pb, uint64_t* c = nullptr,
                           uint32_t pc = 0) {
        if (a == nullptr) {
          a = b;
          pa = pb;
        }
        if (b == nullptr) {
          b = a;
          pb = pa;
        }
        ok = (a == nullptr) || mbar_wait2(a, pa, b, pb, lim, p.status, abort_flag, c, pc);
        if (!C::SOLO_ISSUE) ok = __all_sync(0xffffffffu, ok);
        tc_fence_after();
        return ok;
      };

      // The thread that issues this warp's MMAs and commits: the elected lane
      // of the converged warp (ELECT_ISSUE), else lane 0.
      auto issuer = [&]() -> bool {
        if constexpr (C::ELECT_ISSUE) return elect_one();
        else return lane == 0;
      };
      if (C::ELECT_ISSUE && FA_DEBUG && elected_lane() != 0u) dbg_fail(p.dbg, FA_DBG_PHASE, DBG_ELECT, 0, 0, 0);

      int g0 = 0;          // key tiles of earlier units (ring position)
      int c0 = 0, c1 = 0;  // steps of tile 0 / tile 1 in earlier units
      for (int k = 0; ok && (!C::SOLO_ISSUE || lane == 0); ++k) {
        const int u = unit_at(k);
        if (u >= U) break;
        const Unit w = unit_info(p, u, kv_keep);
        const int nt = t ? w.n1 : w.n0;
        const int ct = t ? c1 : c0;  // this tile's step count before the unit
        const int n_max = max(w.n0, w.n1);
        // Neither issuer starts unit k before both tiles' score MMAs of unit
        // k-1 have completed (each issuer commits to unit_done after its last
        // S of a unit, or arrives at the start when it has none): every phase
        // of the other tile's s_full before this unit is then complete, which
        // keeps the parity waits on it below unambiguous.
        if (k > 0 && !wait_bar(unit_done, (k - 1) & 1)) break;
        if (C::UNIT_DONE_EARLY && nt == 0 && lane == 0) mbar_arrive(unit_done);
        // Q_t of unit k has landed (the Q producer has passed its wait for
        // unit k-1). A tile without key tiles releases its Q buffer only after
        // that: otherwise q_free_t could run two phases ahead of the Q
        // producer's parity wait on it.
        if (!wait_bar(q_full + C::QB * t + qbuf(k), qpar(k))) break;
        if (nt == 0 && C::O_STAGE && lane == 0) mbar_arrive(q_free + C::QB * t + qbuf(k));
        // Q_t of this unit (descriptor low word)
        const uint32_t q_lo_u = q_lo + static_cast<uint32_t>((qbuf(k) * Q_TILES * C::TILE_BYTES) >> 4);

        auto fk_bar = [&](int jj) { return full_k + ((g0 + jj) % NK); };
        auto fk_par = [&](int jj) { return static_cast<uint32_t>(((g0 + jj) / NK) & 1); };
        auto fv_bar = [&](int jj) { return full_v + ((g0 + jj) % NV); };
        auto fv_par = [&](int jj) { return static_cast<uint32_t>(((g0 + jj) / NV) & 1); };
        auto issue_s = [&](int jj) {  // S_t = Q_t K_jj^T
          const uint32_t kb = k_lo + static_cast<uint32_t>((((g0 + jj) % NK) * C::TILE_BYTES) >> 4);
#pragma unroll
          for (int kk = 0; kk < C::KSTEPS_S; ++kk) {
            const uint32_t off = static_cast<uint32_t>(((kk >> 2) * C::BOX_BYTES + (kk & 3) * 32) >> 4);
            if (!dbg_tmem_mma_ok(p.dbg, DBG_MMA_S, dS, BLOCK_N, 0u, 0)) continue;
            if (issuer()) {
              if constexpr (F8) mma_ss_w_f8(dS, q_lo_u + off, DHI, kb + off, DHI, idesc_s, kk > 0 ? 1u : 0u);
              else mma_ss_w(dS, q_lo_u + off, DHI, kb + off, DHI, idesc_s, kk > 0 ? 1u : 0u);
            }
          }
          if (issuer()) mma_commit(s_full + t);
          // the unit's last score MMA: Q_t is free once it (and all before it)
          // completed, and the other issuer may start the next unit
          if (jj == nt - 1) {
            if (C::O_STAGE && issuer()) mma_commit(q_free + C::QB * t + qbuf(k));
            if (C::UNIT_DONE_EARLY && issuer()) mma_commit(unit_done);
          }
          issued_any = true;
        };
        auto issue_pv = [&](int jj) {  // O_t (+)= P_t V_jj
          const uint32_t vb = v_lo + static_cast<uint32_t>((((g0 + jj) % NV) * C::TILE_BYTES) >> 4);
#pragma unroll
          for (int kk = 0; kk < C::KSTEPS_PV; ++kk) {
            // A: 8 TMEM columns (32 bytes of P per row) per K-step; B: PV_KROWS rows of V
            const uint32_t vk = vb + static_cast<uint32_t>((kk * C::PV_KROWS * C::ROW_BYTES) >> 4);
            if (!dbg_tmem_mma_ok(p.dbg, DBG_MMA_PV, dO, D, aP + kk * 8, 8)) continue;
            if (issuer()) {
              if constexpr (F8) mma_ts_w_f8(dO, aP + kk * 8, vk, DHI, C::IDESC_O, (jj > 0 || kk > 0) ? 1u : 0u);
              else mma_ts_w(dO, aP + kk * 8, vk, DHI, C::IDESC_O, (jj > 0 || kk > 0) ? 1u : 0u);
            }
          }
          if (issuer()) mma_commit(o_done + t);
        };
        // Key tile jj is released by both issuers (rel counts 2): by a commit
        // when this warp's MMAs read it, by a plain arrive when they did not (a
        // tile past this Q tile's range). A commit from a thread with no
        // tcgen05 operation to track is not relied on to arrive. An unused tile
        // is first waited for (both loads landed), so the arrive lands in that
        // tile's phase: an idle warp must not run around the ring ahead of the
        // loads.
        auto release = [&](int jj, bool used) {
          if (!used && !wait_bars(fk_bar(jj), fk_par(jj), fv_bar(jj), fv_par(jj))) return;
          if (used) {
            if (issuer()) mma_commit(rel + ((g0 + jj) % NR));
          } else if (lane == 0) {
            mbar_arrive(rel + ((g0 + jj) % NR));
          }
        };
        // The two tiles' score MMAs alternate: the leading tile's S_j is issued
        // only after the other tile's S_{j-1} has completed, and the other
        // tile's S_j only after the leader's S_j has completed (while both
        // still have key tiles). Without this order nothing keeps the tiles
        // half a period apart, and they drift into lockstep: both score MMAs
        // share the tensor pipe at once and then both softmax warpgroups share
        // the SM's exponential units at once. The chain of waits also keeps
        // each parity wait on the other tile's s_full unambiguous (that barrier
        // is at most one phase behind or ahead). The tile with more key tiles
        // (tile 1 under a causal mask) leads, so both end close together.
        const int lead = (FA_LEAD_LONGER && w.n1 > w.n0) ? 1 : 0;
        const int n_lead = lead ? w.n1 : w.n0, n_fol = lead ? w.n0 : w.n1;
        const int c_lead = lead ? c1 : c0, c_fol = lead ? c0 : c1;
        auto order_bar = [&](int jj) -> uint64_t* {
          if (!FA_SORDER) return nullptr;
          if (t == lead) return (jj >= 1 && jj - 1 < n_fol) ? s_full + (1 - lead) : nullptr;
          return (jj < n_lead) ? s_full + lead : nullptr;
        };
        auto order_par = [&](int jj) -> uint32_t {
          return static_cast<uint32_t>((t == lead ? c_fol + jj - 1 : c_lead + jj) & 1);
        };
        // (The first PV of a unit overwrites O_t, which the previous unit's
        // epilogue read: that is implied by p_full of the unit's first step,
        // which the softmax arrives on only after that epilogue.)

        // Ping-pong: the following Q tile starts once the leader's first
        // softmax is done, so one tile's exponentials overlap the other tile's
        // MMAs instead of both tiles competing for the same unit at once. Not
        // under a causal mask, where the two tiles' key ranges differ and the
        // delayed start measured slower.
        if (C::STAGGER && !p.causal && t != lead && n_lead >= FA_STAGGER_MIN_TILES && nt > 0 &&
            !wait_bar(p_full + lead, c_lead & 1))
          break;

        if (C::SEP_P) {
          // Software pipeline: S_{j+1} is issued as soon as the softmax has
          // read S_j (s_free), so the next scores are computed while it
          // exponentiates. The first S of a unit needs the last S of the
          // previous one read.
          if (nt > 0) {
            if (!wait_bars(fk_bar(0), fk_par(0), ct > 0 ? s_free + t : nullptr,
                           static_cast<uint32_t>((ct - 1) & 1), order_bar(0), order_par(0)))
              break;
            issue_s(0);
          }
          for (int jj = 0; ok && jj < n_max; ++jj) {
            if (jj + 1 < nt) {
              if (!wait_bars(fk_bar(jj + 1), fk_par(jj + 1), s_free + t, static_cast<uint32_t>((ct + jj) & 1),
                             order_bar(jj + 1), order_par(jj + 1)))
                break;
              issue_s(jj + 1);
            }
            if (jj < nt) {
              if (!wait_bars(p_full + t, static_cast<uint32_t>((ct + jj) & 1), fv_bar(jj), fv_par(jj))) break;
              issue_pv(jj);
            }
            release(jj, jj < nt);
          }
        } else {
          // P aliases S in TMEM: S_{t,j} may only be written after PV_{t,j-1}
          // (which reads P_{t,j-1} from the same columns) has completed; across
          // units that is the previous unit's last PV.
          for (int jj = 0; ok && jj < n_max; ++jj) {
            if (jj < nt) {
              if (!wait_bars(fk_bar(jj), fk_par(jj), (ct + jj > 0) ? o_done + t : nullptr,
                             static_cast<uint32_t>((ct + jj - 1) & 1), order_bar(jj), order_par(jj)))
                break;
              issue_s(jj);
              if (!wait_bars(p_full + t, static_cast<uint32_t>((ct + jj) & 1), fv_bar(jj), fv_par(jj))) break;
              issue_pv(jj);
            }
            release(jj, jj < nt);
          }
        }
        if (!ok) break;
        if (!C::UNIT_DONE_EARLY && lane == 0) mbar_arrive(unit_done);
        g0 += n_max;
        c0 += w.n0;
        c1 += w.n1;
      }
      // every MMA both issuers issued must finish before TMEM is released
      if (!C::SOLO_ISSUE) __syncwarp();
      if (issued_any) {
        if (issuer()) mma_commit(drain);
      } else if (lane == 0) {
        mbar_arrive(drain);
      }
      if (lane == 0) mbar_wait_drain(drain, 0, lim);
      __syncwarp();
    }
  } else {
    setmaxnreg_inc<prefill_softmax_regs(D)>();
    // ------------------------------------------------- softmax / correction
    const int t = sw >> 2;
    const int wq = sw & 3;  // = warp % 4: the TMEM lane quarter this warp may access
    const int row = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + BLOCK_N * t;
    const uint32_t tO = tmem + lane_base + C::O_COL + D * t;
    const uint32_t tP = tmem + lane_base + C::P_COL + C::P_STRIDE * t;
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = f2pack(sl2, sl2);
    const int delta = p.Nk - p.Nq;
    const int nwords = (p.Nk + 31) >> 5;
    uint8_t* sO = C::O_STAGE ? smem + C::O_OFF + t * C::O_TILE_BYTES : sQ + t * C::TILE_BYTES;
    const bool storer = wq == 0 && lane == 0;
    bool ok = true;
    int ct = 0;  // this tile's steps in earlier units

    // Every thread of the tile walks every unit and reaches the epilogue's
    // named barrier once per unit, on the error path too (work is skipped,
    // barriers are not).
    for (int k = 0;; ++k) {
      const int u = unit_at(k);
      if (u >= U) break;
      const Unit w = unit_info(p, u, kv_keep);
      const int bh = w.bh;
      const int n = t ? w.n1 : w.n0;
      const bool active = t ? w.act1 : w.act0;  // else another unit computes these rows
      const int r0 = w.pair * (Q_TILES * BLOCK_M) + t * BLOCK_M;
      const int qi = r0 + row;
      const int diag = qi + delta;      // last key this row may see (causal)
      const int tile_lim = r0 + delta;  // last key the first row of the tile may see
      const uint32_t* krow = nullptr;
      if (p.keep != nullptr && qi < p.Nq) {
        const int b = bh / p.H, h = bh % p.H;
        krow = p.keep + b * p.msb + h * p.msh + static_cast<int64_t>(qi) * p.msq;
      }
      float m = -INFINITY;  // running max (possibly stale, see below), log2 units of the scaled score
      float l = 0.f;        // running sum of exponentials on the base m

      // Barrier polls are issued early and their results used late: s_full of
      // the next key tile right after P is stored, o_done of the previous PV
      // halfway through the exponentials. A poll that finds the phase
      // incomplete falls back to the bounded wait.
      uint32_t s_ready = 0;
      for (int j = 0; ok && j < n; ++j) {
        const uint32_t ph = static_cast<uint32_t>((ct + j) & 1);  // this step's phase parity
        if (!__all_sync(0xffffffffu, s_ready)) {
          ok = mbar_wait(s_full + t, ph, lim, p.status, abort_flag);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
        }
        tc_fence_after();
        uint32_t s[BLOCK_N];
        if (FA_DEBUG && !dbg_tmem_warp_ok(p.dbg, DBG_LD_S, tS, BLOCK_N)) {
          for (int c = 0; c < BLOCK_N; ++c) s[c] = 0u;  // the load is skipped
        } else {
          tmem_ld32(tS + 0, s);
          tmem_ld32(tS + 32, s + 32);
          tmem_ld32(tS + 64, s + 64);
          tmem_ld32(tS + 96, s + 96);
        }
        tmem_ld_wait32(s);
        reg_fence32(s + 32);
        reg_fence32(s + 64);
        reg_fence32(s + 96);
        if (C::SEP_P) {  // S_t may be overwritten with the next tile's scores
          tc_fence_before();
          mbar_arrive(s_free + t);
        }

        const int kbase = j * BLOCK_N;
        uint32_t kw[4] = {0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu};
        bool keep_all = true;
        if (krow != nullptr) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int wi = (kbase >> 5) + q;
            kw[q] = wi < nwords ? __ldg(krow + wi) : 0u;
          }
          keep_all = (kw[0] & kw[1] & kw[2] & kw[3]) == 0xffffffffu;
        }
        // tiles whose 128 keys are all kept for every row of the warp skip the
        // element-wise mask (warp-uniform choice of code path)
        const bool all_kept = __all_sync(0xffffffffu, keep_all) != 0;
        const bool need_mask = (kbase + BLOCK_N > p.Nk) || (p.causal && kbase + BLOCK_N - 1 > tile_lim) || !all_kept;
        if (need_mask) {
          if (all_kept) {
            // every key of the tile kept: keys past min(Nk - 1, diag) are
            // hidden, a threshold (much cheaper than testing mask bits)
            const int lim = min(p.causal ? diag : INT_MAX, p.Nk - 1) - kbase;  // last visible column
#pragma unroll
            for (int c = 0; c < BLOCK_N; ++c)
              if (c > lim) s[c] = f2u(-INFINITY);
          } else {
#pragma unroll
            for (int c = 0; c < BLOCK_N; ++c) {
              const int key = kbase + c;
              bool vis = key < p.Nk;
              if (p.causal) vis = vis && key <= diag;
              vis = vis && ((kw[c >> 5] >> (c & 31)) & 1u);
              if (!vis) s[c] = f2u(-INFINITY);
            }
          }
        }
        // row max: 8 independent chains of three-input maxima, then a short tree
        float mxa[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) {
          float v = u2f(s[a * 16]);
#pragma unroll
          for (int e = 1; e + 1 < 16; e += 2) v = fmax3(v, u2f(s[a * 16 + e]), u2f(s[a * 16 + e + 1]));
          mxa[a] = fmaxf(v, u2f(s[a * 16 + 15]));
        }
        const float mx =
            fmaxf(fmax3(mxa[0], mxa[1], mxa[2]), fmax3(fmax3(mxa[3], mxa[4], mxa[5]), mxa[6], mxa[7]));
        const float m_tile = (mx == -INFINITY) ? -INFINITY : mx * sl2;
        // Lazy rescale: keep the running base m unless this tile's max exceeds it
        // by more than RESCALE_LOG2; exponentials are then at most 2^RESCALE_LOG2,
        // and l and O share the same (stale) base, so o / l is unchanged.
        const bool bump = m_tile > m + C::RESCALE_LOG2;
        const float m_new = bump ? m_tile : m;
        const float alpha = bump ? ex2_approx(m - m_new) : 1.f;  // 0 while nothing was accumulated
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const uint64_t nm2 = f2pack(-m_use, -m_use);
        uint32_t o_ready = 0;
        const uint32_t o_poll = (C::SEP_P && j > 0) ? smem_u32(o_done + t) : 0u;
        const uint32_t o_par = ph ^ 1u;  // the previous step's phase
        // (with no FMA-pipe pairs both instantiations are the same code: keep
        // one copy of the unrolled loop in the instruction cache)
        const float rowsum = (C::EMU_PAIRS > 0 && need_mask)
                                 ? softmax_tile_p<true, C::EMU_PAIRS, F8>(s, sl2x2, nm2, o_poll, o_par, &o_ready)
                                 : softmax_tile_p<false, C::EMU_PAIRS, F8>(s, sl2x2, nm2, o_poll, o_par, &o_ready);
        if (C::SEP_P && j > 0) {
          // P_t and O_t are free once PV_{t,j-1} has completed; it ran while
          // the exponentials above were computed. (At a unit's first step the
          // previous unit's epilogue already waited for its last PV.)
          if (!__all_sync(0xffffffffu, o_ready)) {
            ok = mbar_wait(o_done + t, o_par, lim, p.status, abort_flag);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
          }
          tc_fence_after();
        }
        if (dbg_tmem_warp_ok(p.dbg, DBG_ST_P, tP, C::P_WORDS)) {
          tmem_st32(tP, s);  // P: the packed words now in s[0 .. P_WORDS)
          if constexpr (C::P_WORDS > 32) tmem_st32(tP + 32, s + 32);
        }
        s_ready = (FA_EARLY_POLL && j + 1 < n) ? mbar_test(smem_u32(s_full + t), ph ^ 1u) : 0u;
        l = fmaf(l, alpha, rowsum);
        // O_t is quiescent here: PV_{t,j-1} has completed (waited above, or before
        // S_{t,j} was issued) and PV_{t,j} waits for p_full.
        if (j > 0 && __any_sync(0xffffffffu, bump)) {
          const uint64_t al2 = f2pack(alpha, alpha);
#pragma unroll
          for (int ch = 0; ch < D / 32; ++ch) {
            if (!dbg_tmem_warp_ok(p.dbg, DBG_ST_O, tO + ch * 32, 32)) continue;
            uint32_t o[32];
            tmem_ld32(tO + ch * 32, o);
            tmem_ld_wait32(o);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float y0, y1;
              f2unpack(fmul2(f2pack(u2f(o[2 * i]), u2f(o[2 * i + 1])), al2), y0, y1);
              o[2 * i] = f2u(y0);
              o[2 * i + 1] = f2u(y1);
            }
            tmem_st32(tO + ch * 32, o);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(p_full + t);
        m = m_new;
      }

      // ---- epilogue: O = o / l (0 for an empty row), lse = m + ln l (-inf for an empty row)
      // O goes through shared memory into one TMA store per 64-column box. The
      // staging buffer is this tile's Q tile: every S MMA that read it has
      // completed once the last PV has (the issuer's commit covers all its
      // earlier MMAs); a tile with no key tile ran no MMA, so there the Q load
      // itself is waited for. Rows are written in the 128-byte-swizzled layout
      // the tensor map expects; rows past Nq are clipped by the store. Once the
      // store has read the buffer (q_free) the next Q may be loaded into it.
      // With separate O staging the previous unit's store must have read the
      // buffer before it is rewritten: the storer waits for that here, where
      // the store has long finished, rather than right after issuing it,
      // where the wait would delay its warp's first softmax step of the next
      // unit.
      if (C::O_STAGE && FA_LATE_STORE_WAIT) {
        if (storer) bulk_wait_group_read_all();
        named_bar_sync(1 + t, 128);
      }
      if (ok && active && (n > 0 || !C::O_STAGE)) {
        ok = (n > 0) ? mbar_wait(o_done + t, static_cast<uint32_t>((ct + n - 1) & 1), lim, p.status, abort_flag)
                     : mbar_wait(q_full + C::QB * t + qbuf(k), qpar(k), lim, p.status, abort_flag);
        ok = __all_sync(0xffffffffu, ok);
        tc_fence_after();
      }
      // a separate staging buffer is rewritten only after the previous unit's
      // store has read it (the storer waited for that before this barrier)
      if (C::O_STAGE && k > 0) named_bar_sync(1 + t, 128);
      if (ok && active) {
        const float inv = (l > 0.f) ? p.o_scale / l : 0.f;  // o_scale: the v descale (1 for bf16)
        const uint32_t srow = smem_u32(sO) + static_cast<uint32_t>(row) * 128u;
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t o[32];
          if (n > 0 && dbg_tmem_warp_ok(p.dbg, DBG_LD_O, tO + ch * 32, 32)) {
            tmem_ld32(tO + ch * 32, o);
            tmem_ld_wait32(o);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = 0u;
          }
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(u2f(o[2 * i]) * inv, u2f(o[2 * i + 1]) * inv);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const int c = ch * 4 + v;  // 16-byte chunk of the row: box c / 8, chunk c % 8 of the box
            const uint32_t a = srow + static_cast<uint32_t>((c >> 3) * C::O_BOX_BYTES) +
                               (static_cast<uint32_t>((c & 7) ^ (row & 7)) << 4);
            st_shared_v4(a, pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
        if (p.lse != nullptr && qi < p.Nq)
          p.lse[static_cast<size_t>(bh) * p.Nq + qi] =
              (l > 0.f) ? (m + lg2_approx(l)) * 0.69314718055994530942f : -INFINITY;
      }
      fence_proxy_async_smem();
      named_bar_sync(1 + t, 128);  // every thread of the tile, every unit, on every path
      if (storer && *abort_flag == 0) {
        if (active && r0 < p.Nq) {
#pragma unroll
          for (int b = 0; b < C::NBOX_O; ++b)
            if (dbg_tma_ok(p.dbg, DBG_STORE_O, 64 * b, r0, bh, D, p.Nq, p.B * p.H, 2))
              tma_store_3d(&tmO, sO + b * C::O_BOX_BYTES, 64 * b, r0, bh);
          bulk_commit_group();
          if (!(C::O_STAGE && FA_LATE_STORE_WAIT)) bulk_wait_group_read_all();
        }
        if (!C::O_STAGE) mbar_arrive(q_free + C::QB * t + qbuf(k));
      }
      ct += n;
    }
    if (storer) bulk_wait_group_all();  // the last stores are complete before the CTA exits
    dbg_count0 = ct;
  }

  tc_fence_before();
  __syncthreads();
  if (FA_DEBUG && *abort_flag == 0 && lane == 0) {
    // every barrier has completed as many phases as its users counted
    if (!producer && (sw & 3) == 0) {
      const int t = sw >> 2;
      dbg_phase_check(p.dbg, DBG_PHASE_S, smem_u32(s_full + t), dbg_count0, t);
      dbg_phase_check(p.dbg, DBG_PHASE_P, smem_u32(p_full + t), dbg_count0, t);
      dbg_phase_check(p.dbg, DBG_PHASE_O, smem_u32(o_done + t), dbg_count0, t);
      if (C::SEP_P) dbg_phase_check(p.dbg, DBG_PHASE_SFREE, smem_u32(s_free + t), dbg_count0, t);
    } else if (producer && pw == 0) {
      for (int i = 0; i < NK; ++i)
        dbg_phase_check(p.dbg, DBG_PHASE_K, smem_u32(full_k + i), dbg_count0 > i ? (dbg_count0 - i + NK - 1) / NK : 0, i);
      for (int i = 0; i < NV; ++i)
        dbg_phase_check(p.dbg, DBG_PHASE_V, smem_u32(full_v + i), dbg_count1 > i ? (dbg_count1 - i + NV - 1) / NV : 0, i);
    }
  }
  if (alloc_warp) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// Runs every debug check once on values it must reject (a misaligned TMA x
// coordinate, another warp's TMEM lanes, columns past the allocation, a
// barrier whose phase count disagrees), performing no access at all. In a
// debug build each check must set its bit; in a release build the checks are
// compiled out and the record stays clear.
__global__ void fa_debug_selftest_kernel(unsigned int* rec) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;  // lane 0 of warp 0: TMEM lane quarter 0
  (void)dbg_tma_ok(rec, DBG_SELFTEST, 8, 0, 0, 64, 128, 1, 1);           // x = 8 one-byte codes: off 16 bytes
  (void)dbg_tmem_warp_ok(rec, DBG_SELFTEST, 32u << 16, 32);              // lanes 32..63 from warp 0
  (void)dbg_tmem_mma_ok(rec, DBG_SELFTEST, 480u, 64, 0u, 0);             // columns 480..543
  mbar_init(&bar, 1);
  fence_mbar_init();
  mbar_arrive(&bar);                                                     // one phase completed ...
  dbg_phase_check(rec, DBG_SELFTEST, smem_u32(&bar), 2, 0);              // ... where two were counted
}

cudaError_t launch_debug_selftest(unsigned int* rec, cudaStream_t stream) {
  fa_debug_selftest_kernel<<<1, 32, 0, stream>>>(rec);
  return cudaGetLastError();
}

template <int D, bool F8>
static cudaError_t launch_prefill_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                    const CUtensorMap& to, const PrefillParams& p, cudaStream_t stream) {
  // Persistent: one CTA per SM walks its share of the units, so the next
  // unit's loads and first MMAs overlap the current one's epilogue. A key
  // mask broadcast over rows (trimmed per unit) gets one CTA per unit, as does
  // a head dimension where that measured faster.
  using C = PrefillCfg<D, F8>;
  const long long units = p.units;
  const bool trim = p.keep != nullptr && p.msq == 0;
  const long long ctas = (trim || !C::PERSIST) ? units : std::min<long long>(units, std::max(1, p.max_ctas));
  fa_prefill_kernel<D, F8><<<static_cast<unsigned>(ctas), prefill_threads(D), C::SMEM, stream>>>(tq, tk, tv, to, p);
  return cudaGetLastError();
}

// The instantiations: bf16 and e4m3, each at d = 64 and 128.
template <int D, bool F8>
static int num_regs_t() {
  cudaFuncAttributes a{};
  return cudaFuncGetAttributes(&a, fa_prefill_kernel<D, F8>) == cudaSuccess ? a.numRegs : -1;
}
int prefill_num_regs(int d, bool f8) {
  if (f8) return d == 64 ? num_regs_t<64, true>() : num_regs_t<128, true>();
  return d == 64 ? num_regs_t<64, false>() : num_regs_t<128, false>();
}

size_t prefill_smem_bytes(int d, bool f8) {
  if (f8) return d == 64 ? PrefillCfg<64, true>::SMEM : PrefillCfg<128, true>::SMEM;
  return d == 64 ? PrefillCfg<64>::SMEM : PrefillCfg<128>::SMEM;
}

template <int D, bool F8>
static cudaError_t set_attributes_t() {
  return cudaFuncSetAttribute(fa_prefill_kernel<D, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              PrefillCfg<D, F8>::SMEM);
}
cudaError_t prefill_set_attributes(int d, bool f8) {
  if (f8) return d == 64 ? set_attributes_t<64, true>() : set_attributes_t<128, true>();
  return d == 64 ? set_attributes_t<64, false>() : set_attributes_t<128, false>();
}

cudaError_t launch_prefill(int d, bool f8, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& to, const PrefillParams& p, cudaStream_t stream) {
  if (f8)
    return d == 64 ? launch_prefill_t<64, true>(tq, tk, tv, to, p, stream)
                   : launch_prefill_t<128, true>(tq, tk, tv, to, p, stream);
  return d == 64 ? launch_prefill_t<64, false>(tq, tk, tv, to, p, stream)
                 : launch_prefill_t<128, false>(tq, tk, tv, to, p, stream);
}

}  // namespace fa
