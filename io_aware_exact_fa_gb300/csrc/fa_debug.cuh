// Device-side checks of the debug build (FA_DEBUG=1): tile coordinates of
// every TMA copy, the TMEM lanes and columns of every tensor-memory access and
// product, and the barrier phase counts at the end of a launch. A failed check
// sets a bit in a device record, keeps the first failure's site and values,
// and skips the access it guards; nothing traps. The release build compiles
// every check away.
#pragma once

#include <cstdint>

#ifndef FA_DEBUG
#define FA_DEBUG 0
#endif

namespace fa {

// Bits of the debug record's word 0.
constexpr unsigned int FA_DBG_TMA = 1u;     // a TMA coordinate out of range or misaligned
constexpr unsigned int FA_DBG_TMEM = 2u;    // a TMEM lane or column range outside the warp's part / the allocation
constexpr unsigned int FA_DBG_PHASE = 4u;   // a barrier's completed-phase count disagrees with its expected count
// Record layout (8 words): bits, site, block, thread, value 0, value 1, value 2, failures counted.
constexpr int FA_DBG_WORDS = 8;

// Sites (word 1 of the record): which access failed.
enum DbgSite : int {
  DBG_LOAD_Q = 1, DBG_LOAD_K, DBG_LOAD_V, DBG_STORE_O, DBG_MMA_S, DBG_MMA_PV, DBG_LD_S, DBG_ST_P, DBG_LD_O,
  DBG_ST_O, DBG_PHASE_S, DBG_PHASE_P, DBG_PHASE_O, DBG_PHASE_SFREE, DBG_PHASE_K, DBG_PHASE_V, DBG_ELECT, DBG_SELFTEST = 99
};

__device__ __forceinline__ void dbg_fail(unsigned int* rec, unsigned int bit, int site, int v0, int v1, int v2) {
  if (rec == nullptr) return;
  atomicAdd(rec + 7, 1u);
  if (atomicOr(rec, bit) == 0u) {  // the first failure keeps its site
    rec[1] = static_cast<unsigned int>(site);
    rec[2] = blockIdx.x;
    rec[3] = threadIdx.x;
    rec[4] = static_cast<unsigned int>(v0);
    rec[5] = static_cast<unsigned int>(v1);
    rec[6] = static_cast<unsigned int>(v2);
  }
}

// TMA tile at (x, y, z) of a [Z, Y, X] tensor whose boxes are box_x elements
// wide: x must start on a 16-byte boundary and inside the row, the tile must
// start inside the tensor (rows past Y read as zero, but a tile that starts
// past Y is never meant), z inside [0, Z). Returns whether the copy may go.
__device__ __forceinline__ bool dbg_tma_ok(unsigned int* rec, int site, int x, int y, int z, int X, int Y, int Z,
                                           int esz) {
  if (!FA_DEBUG) return true;
  const bool ok = x >= 0 && x < X && (x * esz) % 16 == 0 && y >= 0 && y < Y && z >= 0 && z < Z;
  if (!ok) dbg_fail(rec, FA_DBG_TMA, site, x, y, z);
  return ok;
}

// A warp's tcgen05.ld/st at taddr covering `cols` columns: the lane field
// must be the warp's own quarter (32 * (warp % 4)) and the columns inside the
// 512 allocated (the allocation starts at column 0).
__device__ __forceinline__ bool dbg_tmem_warp_ok(unsigned int* rec, int site, uint32_t taddr, int cols) {
  if (!FA_DEBUG) return true;
  const uint32_t lane = taddr >> 16, col = taddr & 0xFFFFu;
  const uint32_t want = 32u * ((threadIdx.x >> 5) & 3u);
  const bool ok = lane == want && col + static_cast<uint32_t>(cols) <= 512u;
  if (!ok) dbg_fail(rec, FA_DBG_TMEM, site, static_cast<int>(lane), static_cast<int>(col), cols);
  return ok;
}

// A product's accumulator (N columns from d_col) and, when a_cols > 0, its
// TMEM A operand (a_cols columns from a_col): lane 0, inside the allocation.
__device__ __forceinline__ bool dbg_tmem_mma_ok(unsigned int* rec, int site, uint32_t d_taddr, int n,
                                                uint32_t a_taddr, int a_cols) {
  if (!FA_DEBUG) return true;
  bool ok = (d_taddr >> 16) == 0u && (d_taddr & 0xFFFFu) + static_cast<uint32_t>(n) <= 512u;
  if (a_cols > 0) ok = ok && (a_taddr >> 16) == 0u && (a_taddr & 0xFFFFu) + static_cast<uint32_t>(a_cols) <= 512u;
  if (!ok) dbg_fail(rec, FA_DBG_TMEM, site, static_cast<int>(d_taddr & 0xFFFFu), n, static_cast<int>(a_taddr));
  return ok;
}

// At the end of a launch: the barrier at shared address `bar` must have
// completed exactly `phases` phases, as far as its parity shows (the last one
// complete, the next one not).
__device__ __forceinline__ void dbg_phase_check(unsigned int* rec, int site, uint32_t bar, int phases, int idx) {
  if (!FA_DEBUG) return;
  uint32_t last_done = 1u, next_done = 0u;
  {
    uint32_t r;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}" : "=r"(r) : "r"(bar), "r"(static_cast<uint32_t>(phases & 1)) : "memory");
    next_done = r;
    if (phases > 0) {
      asm volatile("{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                   "selp.u32 %0, 1, 0, p;\n\t}" : "=r"(r) : "r"(bar), "r"(static_cast<uint32_t>((phases - 1) & 1))
                   : "memory");
      last_done = r;
    }
  }
  if (!last_done || next_done) dbg_fail(rec, FA_DBG_PHASE, site, phases, idx, static_cast<int>(last_done * 2 + next_done));
}

}  // namespace fa
