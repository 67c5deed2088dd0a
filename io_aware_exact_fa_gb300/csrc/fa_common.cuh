// Definitions shared by the kernels and the host side of the C-ABI library.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

// Set the calling thread's error detail string (fa_last_error_detail).
void fa_set_error_detail(const char* fmt, ...);

namespace fa {

// Bits of the device status word (one word per device, cleared by
// fa_get_device_status).
constexpr unsigned int FA_DEV_TIMEOUT = 1u;   // a bounded wait ran out

// Device ordinals the host side keeps per-device state for (0 .. kMaxDevices-1).
constexpr int kMaxDevices = 64;

// Prefill tiling: 128 query rows per Q tile, two Q tiles per CTA, 128 keys per
// K/V tile.
constexpr int BLOCK_M = 128;
constexpr int BLOCK_N = 128;
constexpr int Q_TILES = 2;
constexpr int PREFILL_THREADS = 384;       // 2 softmax warpgroups + 1 producer warpgroup
constexpr int PREFILL_SOFTMAX_WARPS = 8;   // warps 0-3: Q tile 0, warps 4-7: Q tile 1; 8-11 producers
// Register split after set-up (setmaxnreg): the launch gives every thread
// PREFILL_LAUNCH_REGS; each SM sub-partition holds one warp of every
// warpgroup, so 2 * SOFTMAX + PRODUCER must not exceed 3 * PREFILL_LAUNCH_REGS.
constexpr int PREFILL_LAUNCH_REGS = 168;
#ifndef FA_SOFTMAX_REGS_D64
#define FA_SOFTMAX_REGS_D64 216
#endif
#ifndef FA_SOFTMAX_REGS_D128
#define FA_SOFTMAX_REGS_D128 216
#endif
// registers of the softmax warpgroups and of the producer/MMA warpgroup after
// setmaxnreg, per head dimension (the d = 128 MMA issuers keep more state)
__host__ __device__ constexpr int prefill_softmax_regs(int d) {
  return d == 64 ? FA_SOFTMAX_REGS_D64 : FA_SOFTMAX_REGS_D128;
}
__host__ __device__ constexpr int prefill_producer_regs(int d) {
  return 3 * PREFILL_LAUNCH_REGS - 2 * prefill_softmax_regs(d) < 256 ? 3 * PREFILL_LAUNCH_REGS - 2 * prefill_softmax_regs(d)
                                                                      : 256;
}
static_assert(2 * prefill_softmax_regs(64) + prefill_producer_regs(64) <= 3 * PREFILL_LAUNCH_REGS &&
                  2 * prefill_softmax_regs(128) + prefill_producer_regs(128) <= 3 * PREFILL_LAUNCH_REGS,
              "setmaxnreg split exceeds the launch allocation");
static_assert(prefill_softmax_regs(64) % 8 == 0 && prefill_softmax_regs(128) % 8 == 0 &&
                  prefill_producer_regs(64) % 8 == 0 && prefill_producer_regs(128) % 8 == 0 &&
                  prefill_producer_regs(64) >= 24 && prefill_producer_regs(128) >= 24,
              "setmaxnreg counts are multiples of 8 in [24, 256]");

struct PrefillParams {
  void* o;                   // bf16 [B*H, Nq, d]
  float* lse;                // fp32 [B*H, Nq] or nullptr
  const uint32_t* keep;      // packed key mask or nullptr
  int64_t msb, msh, msq;     // mask strides in 32-bit words
  int B, H, Nq, Nk;
  int n_qpairs;              // ceil(Nq / 256)
  int causal;
  float scale_log2;          // |scale| * log2(e)
  int negate_s;              // scale < 0: the score MMA computes -(Q K^T)
  uint64_t wait_limit_ns;
  unsigned int* status;      // device status word
  int max_ctas;              // CTAs of a persistent launch (the SM count)
  int units;                 // work units: Q-tile pairs, then single Q tiles (see split_from)
  int split_from;            // units from here on are single tiles of the last pairs
};

struct BwdParams {
  float* dq_acc;             // fp32 workspace: dQ / scale, accumulated, tiled as
                             // [B*H][ceil(Nq/128)][d/4][128 rows][4] (one 4-column
                             // chunk of a 128-row Q tile is 2 KB contiguous)
  float* lse2;               // fp32 [B*H, Nq] workspace: lse * log2(e) (+inf for an empty row)
  float* drow;               // fp32 [B*H, Nq] workspace: sum_c dO * O per row
  void* dk;                  // bf16 [B*H, Nk, d]
  void* dv;                  // bf16 [B*H, Nk, d]
  int B, H, Nq, Nk;
  int causal;
  float scale;               // softmax scale
  float scale_log2;          // scale * log2(e)
  uint64_t wait_limit_ns;
  unsigned int* status;      // device status word
};

struct DecodeParams {
  const void* q;             // bf16 [B*H, d]
  const void* k;             // bf16 [B*H, Nk, d]
  const void* v;             // bf16 [B*H, Nk, d]
  void* o;                   // bf16 [B*H, d]
  float* lse;                // fp32 [B*H] or nullptr
  float* ws_o;               // fp32 [B*H, S, d]   unnormalised partial outputs
  float* ws_ml;              // fp32 [B*H, S, 2]   partial (max in log2 units, sum)
  int BH, Nk, S, chunk;
  float scale_log2;
};

// Launchers (defined next to their kernels). Return a CUDA error code.
cudaError_t launch_prefill(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& to, const PrefillParams& p, cudaStream_t stream);
size_t prefill_smem_bytes(int d);
cudaError_t prefill_set_attributes(int d);
int prefill_num_regs(int d);   // registers per thread the prefill kernel launches with
cudaError_t launch_decode(int d, const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_bwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const BwdParams& p, const void* o, const void* dout, const float* lse,
                       void* dq, cudaStream_t stream);
cudaError_t bwd_set_attributes(int d);
cudaError_t launch_wait_selftest(uint64_t limit_ns, unsigned int* status, cudaStream_t stream);
cudaError_t launch_exp2_selftest(const float* x, float* y, int n, cudaStream_t stream);

}  // namespace fa
