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
constexpr int PREFILL_SOFTMAX_WARPS = 8;   // warps 0-3: Q tile 0, warps 4-7: Q tile 1; then the producers
// Two softmax warpgroups and one producer warpgroup (K/V TMA, two MMA
// issuers, Q TMA) at both head dimensions.
__host__ __device__ constexpr int prefill_warpgroups(int) { return 3; }
__host__ __device__ constexpr int prefill_threads(int d) { return 128 * prefill_warpgroups(d); }
// Register split after set-up (setmaxnreg): the launch gives every thread
// prefill_launch_regs(d) (the whole register file over the CTA's threads);
// each SM sub-partition holds one warp of every warpgroup, so
// 2 * SOFTMAX + (warpgroups - 2) * PRODUCER must not exceed
// warpgroups * LAUNCH.
__host__ __device__ constexpr int prefill_launch_regs(int d) { return prefill_warpgroups(d) == 4 ? 128 : 168; }
#ifndef FA_SOFTMAX_REGS_D64
#define FA_SOFTMAX_REGS_D64 216
#endif
#ifndef FA_SOFTMAX_REGS_D128
#define FA_SOFTMAX_REGS_D128 216
#endif
// registers of the softmax warpgroups and of the producer warpgroups after
// setmaxnreg, per head dimension
__host__ __device__ constexpr int prefill_softmax_regs(int d) {
  return d == 64 ? FA_SOFTMAX_REGS_D64 : FA_SOFTMAX_REGS_D128;
}
__host__ __device__ constexpr int prefill_producer_regs(int d) {
  return (prefill_warpgroups(d) * prefill_launch_regs(d) - 2 * prefill_softmax_regs(d)) / (prefill_warpgroups(d) - 2) /
                     8 * 8 < 256
             ? (prefill_warpgroups(d) * prefill_launch_regs(d) - 2 * prefill_softmax_regs(d)) /
                   (prefill_warpgroups(d) - 2) / 8 * 8
             : 256;
}
static_assert(2 * prefill_softmax_regs(64) + (prefill_warpgroups(64) - 2) * prefill_producer_regs(64) <=
                      prefill_warpgroups(64) * prefill_launch_regs(64) &&
                  2 * prefill_softmax_regs(128) + (prefill_warpgroups(128) - 2) * prefill_producer_regs(128) <=
                      prefill_warpgroups(128) * prefill_launch_regs(128),
              "setmaxnreg split exceeds the launch allocation");
static_assert(prefill_softmax_regs(64) % 8 == 0 && prefill_softmax_regs(128) % 8 == 0 &&
                  prefill_producer_regs(64) >= 24 && prefill_producer_regs(128) >= 24 &&
                  prefill_softmax_regs(64) >= prefill_launch_regs(64) &&
                  prefill_softmax_regs(128) >= prefill_launch_regs(128) &&
                  prefill_producer_regs(64) <= prefill_launch_regs(64) &&
                  prefill_producer_regs(128) <= prefill_launch_regs(128),
              "setmaxnreg counts are multiples of 8 in [24, 256], softmax up and producers down");

struct PrefillParams {
  void* o;                   // bf16 [B*H, Nq, d]
  float* lse;                // fp32 [B*H, Nq] or nullptr
  const uint32_t* keep;      // packed key mask or nullptr
  int64_t msb, msh, msq;     // mask strides in 32-bit words
  int B, H, Nq, Nk;
  int n_qpairs;              // ceil(Nq / 256)
  int causal;
  float scale_log2;          // |scale| * log2(e) (e4m3 inputs: times the q and k descales)
  int negate_s;              // scale < 0: the score MMA computes -(Q K^T)
  float o_scale;             // multiplies O / l: the v descale of e4m3 inputs, else 1
  uint64_t wait_limit_ns;
  unsigned int* status;      // device status word
  int max_ctas;              // CTAs of a persistent launch (the SM count)
  int units;                 // work units: Q-tile pairs, then single Q tiles (see split_from)
  unsigned int* dbg;         // debug build: the device check record (FA_DBG_WORDS words); else nullptr
  int split_from;            // units from here on are single tiles of the last pairs
  int band;                  // causal unit order: 0 = pair-major over all heads; else bands of `band`
                             // pair lengths (longest first), each band walked head by head
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
// f8: the e4m3-input instantiation (d = 128 only); otherwise bf16 inputs.
cudaError_t launch_prefill(int d, bool f8, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& to, const PrefillParams& p, cudaStream_t stream);
size_t prefill_smem_bytes(int d, bool f8);
cudaError_t prefill_set_attributes(int d, bool f8);
int prefill_num_regs(int d, bool f8);   // registers per thread the prefill kernel launches with
cudaError_t launch_decode(int d, const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_bwd(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const BwdParams& p, const void* o, const void* dout, const float* lse,
                       void* dq, cudaStream_t stream);
cudaError_t bwd_set_attributes(int d);
cudaError_t launch_wait_selftest(uint64_t limit_ns, unsigned int* status, cudaStream_t stream);
cudaError_t launch_exp2_selftest(const float* x, float* y, int n, cudaStream_t stream);
cudaError_t launch_debug_selftest(unsigned int* rec, cudaStream_t stream);

}  // namespace fa
