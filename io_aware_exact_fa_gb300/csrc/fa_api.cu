// Host side of the C ABI declared in include/fa.h: argument validation,
// TMA descriptor encoding, launch configuration and the device status word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "fa.h"
#include <cublas_v2.h>
#include <dlfcn.h>

#include "decode_grouped.cuh"
#include "materialized.cuh"
#include "fa_common.cuh"
#include "fa_debug.cuh"

// Causal unit order for K/V larger than L2 (see below): off by default. With a
// 40 MB budget the long-context launches read 1.3x their Q+K+V from DRAM
// instead of 2.7x (B=1 H=32 N=8192 d=128: 268 against 545 MB) but ran 6 %
// slower (1,166 against 1,243 TFLOP/s; 32k: 1,293 against 1,364): the
// pair-major order over all heads is faster, and DRAM runs at 17 % of its
// bandwidth there.
#ifndef FA_PREFILL_L2_BUDGET_MB
#define FA_PREFILL_L2_BUDGET_MB 0   // K/V bytes the concurrently running causal units should keep live
#endif
#ifndef FA_TAIL_SPLIT
#define FA_TAIL_SPLIT 1  // split a last, at most half-full round of Q-tile pairs into single tiles
#endif

namespace fa {
// One status word per device; kernels atomicOr FA_DEV_* bits into it.
__device__ unsigned int g_device_status = 0u;
// The debug build's device check record (fa_debug.cuh); untouched otherwise.
__device__ unsigned int g_debug_record[FA_DBG_WORDS] = {0u};
}  // namespace fa

namespace {

thread_local char t_detail[512] = {0};
thread_local uint64_t t_launches = 0;
std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};

fa_status fail(fa_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_detail, sizeof(t_detail), fmt, ap);
  va_end(ap);
  return s;
}

fa_status cuda_fail(cudaError_t e, const char* what) {
  return fail(FA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

struct DeviceState {
  bool ready = false;
  unsigned int* status = nullptr;
  unsigned int* debug = nullptr;  // the device check record
  int num_sms = 0;
};
using fa::kMaxDevices;
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Per-device one-time set-up: device check, status-word address, kernel
// attributes, driver entry point for tensor-map encoding.
fa_status device_state(DeviceState** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(FA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(major)");
    if ((e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(minor)");
    if (major != 10 || minor != 3)
      return fail(FA_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a only", dev, major,
                  minor);
    if ((e = cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(multiprocessors)");
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, fa::g_device_status)) != cudaSuccess)
      return cuda_fail(e, "cudaGetSymbolAddress(status)");
    void* pd = nullptr;
    if ((e = cudaGetSymbolAddress(&pd, fa::g_debug_record)) != cudaSuccess)
      return cuda_fail(e, "cudaGetSymbolAddress(debug record)");
    st.debug = static_cast<unsigned int*>(pd);
    st.status = static_cast<unsigned int*>(p);
    if ((e = fa::prefill_set_attributes(64, false)) != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(d=64)");
    if ((e = fa::prefill_set_attributes(128, false)) != cudaSuccess)
      return cuda_fail(e, "cudaFuncSetAttribute(d=128)");
    if ((e = fa::prefill_set_attributes(128, true)) != cudaSuccess)
      return cuda_fail(e, "cudaFuncSetAttribute(e4m3 d=128)");
    if ((e = fa::prefill_set_attributes(64, true)) != cudaSuccess)
      return cuda_fail(e, "cudaFuncSetAttribute(e4m3 d=64)");
    if ((e = fa::bwd_set_attributes(64)) != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(bwd d=64)");
    if ((e = fa::bwd_set_attributes(128)) != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(bwd d=128)");
    if ((e = fa::materialized_set_attributes()) != cudaSuccess)
      return cuda_fail(e, "cudaFuncSetAttribute(materialized softmax)");
    if ((e = fa::decode_grouped_set_attributes(64)) != cudaSuccess)
      return cuda_fail(e, "cudaFuncSetAttribute(grouped decode d=64)");
    if ((e = fa::decode_grouped_set_attributes(128)) != cudaSuccess)
      return cuda_fail(e, "cudaFuncSetAttribute(grouped decode d=128)");
    // The in-kernel register split assumes this launch allocation; a
    // different one could make setmaxnreg.inc wait forever, so refuse.
    for (int v = 0; v < 4; ++v) {
      const int d = (v & 1) ? 128 : 64;
      const bool f8 = v >= 2;
      const int regs = fa::prefill_num_regs(d, f8);
      if (regs != fa::prefill_launch_regs(d))
        return fail(FA_ERR_UNSUPPORTED, "prefill kernel (d=%d%s) built with %d registers, expected %d", d,
                    f8 ? ", e4m3" : "", regs, fa::prefill_launch_regs(d));
    }
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
        return fail(FA_ERR_CUDA, "driver entry point cuTensorMapEncodeTiled unavailable");
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    st.ready = true;
  }
  *out = &st;
  return FA_OK;
}

// 3-D bf16 tensor map over [BH, rows, d] with 128-row x 64-column boxes and
// 128-byte swizzle; rows past `rows` read as zeros (loads) or are not written
// (stores).
// 3-D tensor map over [BH, rows, d] with 128-byte-swizzled boxes of 128 rows
// x 128 bytes: 64 bf16 elements, or (e4m3) 128 one-byte codes.
fa_status encode_map(CUtensorMap* map, const void* base, int rows, int BH, int d, bool e4m3 = false,
                     int box_rows = 128) {
  const cuuint64_t esz = e4m3 ? 1 : 2;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * esz, static_cast<cuuint64_t>(rows) * d * esz};
  // a box row is 128 bytes (128-byte swizzle), or the whole 64-byte row of an
  // e4m3 tensor with d = 64 (64-byte swizzle)
  const cuuint64_t row_bytes = std::min<cuuint64_t>(static_cast<cuuint64_t>(d) * esz, 128);
  cuuint32_t box[3] = {static_cast<cuuint32_t>(row_bytes / esz), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, e4m3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                        const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(r));
  return FA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

fa_status check_scale(float scale) {
  if (!std::isfinite(scale)) return fail(FA_ERR_INVALID_ARG, "scale must be finite");
  return FA_OK;
}

// Streams and events of the host-buffer forward pass, one set per host
// thread and device (so concurrent callers on different threads never share
// them). Created on first use and kept for the life of the process.
struct HostPipe {
  bool ready = false;
  cudaStream_t up[3] = {nullptr, nullptr, nullptr};  // q, k, v uploads (several copy engines)
  cudaStream_t comp[2] = {nullptr, nullptr};         // one per device buffer set
  cudaStream_t down = nullptr;
  cudaEvent_t start = nullptr;
  cudaEvent_t up_done[2][3] = {};
  cudaEvent_t comp_done[2] = {};
  cudaEvent_t down_done[2] = {};
};
thread_local HostPipe t_pipe[kMaxDevices];

fa_status host_pipe(int dev, HostPipe** out) {
  HostPipe& hp = t_pipe[dev];
  if (!hp.ready) {
    cudaError_t e = cudaSuccess;
    for (auto& s : hp.up)
      if ((e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking)) != cudaSuccess) return cuda_fail(e, "stream");
    for (auto& s : hp.comp)
      if ((e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking)) != cudaSuccess) return cuda_fail(e, "stream");
    if ((e = cudaStreamCreateWithFlags(&hp.down, cudaStreamNonBlocking)) != cudaSuccess) return cuda_fail(e, "stream");
    cudaEvent_t* evs[] = {&hp.start,         &hp.up_done[0][0], &hp.up_done[0][1], &hp.up_done[0][2],
                          &hp.up_done[1][0], &hp.up_done[1][1], &hp.up_done[1][2], &hp.comp_done[0],
                          &hp.comp_done[1],  &hp.down_done[0],  &hp.down_done[1]};
    for (cudaEvent_t* ev : evs)
      if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess) return cuda_fail(e, "event");
    hp.ready = true;
  }
  *out = &hp;
  return FA_OK;
}

// Byte layout of one device buffer set of the host-buffer forward pass:
// q, k, v, o, lse of `ch` heads, each region 256-byte aligned.
struct HostSet {
  size_t q, k, v, o, lse, bytes;
};
HostSet host_set_layout(long long ch, int Nq, int Nk, int d) {
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  HostSet h{};
  const size_t qb = up(static_cast<size_t>(ch) * Nq * d * 2), kb = up(static_cast<size_t>(ch) * Nk * d * 2);
  h.q = 0;
  h.k = h.q + qb;
  h.v = h.k + kb;
  h.o = h.v + kb;
  h.lse = h.o + qb;
  h.bytes = h.lse + up(static_cast<size_t>(ch) * Nq * 4);
  return h;
}
// Heads per chunk: the caller's choice, else half of B*H. Few, large chunks
// keep every chunk's launch wide enough to fill the GPU; two still let one
// chunk's uploads overlap the other's kernel, and consecutive calls on
// different streams overlap each other.
long long host_chunk_heads(long long BH, int chunk_heads) {
  const long long ch = chunk_heads > 0 ? chunk_heads : (BH + 1) / 2;
  return std::max(1LL, std::min(ch, BH));
}

}  // namespace

// Set the calling thread's error detail (used by entry points in other files).
void fa_set_error_detail(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_detail, sizeof(t_detail), fmt, ap);
  va_end(ap);
}

extern "C" {

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE";
  }
  return "FA_UNKNOWN_STATUS";
}

const char* fa_last_error_detail(void) { return t_detail; }

uint64_t fa_launch_count(void) { return t_launches; }

void fa_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns); }
uint64_t fa_get_wait_limit_ns(void) { return g_wait_limit_ns.load(); }

namespace {
// e4m3 inputs of fa_fwd_fp8: the descale factors of q, k and v
struct E4m3Inputs {
  bool on = false;
  float dq = 1.f, dk = 1.f, dv = 1.f;
};

// The prefill launch behind fa_fwd_masked and fa_fwd_fp8.
fa_status prefill_common(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                         int Nk, int d, float scale, int causal, const uint32_t* keep_bits, int64_t mstride_b,
                         int64_t mstride_h, int64_t mstride_q, const E4m3Inputs& f8, void* stream) {
  t_detail[0] = 0;
  if (B < 1 || H < 1 || Nk < 1 || Nq < 0)
    return fail(FA_ERR_INVALID_ARG, "need B >= 1, H >= 1, Nk >= 1, Nq >= 0 (got %d %d %d %d)", B, H, Nk, Nq);
  if (fa_status s = check_scale(scale)) return s;
  if (f8.on) {
    for (float x : {f8.dq, f8.dk, f8.dv})
      if (!std::isfinite(x) || !(x > 0.f)) return fail(FA_ERR_INVALID_ARG, "descale factors must be finite and > 0");
    if (!std::isfinite(scale * f8.dq * f8.dk)) return fail(FA_ERR_INVALID_ARG, "scale * descale_q * descale_k overflows");
    if (d != 64 && d != 128)
      return fail(FA_ERR_UNSUPPORTED, "head dim %d unsupported for e4m3 inputs (64 or 128)", d);
  }
  if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "head dim %d unsupported (64 or 128)", d);
  if (Nq == 0) return FA_OK;  // nothing to compute (an empty q may have a NULL data pointer)
  if (!q || !k || !v || !o) return fail(FA_ERR_INVALID_ARG, "q, k, v and o must be non-NULL");
  if (mstride_b < 0 || mstride_h < 0 || mstride_q < 0) return fail(FA_ERR_INVALID_ARG, "mask strides must be >= 0");
  const long long BH = static_cast<long long>(B) * H;
  const long long n_qpairs = (static_cast<long long>(Nq) + 2 * fa::BLOCK_M - 1) / (2 * fa::BLOCK_M);
  if (BH > INT_MAX || n_qpairs * BH > INT_MAX) return fail(FA_ERR_INVALID_ARG, "B*H or the grid is too large");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
    return fail(FA_ERR_UNSUPPORTED, "q, k, v, o must be 16-byte aligned");
  if (keep_bits && !aligned(keep_bits, 4)) return fail(FA_ERR_UNSUPPORTED, "keep_bits must be 4-byte aligned");
  if (lse && !aligned(lse, 4)) return fail(FA_ERR_UNSUPPORTED, "lse must be 4-byte aligned");

  DeviceState* st = nullptr;
  if (fa_status s = device_state(&st)) return s;
  CUtensorMap tq, tk, tv, to;
  if (fa_status s = encode_map(&tq, q, Nq, static_cast<int>(BH), d, f8.on)) return s;
  if (fa_status s = encode_map(&to, o, Nq, static_cast<int>(BH), d)) return s;
  if (fa_status s = encode_map(&tk, k, Nk, static_cast<int>(BH), d, f8.on)) return s;
  if (fa_status s = encode_map(&tv, v, Nk, static_cast<int>(BH), d, f8.on)) return s;

  fa::PrefillParams p{};
  p.o = o;
  p.lse = lse;
  p.keep = keep_bits;
  p.msb = mstride_b;
  p.msh = mstride_h;
  p.msq = mstride_q;
  p.B = B;
  p.H = H;
  p.Nq = Nq;
  p.Nk = Nk;
  p.n_qpairs = static_cast<int>(n_qpairs);
  p.causal = causal ? 1 : 0;
  // A negative scale runs as |scale| times the negated scores (the score MMA
  // negates Q), so the row maximum is taken where the weights are largest.
  // Scale 0 (uniform weights) runs with the smallest normal multiplier
  // instead, so masked scores (-inf) still map to -inf and exponentiate to
  // exactly 0; every weight then differs from 1 by far less than fp32
  // resolution.
  // e4m3 inputs: the scores the MMA returns are in units of the codes, so
  // the q and k descales join the scale, and O / l takes the v descale.
  p.scale_log2 = fmaxf(fabsf(scale) * f8.dq * f8.dk * 1.4426950408889634f, 1.17549435e-38f);
  p.negate_s = scale < 0.f ? 1 : 0;
  p.o_scale = f8.dv;
  p.dbg = FA_DEBUG ? st->debug : nullptr;
  p.wait_limit_ns = g_wait_limit_ns.load();
  p.status = st->status;
  p.max_ctas = st->num_sms;
  // Work units are Q-tile pairs. When the pairs leave a last round of CTAs
  // (one per SM) at most half full, those last pairs are split into single
  // Q tiles so that round ends sooner; not with a broadcast key mask, whose
  // trimming assumes pair units.
  {
    const long long U = n_qpairs * BH;
    const long long G = std::max(1, st->num_sms);
    const long long r = U % G;
    const bool trim = keep_bits != nullptr && mstride_q == 0;
    const bool split = FA_TAIL_SPLIT && !trim && U >= G && r > 0 && 2 * r <= G;
    p.split_from = static_cast<int>(split ? U - r : U);
    p.units = static_cast<int>(split ? U + r : U);
    // Causal order: when all heads' K/V exceed the L2 budget, walk bands of
    // pair lengths head by head, with bands wide enough that the units running
    // at once (one per SM) touch about budget / (K/V of a head) heads.
    p.band = 0;
#if FA_PREFILL_L2_BUDGET_MB > 0
    const double kv_head = 2.0 * Nk * d * (f8.on ? 1.0 : 2.0);
    const double budget = FA_PREFILL_L2_BUDGET_MB * 1048576.0;
    if (causal && kv_head * static_cast<double>(BH) > budget) {
      const long long want = static_cast<long long>(std::ceil(static_cast<double>(G) * kv_head / budget));
      long long band = 1;
      while (band < want) band *= 2;
      p.band = static_cast<int>(std::min<long long>(band, n_qpairs));
    }
#endif
  }
  cudaError_t e = fa::launch_prefill(d, f8.on, tq, tk, tv, to, p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
  t_launches += 1;
  return FA_OK;
}
}  // namespace

fa_status fa_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                        int Nk, int d, float scale, int causal, const uint32_t* keep_bits, int64_t mstride_b,
                        int64_t mstride_h, int64_t mstride_q, void* stream) {
  return prefill_common(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, keep_bits, mstride_b, mstride_h, mstride_q,
                        E4m3Inputs{}, stream);
}

fa_status fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                     int Nk, int d, float scale, float descale_q, float descale_k, float descale_v, int causal,
                     void* stream) {
  E4m3Inputs f8;
  f8.on = true;
  f8.dq = descale_q;
  f8.dk = descale_k;
  f8.dv = descale_v;
  return prefill_common(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, nullptr, 0, 0, 0, f8, stream);
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq, int Nk,
                 int d, float scale, int causal, void* stream) {
  return fa_fwd_masked(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, nullptr, 0, 0, 0, stream);
}

size_t fa_fwd_host_workspace_size(int B, int H, int Nq, int Nk, int d, int chunk_heads) {
  if (B < 1 || H < 1 || Nq < 0 || Nk < 1 || (d != 64 && d != 128)) return 0;
  const long long ch = host_chunk_heads(static_cast<long long>(B) * H, chunk_heads);
  return 2 * host_set_layout(ch, Nq, Nk, d).bytes;
}

fa_status fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                      int Nk, int d, float scale, int causal, int chunk_heads, void* workspace,
                      size_t workspace_bytes, void* stream) {
  t_detail[0] = 0;
  if (B < 1 || H < 1 || Nk < 1 || Nq < 0)
    return fail(FA_ERR_INVALID_ARG, "need B >= 1, H >= 1, Nk >= 1, Nq >= 0 (got %d %d %d %d)", B, H, Nk, Nq);
  if (fa_status s = check_scale(scale)) return s;
  if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "head dim %d unsupported (64 or 128)", d);
  if (Nq == 0) return FA_OK;
  if (!q || !k || !v || !o) return fail(FA_ERR_INVALID_ARG, "q, k, v and o must be non-NULL");
  const long long BH = static_cast<long long>(B) * H;
  if (BH > INT_MAX) return fail(FA_ERR_INVALID_ARG, "B*H is too large");
  const long long ch = host_chunk_heads(BH, chunk_heads);
  const HostSet L = host_set_layout(ch, Nq, Nk, d);
  if (workspace == nullptr || workspace_bytes < 2 * L.bytes)
    return fail(FA_ERR_WORKSPACE, "workspace of %zu bytes given, %zu needed", workspace_bytes, 2 * L.bytes);
  if (!aligned(workspace, 256)) return fail(FA_ERR_WORKSPACE, "workspace must be 256-byte aligned");
  DeviceState* st = nullptr;
  if (fa_status s = device_state(&st)) return s;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  HostPipe* hp = nullptr;
  if (fa_status s = host_pipe(dev, &hp)) return s;

  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  // everything below is ordered after the work already queued on `stream`
  if ((e = cudaEventRecord(hp->start, cs)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  for (cudaStream_t s2 : {hp->up[0], hp->up[1], hp->up[2], hp->comp[0], hp->comp[1], hp->down})
    if ((e = cudaStreamWaitEvent(s2, hp->start, 0)) != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent");

  // On a failure after work was queued, `stream` still waits for whatever
  // the internal streams had been given, so later work on it stays ordered.
  auto join = [&](fa_status s2) {
    for (cudaStream_t x : {hp->up[0], hp->up[1], hp->up[2], hp->comp[0], hp->comp[1], hp->down})
      if (cudaEventRecord(hp->start, x) == cudaSuccess) cudaStreamWaitEvent(cs, hp->start, 0);
    return s2;
  };
  const size_t qrow = static_cast<size_t>(Nq) * d * 2, krow = static_cast<size_t>(Nk) * d * 2;
  const uint8_t* hin[3] = {static_cast<const uint8_t*>(q), static_cast<const uint8_t*>(k),
                           static_cast<const uint8_t*>(v)};
  const size_t per_head[3] = {qrow, krow, krow};
  const long long nchunks = (BH + ch - 1) / ch;
  for (long long c = 0; c < nchunks; ++c) {
    const int sidx = static_cast<int>(c & 1);
    uint8_t* set = static_cast<uint8_t*>(workspace) + sidx * L.bytes;
    const long long h0 = c * ch, nh = std::min(ch, BH - h0);
    uint8_t* din[3] = {set + L.q, set + L.k, set + L.v};
    // uploads into set sidx, once chunk c-2's kernel has finished reading it
    for (int t = 0; t < 3; ++t) {
      if (c >= 2 && (e = cudaStreamWaitEvent(hp->up[t], hp->comp_done[sidx], 0)) != cudaSuccess)
        return join(cuda_fail(e, "cudaStreamWaitEvent"));
      if ((e = cudaMemcpyAsync(din[t], hin[t] + h0 * per_head[t], nh * per_head[t], cudaMemcpyHostToDevice,
                               hp->up[t])) != cudaSuccess)
        return join(cuda_fail(e, "cudaMemcpyAsync(host to device)"));
      if ((e = cudaEventRecord(hp->up_done[sidx][t], hp->up[t])) != cudaSuccess)
        return join(cuda_fail(e, "cudaEventRecord"));
    }
    // the chunk's forward pass, once its inputs landed and chunk c-2's
    // outputs have been read back from this set
    cudaStream_t comp = hp->comp[sidx];
    for (int t = 0; t < 3; ++t)
      if ((e = cudaStreamWaitEvent(comp, hp->up_done[sidx][t], 0)) != cudaSuccess)
        return join(cuda_fail(e, "cudaStreamWaitEvent"));
    if (c >= 2 && (e = cudaStreamWaitEvent(comp, hp->down_done[sidx], 0)) != cudaSuccess)
      return join(cuda_fail(e, "cudaStreamWaitEvent"));
    float* dlse = lse ? reinterpret_cast<float*>(set + L.lse) : nullptr;
    if (fa_status s2 = fa_fwd(din[0], din[1], din[2], set + L.o, dlse, 1, static_cast<int>(nh), Nq, Nk, d, scale,
                              causal, comp))
      return join(s2);
    if ((e = cudaEventRecord(hp->comp_done[sidx], comp)) != cudaSuccess)
      return join(cuda_fail(e, "cudaEventRecord"));
    // read-back of the chunk's o and lse
    if ((e = cudaStreamWaitEvent(hp->down, hp->comp_done[sidx], 0)) != cudaSuccess)
      return join(cuda_fail(e, "cudaStreamWaitEvent"));
    if ((e = cudaMemcpyAsync(static_cast<uint8_t*>(o) + h0 * qrow, set + L.o, nh * qrow, cudaMemcpyDeviceToHost,
                             hp->down)) != cudaSuccess)
      return join(cuda_fail(e, "cudaMemcpyAsync(device to host)"));
    if (lse && (e = cudaMemcpyAsync(lse + h0 * Nq, dlse, nh * Nq * sizeof(float), cudaMemcpyDeviceToHost,
                                    hp->down)) != cudaSuccess)
      return join(cuda_fail(e, "cudaMemcpyAsync(device to host)"));
    if ((e = cudaEventRecord(hp->down_done[sidx], hp->down)) != cudaSuccess)
      return join(cuda_fail(e, "cudaEventRecord"));
  }
  // the read-back stream runs the chunks in order: its last event covers them all
  if ((e = cudaStreamWaitEvent(cs, hp->down_done[(nchunks - 1) & 1], 0)) != cudaSuccess)
    return join(cuda_fail(e, "cudaStreamWaitEvent"));
  return FA_OK;
}

size_t fa_decode_workspace_size(int B, int H, int d, int num_splits) {
  if (B < 1 || H < 1 || (d != 64 && d != 128) || num_splits < 1 || num_splits > 1024) return 0;
  const size_t parts = static_cast<size_t>(B) * H * num_splits;
  const size_t o_bytes = (parts * d * 4 + 255) & ~size_t(255);
  const size_t ml_bytes = (parts * 2 * 4 + 255) & ~size_t(255);
  return o_bytes + ml_bytes;
}

fa_status fa_decode_splitkv(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse, int B,
                            int H, int Nk, int d, float scale, int num_splits, void* workspace,
                            size_t workspace_bytes, void* stream) {
  t_detail[0] = 0;
  if (!q || !k_cache || !v_cache || !o) return fail(FA_ERR_INVALID_ARG, "q, k_cache, v_cache and o must be non-NULL");
  if (B < 1 || H < 1 || Nk < 1) return fail(FA_ERR_INVALID_ARG, "need B >= 1, H >= 1, Nk >= 1");
  if (num_splits < 1 || num_splits > 1024) return fail(FA_ERR_INVALID_ARG, "num_splits must be in [1, 1024]");
  if (fa_status s = check_scale(scale)) return s;
  const long long BH = static_cast<long long>(B) * H;
  if (BH * num_splits > INT_MAX) return fail(FA_ERR_INVALID_ARG, "B*H*num_splits is too large");
  if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "head dim %d unsupported (64 or 128)", d);
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(o, 16))
    return fail(FA_ERR_UNSUPPORTED, "q, k_cache, v_cache, o must be 16-byte aligned");
  if (lse && !aligned(lse, 4)) return fail(FA_ERR_UNSUPPORTED, "lse must be 4-byte aligned");
  const size_t need = fa_decode_workspace_size(B, H, d, num_splits);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < need)
    return fail(FA_ERR_WORKSPACE, "workspace must be 256-byte aligned and >= %zu bytes", need);

  DeviceState* st = nullptr;
  if (fa_status s = device_state(&st)) return s;
  const size_t parts = static_cast<size_t>(BH) * num_splits;
  fa::DecodeParams p{};
  p.q = q;
  p.k = k_cache;
  p.v = v_cache;
  p.o = o;
  p.lse = lse;
  p.ws_o = static_cast<float*>(workspace);
  p.ws_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) + ((parts * d * 4 + 255) & ~size_t(255)));
  p.BH = static_cast<int>(BH);
  p.Nk = Nk;
  p.S = num_splits;
  p.chunk = (Nk + num_splits - 1) / num_splits;
  p.scale_log2 = scale * 1.4426950408889634f;
  cudaError_t e = fa::launch_decode(d, p, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  t_launches += 2;
  return FA_OK;
}

size_t fa_decode_grouped_workspace_size(int B, int H, int Nq, int d, int num_splits) {
  if (Nq < 1 || Nq > 128 || static_cast<long long>(H) * Nq > INT_MAX) return 0;
  return fa_decode_workspace_size(B, H * Nq, d, num_splits);
}

fa_status fa_decode_grouped(const void* q, const void* k_cache, const void* v_cache, const int* seqlens_k, void* o,
                            float* lse, int B, int H, int Hkv, int Nq, int Nk, int d, float scale, int num_splits,
                            void* workspace, size_t workspace_bytes, void* stream) {
  t_detail[0] = 0;
  if (!q || !k_cache || !v_cache || !o) return fail(FA_ERR_INVALID_ARG, "q, k_cache, v_cache and o must be non-NULL");
  if (B < 1 || H < 1 || Hkv < 1 || Nq < 1 || Nk < 1)
    return fail(FA_ERR_INVALID_ARG, "need B, H, Hkv, Nq, Nk >= 1 (got %d %d %d %d %d)", B, H, Hkv, Nq, Nk);
  if (H % Hkv != 0) return fail(FA_ERR_INVALID_ARG, "H (%d) must be a multiple of Hkv (%d)", H, Hkv);
  if (num_splits < 1 || num_splits > 1024) return fail(FA_ERR_INVALID_ARG, "num_splits must be in [1, 1024]");
  if (fa_status s = check_scale(scale)) return s;
  if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "head dim %d unsupported (64 or 128)", d);
  const int G = H / Hkv;
  if (static_cast<long long>(G) * Nq > 128)
    return fail(FA_ERR_UNSUPPORTED, "(H / Hkv) * Nq = %lld query rows per K/V head; at most 128",
                static_cast<long long>(G) * Nq);
  const long long rows = static_cast<long long>(B) * H * Nq;
  if (static_cast<long long>(B) * Hkv * num_splits > INT_MAX || rows * num_splits > INT_MAX)
    return fail(FA_ERR_INVALID_ARG, "B * H * Nq * num_splits is too large");
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(o, 16))
    return fail(FA_ERR_UNSUPPORTED, "q, k_cache, v_cache, o must be 16-byte aligned");
  if (lse && !aligned(lse, 4)) return fail(FA_ERR_UNSUPPORTED, "lse must be 4-byte aligned");
  if (seqlens_k && !aligned(seqlens_k, 4)) return fail(FA_ERR_UNSUPPORTED, "seqlens_k must be 4-byte aligned");
  const size_t need = fa_decode_grouped_workspace_size(B, H, Nq, d, num_splits);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < need)
    return fail(FA_ERR_WORKSPACE, "workspace must be 256-byte aligned and >= %zu bytes", need);

  DeviceState* st = nullptr;
  if (fa_status s = device_state(&st)) return s;
  const int BHkv = B * Hkv;
  CUtensorMap tq, tk, tv;
  // the G*Nq rows of a group are contiguous; the box covers the kernel's query tile
  if (fa_status s = encode_map(&tq, q, G * Nq, BHkv, d, false, fa::decode_grouped_q_box_rows(d, G * Nq))) return s;
  if (fa_status s = encode_map(&tk, k_cache, Nk, BHkv, d)) return s;
  if (fa_status s = encode_map(&tv, v_cache, Nk, BHkv, d)) return s;
  const size_t parts = static_cast<size_t>(rows) * num_splits;
  float* ws_o = static_cast<float*>(workspace);
  float* ws_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) + ((parts * d * 4 + 255) & ~size_t(255)));
  fa::DecodeGroupedParams p{};
  p.q = q;
  p.k = k_cache;
  p.v = v_cache;
  p.seqlens = seqlens_k;
  p.ws_o = ws_o;
  p.ws_ml = ws_ml;
  p.B = B;
  p.H = H;
  p.Hkv = Hkv;
  p.G = G;
  p.Nq = Nq;
  p.R = G * Nq;
  p.Nk = Nk;
  p.S = num_splits;
  p.chunk = ((Nk + num_splits - 1) / num_splits + 127) / 128 * 128;
  // as in the prefill: a negative scale negates the scores in the MMA
  p.scale_log2 = fmaxf(fabsf(scale) * 1.4426950408889634f, 1.17549435e-38f);
  p.negate_s = scale < 0.f ? 1 : 0;
  p.wait_limit_ns = g_wait_limit_ns.load();
  p.status = st->status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = fa::launch_decode_grouped(d, tq, tk, tv, p, s);
  if (e != cudaSuccess) return cuda_fail(e, "grouped decode launch");
  fa::DecodeParams m{};
  m.o = o;
  m.lse = lse;
  m.ws_o = ws_o;
  m.ws_ml = ws_ml;
  m.BH = static_cast<int>(rows);
  m.S = num_splits;
  if ((e = fa::launch_decode_merge(d, m, s)) != cudaSuccess) return cuda_fail(e, "grouped decode merge launch");
  t_launches += 2;
  return FA_OK;
}

// ---------------------------------------------------------------------------
// Materialising baseline: two cuBLAS GEMMs around the row-softmax kernel.
// cuBLAS is opened on first use (the library itself does not link it), with
// one handle per device; calls are serialised on a mutex because the handle's
// stream is set per call.
namespace {

struct CublasApi {
  bool tried = false;
  bool ok = false;
  decltype(&cublasCreate_v2) create = nullptr;
  decltype(&cublasSetStream_v2) set_stream = nullptr;
  // the exported C symbol (32-bit sizes); the C++ header also declares a 64-bit overload
  using gemm_t = cublasStatus_t (*)(cublasHandle_t, cublasOperation_t, cublasOperation_t, int, int, int, const void*,
                                    const void*, cudaDataType, int, long long int, const void*, cudaDataType, int,
                                    long long int, const void*, void*, cudaDataType, int, long long int, int,
                                    cublasComputeType_t, cublasGemmAlgo_t);
  gemm_t gemm = nullptr;
  cublasHandle_t handle[kMaxDevices] = {};
};
CublasApi g_cublas;
std::mutex g_cublas_mu;

// Returns the device's handle, or nullptr with the error detail set.
cublasHandle_t cublas_handle(int dev) {
  if (!g_cublas.tried) {
    g_cublas.tried = true;
    void* lib = nullptr;
    for (const char* name : {"libcublas.so.13", "libcublas.so"})
      if ((lib = dlopen(name, RTLD_NOW | RTLD_LOCAL)) != nullptr) break;
    if (lib) {
      g_cublas.create = reinterpret_cast<decltype(g_cublas.create)>(dlsym(lib, "cublasCreate_v2"));
      g_cublas.set_stream = reinterpret_cast<decltype(g_cublas.set_stream)>(dlsym(lib, "cublasSetStream_v2"));
      g_cublas.gemm = reinterpret_cast<CublasApi::gemm_t>(dlsym(lib, "cublasGemmStridedBatchedEx"));
      g_cublas.ok = g_cublas.create && g_cublas.set_stream && g_cublas.gemm;
    }
  }
  if (!g_cublas.ok) {
    fail(FA_ERR_UNSUPPORTED, "cuBLAS (libcublas.so.13) could not be loaded");
    return nullptr;
  }
  if (!g_cublas.handle[dev]) {
    cublasHandle_t h = nullptr;
    if (g_cublas.create(&h) != CUBLAS_STATUS_SUCCESS) {
      fail(FA_ERR_CUDA, "cublasCreate failed");
      return nullptr;
    }
    g_cublas.handle[dev] = h;
  }
  return g_cublas.handle[dev];
}

}  // namespace

size_t fa_materialized_workspace_size(int B, int H, int Nq, int Nk) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return 0;
  return (static_cast<size_t>(B) * H * Nq * Nk * 2 + 255) & ~size_t(255);
}

fa_status fa_fwd_materialized(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                              int Nk, int d, float scale, int causal, void* workspace, size_t workspace_bytes,
                              void* stream) {
  t_detail[0] = 0;
  if (!q || !k || !v || !o) return fail(FA_ERR_INVALID_ARG, "q, k, v and o must be non-NULL");
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1)
    return fail(FA_ERR_INVALID_ARG, "need B >= 1, H >= 1, Nq >= 1, Nk >= 1 (got %d %d %d %d)", B, H, Nq, Nk);
  if (fa_status s = check_scale(scale)) return s;
  if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "head dim %d unsupported (64 or 128)", d);
  if (Nk % 8 != 0 || Nk > fa::MATERIALIZED_MAX_NK)
    return fail(FA_ERR_UNSUPPORTED, "the materialising baseline takes Nk a multiple of 8 and at most %d (got %d)",
                fa::MATERIALIZED_MAX_NK, Nk);
  const long long BH = static_cast<long long>(B) * H;
  if (BH > INT_MAX || BH * Nq > INT_MAX) return fail(FA_ERR_INVALID_ARG, "B * H * Nq is too large");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
    return fail(FA_ERR_UNSUPPORTED, "q, k, v, o must be 16-byte aligned");
  if (lse && !aligned(lse, 4)) return fail(FA_ERR_UNSUPPORTED, "lse must be 4-byte aligned");
  const size_t need = fa_materialized_workspace_size(B, H, Nq, Nk);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < need)
    return fail(FA_ERR_WORKSPACE, "workspace must be 256-byte aligned and >= %zu bytes", need);
  DeviceState* st = nullptr;
  if (fa_status s = device_state(&st)) return s;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lock(g_cublas_mu);
  cublasHandle_t h = cublas_handle(dev);
  if (!h) return g_cublas.ok ? FA_ERR_CUDA : FA_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (g_cublas.set_stream(h, s) != CUBLAS_STATUS_SUCCESS) return fail(FA_ERR_CUDA, "cublasSetStream failed");
  // Row-major S [Nq, Nk] is column-major S^T = K Q^T: A = K (row-major [Nk, d], read transposed), B = Q.
  const float alpha = scale, beta = 0.f, one = 1.f;
  cublasStatus_t cs = g_cublas.gemm(h, CUBLAS_OP_T, CUBLAS_OP_N, Nk, Nq, d, &alpha, k, CUDA_R_16BF, d,
                                    static_cast<long long>(Nk) * d, q, CUDA_R_16BF, d,
                                    static_cast<long long>(Nq) * d, &beta, workspace, CUDA_R_16BF, Nk,
                                    static_cast<long long>(Nq) * Nk, static_cast<int>(BH), CUBLAS_COMPUTE_32F,
                                    CUBLAS_GEMM_DEFAULT);
  if (cs != CUBLAS_STATUS_SUCCESS) return fail(FA_ERR_CUDA, "cublasGemmStridedBatchedEx (scores) failed: %d", cs);
  fa::MaterializedParams mp{};
  mp.s = workspace;
  mp.lse = lse;
  mp.rows = BH * Nq;
  mp.Nq = Nq;
  mp.Nk = Nk;
  mp.causal = causal ? 1 : 0;
  if ((e = fa::launch_materialized_softmax(mp, s)) != cudaSuccess) return cuda_fail(e, "materialized softmax");
  // Row-major O [Nq, d] is column-major O^T = V^T P^T: A = V (column-major [d, Nk]), B = P (column-major [Nk, Nq]).
  cs = g_cublas.gemm(h, CUBLAS_OP_N, CUBLAS_OP_N, d, Nq, Nk, &one, v, CUDA_R_16BF, d,
                     static_cast<long long>(Nk) * d, workspace, CUDA_R_16BF, Nk, static_cast<long long>(Nq) * Nk,
                     &beta, o, CUDA_R_16BF, d, static_cast<long long>(Nq) * d, static_cast<int>(BH),
                     CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
  if (cs != CUBLAS_STATUS_SUCCESS) return fail(FA_ERR_CUDA, "cublasGemmStridedBatchedEx (values) failed: %d", cs);
  t_launches += 1;  // the softmax kernel; the two GEMMs are cuBLAS's
  return FA_OK;
}

size_t fa_bwd_workspace_size(int B, int H, int Nq, int d) {
  if (B < 1 || H < 1 || Nq < 1 || (d != 64 && d != 128)) return 0;
  const size_t rows = static_cast<size_t>(B) * H * Nq;
  const size_t rows_pad = static_cast<size_t>(B) * H * ((static_cast<size_t>(Nq) + 127) / 128) * 128;
  const size_t acc = (rows_pad * d * 4 + 255) & ~size_t(255);
  const size_t stat = (rows * 4 + 255) & ~size_t(255);
  return acc + 2 * stat;
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                 void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d, float scale, int causal,
                 void* workspace, size_t workspace_bytes, void* stream) {
  t_detail[0] = 0;
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1)
    return fail(FA_ERR_INVALID_ARG, "need B >= 1, H >= 1, Nq >= 1, Nk >= 1 (got %d %d %d %d)", B, H, Nq, Nk);
  if (fa_status s = check_scale(scale)) return s;
  if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "head dim %d unsupported (64 or 128)", d);
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv)
    return fail(FA_ERR_INVALID_ARG, "q, k, v, o, dout, lse, dq, dk and dv must be non-NULL");
  const long long BH = static_cast<long long>(B) * H;
  const long long ctas = BH * ((Nk + 127) / 128);
  if (BH > INT_MAX || ctas > INT_MAX || BH * Nq > (1LL << 40))
    return fail(FA_ERR_INVALID_ARG, "B*H or the grid is too large");
  for (const void* ptr : {q, k, v, o, dout, static_cast<const void*>(dq), static_cast<const void*>(dk),
                          static_cast<const void*>(dv)})
    if (!aligned(ptr, 16)) return fail(FA_ERR_UNSUPPORTED, "q, k, v, o, dout, dq, dk, dv must be 16-byte aligned");
  if (!aligned(lse, 4)) return fail(FA_ERR_UNSUPPORTED, "lse must be 4-byte aligned");
  const size_t need = fa_bwd_workspace_size(B, H, Nq, d);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < need)
    return fail(FA_ERR_WORKSPACE, "workspace must be 256-byte aligned and >= %zu bytes", need);

  DeviceState* st = nullptr;
  if (fa_status s = device_state(&st)) return s;
  CUtensorMap tq, tk, tv, tdo;
  if (fa_status s = encode_map(&tq, q, Nq, static_cast<int>(BH), d)) return s;
  if (fa_status s = encode_map(&tk, k, Nk, static_cast<int>(BH), d)) return s;
  if (fa_status s = encode_map(&tv, v, Nk, static_cast<int>(BH), d)) return s;
  if (fa_status s = encode_map(&tdo, dout, Nq, static_cast<int>(BH), d)) return s;
  const size_t rows = static_cast<size_t>(BH) * Nq;
  const size_t rows_pad = static_cast<size_t>(BH) * ((static_cast<size_t>(Nq) + 127) / 128) * 128;
  const size_t acc = (rows_pad * d * 4 + 255) & ~size_t(255);
  const size_t stat = (rows * 4 + 255) & ~size_t(255);
  fa::BwdParams p{};
  p.dq_acc = static_cast<float*>(workspace);
  p.lse2 = reinterpret_cast<float*>(static_cast<char*>(workspace) + acc);
  p.drow = reinterpret_cast<float*>(static_cast<char*>(workspace) + acc + stat);
  p.dk = dk;
  p.dv = dv;
  p.B = B;
  p.H = H;
  p.Nq = Nq;
  p.Nk = Nk;
  p.causal = causal ? 1 : 0;
  p.scale = scale;
  // as in the forward pass, scale 0 runs with the smallest normal multiplier;
  // the backward pass takes no row maximum, so a negative scale keeps its sign
  p.scale_log2 = scale == 0.f ? 1.17549435e-38f : scale * 1.4426950408889634f;
  p.wait_limit_ns = g_wait_limit_ns.load();
  p.status = st->status;
  cudaError_t e = fa::launch_bwd(d, tq, tk, tv, tdo, p, o, dout, lse, dq, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "backward launch");
  t_launches += 3;
  return FA_OK;
}

fa_status fa_get_device_status(void* stream) {
  t_detail[0] = 0;
  DeviceState* st = nullptr;
  if (fa_status s = device_state(&st)) return s;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned int word = 0;
  if ((e = cudaMemcpyAsync(&word, st->status, sizeof(word), cudaMemcpyDeviceToHost, s)) != cudaSuccess)
    return cuda_fail(e, "read status");
  if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  if (word != 0u) {
    if ((e = cudaMemsetAsync(st->status, 0, sizeof(word), s)) != cudaSuccess) return cuda_fail(e, "clear status");
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  }
  if (word & fa::FA_DEV_TIMEOUT) return fail(FA_ERR_TIMEOUT, "a bounded wait inside a kernel gave up");
  return FA_OK;
}

fa_status fa_selftest_wait_timeout(uint64_t limit_ns, void* stream) {
  t_detail[0] = 0;
  DeviceState* st = nullptr;
  if (fa_status s = device_state(&st)) return s;
  cudaError_t e = fa::launch_wait_selftest(limit_ns, st->status, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  t_launches += 1;
  return fa_get_device_status(stream);
}

fa_status fa_selftest_exp2(const float* x, float* y, int n, void* stream) {
  t_detail[0] = 0;
  if (n < 0 || (n > 0 && (!x || !y))) return fail(FA_ERR_INVALID_ARG, "need n >= 0 and non-NULL x, y");
  if (n == 0) return FA_OK;
  DeviceState* st = nullptr;
  if (fa_status s = device_state(&st)) return s;
  cudaError_t e = fa::launch_exp2_selftest(x, y, n, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "exp2 self-test launch");
  t_launches += 1;
  return FA_OK;
}

int fa_debug_enabled(void) { return FA_DEBUG ? 1 : 0; }

fa_status fa_debug_record(uint32_t* out, void* stream) {
  t_detail[0] = 0;
  if (!out) return fail(FA_ERR_INVALID_ARG, "out must hold 8 words");
  DeviceState* st = nullptr;
  if (fa_status s = device_state(&st)) return s;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(out, st->debug, fa::FA_DBG_WORDS * sizeof(uint32_t), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e == cudaSuccess) e = cudaMemsetAsync(st->debug, 0, fa::FA_DBG_WORDS * sizeof(uint32_t), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "debug record read-back");
  return FA_OK;
}

fa_status fa_debug_selftest(void* stream) {
  t_detail[0] = 0;
  DeviceState* st = nullptr;
  if (fa_status s = device_state(&st)) return s;
  cudaError_t e = fa::launch_debug_selftest(st->debug, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "debug self-test launch");
  t_launches += 1;
  return FA_OK;
}

}  // extern "C"
