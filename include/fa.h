/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact-attention library libfa_gb300.so.
 *
 * The operation (all entry points): for every batch b, head h and query row i
 *
 *     s_ij  = scale * <q_i, k_j>                       (scaled scores)
 *     allowed(i, j) = (!causal || j <= i + (Nk - Nq)) && keep(b, h, i, j)
 *     O_i   = sum_j softmax_j(s_ij over allowed j) * v_j
 *     lse_i = ln sum_{allowed j} exp(s_ij)
 *
 * "Flash Attention Optimization", section "Attention is not slow because of
 * arithmetic" (S = Q K^T / sqrt(d), P = softmax(S), O = P V); "Explain
 * FlashAttention. Why is it called IO-aware, and what does it actually
 * save?", section "Keep only the state needed for the final weighted average"
 * (scores plus the intended mask or bias; the causal mask uses absolute query
 * and key positions). A row with no allowed key returns O = 0 and
 * lse = -inf (the explicit empty-row policy of the section "Executable
 * recurrence, with an empty-state policy"). lse is the per-row statistic a
 * backward pass recomputes P from ("Flash Attention Optimization", section
 * "Sizing a tile, and why the backward pass recomputes instead of storing").
 * Causal alignment for Nq != Nk is bottom-right (query i sees keys
 * j <= i + Nk - Nq), the reading the library takes where the pages are silent.
 *
 * Layout (all device pointers, row-major, contiguous):
 *   q, o      bf16 [B, H, Nq, d]        k, v   bf16 [B, H, Nk, d]
 *   lse       fp32 [B, H, Nq]           (may be NULL: not written)
 *   keep_bits uint32 words; bit (j % 32) of word (j / 32) is key j, 1 = attend;
 *             the words of row (b, h, i) start at
 *             b*mstride_b + h*mstride_h + i*mstride_q (strides in words;
 *             mstride_q = 0 broadcasts one key mask over all rows). Each row
 *             holds ceil(Nk / 32) words; bits past Nk are ignored.
 *   stream    a cudaStream_t (NULL = the legacy default stream).
 * Supported: d in {64, 128}; q, k, v, o 16-byte aligned; keep_bits 4-byte
 * aligned; 1 <= B*H, Nk < 2^31; scale any finite value (a negative scale
 * gives the largest weights to the smallest dot products, as the definition
 * says; scale 0 gives uniform weights over the visible keys).
 *
 * Ownership: the caller allocates and owns every buffer; the library keeps
 * no pointer after a call returns and allocates no device memory per call
 * (the decode workspace is the caller's). Calls are asynchronous on `stream`:
 * a return of FA_OK means the work was launched.
 *
 * Errors (checked on the host before anything is launched; nothing is
 * written on error):
 *   FA_ERR_INVALID_ARG  a required pointer is NULL, a size is negative or
 *                       zero where it must be positive, scale is NaN or
 *                       infinite, or a size overflows the supported range.
 *   FA_ERR_UNSUPPORTED  d not in {64, 128}, a misaligned pointer, or no
 *                       sm_103 device is current. There is no fallback path.
 *   FA_ERR_WORKSPACE    the decode workspace is NULL or too small.
 *   FA_ERR_CUDA         a CUDA call failed (fa_last_error_detail() says which).
 *   FA_ERR_TIMEOUT      reported later by fa_get_device_status(): a bounded
 *                       wait inside a kernel gave up; that call's outputs are
 *                       undefined, the CUDA context stays usable.
 * Inputs are not scanned for NaN/inf (that would cost bandwidth): a NaN or
 * inf in q, k or v propagates to the rows it touches.
 *
 * Device reset: the first call on a device caches that device's state (the
 * status word's address, kernel attributes, the no-alloc scratch address)
 * for its primary context. cudaDeviceReset while the library is loaded
 * invalidates that state; calls made after a reset are not supported.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,
  FA_ERR_UNSUPPORTED = 2,
  FA_ERR_CUDA = 3,
  FA_ERR_TIMEOUT = 4,
  FA_ERR_WORKSPACE = 5
} fa_status;

/* Fused, tiled forward pass (prefill). Q tiles stay on chip while K/V tiles
 * stream through; the Nq x Nk score matrix never reaches HBM ("Flash
 * Attention Optimization", section "The fix: tile the computation, never
 * materialize the full matrix"). Nq = 0 is a no-op (q and o may then be NULL). */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int H, int Nq, int Nk, int d, float scale, int causal, void* stream);

/* fa_fwd with an additional key mask (see keep_bits above), ANDed with the
 * causal mask when causal != 0. keep_bits = NULL is the same as fa_fwd. */
fa_status fa_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse,
                        int B, int H, int Nq, int Nk, int d, float scale, int causal,
                        const uint32_t* keep_bits, int64_t mstride_b, int64_t mstride_h,
                        int64_t mstride_q, void* stream);

/* Forward pass on FP8 inputs ("FlashAttention: Attention Is Limited by
 * Memory, Not Math", section "FlashAttention 1, 2 and 3", lists FP8 support
 * among FlashAttention-3's changes; the pages give no further detail).
 *   q, k, v   e4m3 codes (one byte each: 1 sign, 4 exponent bits with bias
 *             7, 3 mantissa bits; no infinities), layouts as for fa_fwd;
 *             16-byte aligned.
 *   descale_q, descale_k, descale_v
 *             one fp32 factor per tensor: the real value of a code c of q is
 *             e4m3(c) * descale_q (likewise k, v); finite and > 0.
 *   o, lse    bf16 O and fp32 lse of exact attention on those real values,
 *             softmax(scale * Q K^T + causal mask) V, as fa_fwd defines them.
 * The score and value products run on the tensor cores in e4m3 with fp32
 * accumulation; P is rounded to e4m3 (round to nearest even) before the P V
 * product, which is this path's main error against the exact result.
 * Supported: d = 64 or 128 (FA_ERR_UNSUPPORTED otherwise); no key mask. Errors as
 * for fa_fwd, plus FA_ERR_INVALID_ARG for a descale that is not finite and
 * positive, or a product scale * descale_q * descale_k that overflows. */
fa_status fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int H, int Nq, int Nk, int d, float scale,
                     float descale_q, float descale_k, float descale_v, int causal, void* stream);

/* Bytes of device workspace fa_fwd_host needs: two buffer sets, each holding
 * q, k, v, o and lse of one chunk of heads (every region rounded up to 256
 * bytes). chunk_heads <= 0 selects the default, ceil(B*H / 2) heads. Returns 0
 * for invalid arguments. */
size_t fa_fwd_host_workspace_size(int B, int H, int Nq, int Nk, int d, int chunk_heads);

/* fa_fwd on HOST buffers: q, k, v, o and lse have the layouts above but live
 * in host memory. The B*H heads (contiguous in that layout) are processed in
 * chunks of chunk_heads. Each chunk's q, k and v are copied into one of two
 * device buffer sets in the workspace, and its forward pass runs there. Its o
 * and lse are then copied back. Upload, compute and read-back of consecutive
 * chunks overlap: they run on library-owned streams (three upload streams,
 * one compute stream per buffer set, one read-back stream), one set of
 * streams per host thread and device. The call is ordered after the work
 * already queued on `stream`, and `stream` waits for the last read-back. The
 * outputs are complete once `stream` has been synchronised; the inputs must
 * stay unchanged until then.
 *
 * Host memory should be page-locked (cudaHostAlloc / cudaHostRegister) for
 * the copies to overlap the kernels. Pageable memory gives the same results
 * with serialised copies.
 *
 * workspace: device memory, 256-byte aligned, at least
 * fa_fwd_host_workspace_size(...) bytes, not used by anything else until
 * `stream` reaches the end of the call. Errors: those of fa_fwd (host
 * pointers need no alignment), and FA_ERR_WORKSPACE for a NULL, short or
 * misaligned workspace. A CUDA failure after some chunks were queued returns
 * FA_ERR_CUDA; `stream` still waits for the queued work, and the outputs are
 * undefined. */
fa_status fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse,
                      int B, int H, int Nq, int Nk, int d, float scale, int causal,
                      int chunk_heads, void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device workspace fa_decode_splitkv needs: fp32 partial
 * (o[d], m, l) per (b, h, split), i.e. B*H*num_splits*(d + 2)*4 rounded up
 * to 256. Returns 0 for invalid arguments. */
size_t fa_decode_workspace_size(int B, int H, int d, int num_splits);

/* Split-KV decode: one query token per (b, h) against a KV cache of Nk keys
 * ("FlashAttention: Attention Is Limited by Memory, Not Math", section
 * "Where it helps, and where it does not": split the K/V sequence across the
 * GPU, then merge the partial results; the merge re-bases each split to the
 * global max, "Handwritten Notes on Flash Attention", section "Merging two
 * blocks"). Split s covers keys [s*c, min(Nk, (s+1)*c)) with
 * c = ceil(Nk / num_splits); empty splits contribute nothing.
 *   q, o     bf16 [B, H, 1, d]     k_cache, v_cache  bf16 [B, H, Nk, d]
 *   lse      fp32 [B, H] (may be NULL)
 *   workspace  device memory of at least fa_decode_workspace_size() bytes,
 *              256-byte aligned, owned by the caller; its contents on entry
 *              do not matter and are overwritten.
 *   1 <= num_splits <= 1024. Two launches (split, then merge) on `stream`. */
fa_status fa_decode_splitkv(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                            int B, int H, int Nk, int d, float scale, int num_splits,
                            void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of the static device scratch behind fa_decode_splitkv_noalloc. */
#define FA_DECODE_NOALLOC_SCRATCH_BYTES (20u << 20)

/* Split-KV decode for callers that cannot allocate device memory. (The pages
 * have no counterpart: this is an interface variant, not part of the method.)
 * Some callers only hold the input and output buffers: a plugin or kernel
 * interface that passes no workspace, or a serving loop that must not call
 * cudaMalloc/cudaFree because those calls can synchronise the device or
 * because another allocator owns the device memory. This entry point takes
 * the same arguments as fa_decode_splitkv without the workspace, allocates
 * nothing, and keeps the per-split partial states in one static device array
 * of FA_DECODE_NOALLOC_SCRATCH_BYTES that every GPU loading the library
 * holds until the process exits. It computes exactly what fa_decode_splitkv
 * computes, with the same kernels.
 *   - Requests needing more scratch than that (fa_decode_workspace_size() >
 *     FA_DECODE_NOALLOC_SCRATCH_BYTES) return FA_ERR_WORKSPACE and launch
 *     nothing; use fa_decode_splitkv with a caller workspace instead.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture. The address is cached for the device's
 *     primary context; after cudaDeviceReset it is stale, as is the rest of
 *     the library's per-device state (see "Device reset" above).
 *   - All calls share the one array: calls whose work overlaps on the GPU
 *     (different streams, or host threads without ordering) race and corrupt
 *     each other's results. Calls ordered on one stream are safe; the array
 *     needs no clearing between them because every partial is rewritten. */
fa_status fa_decode_splitkv_noalloc(const void* q, const void* k_cache, const void* v_cache, void* o, float* lse,
                                    int B, int H, int Nk, int d, float scale, int num_splits, void* stream);

/* Bytes of device workspace fa_decode_grouped needs: the split-KV partial
 * states of B*H*Nq query rows, fa_decode_workspace_size(B, H*Nq, d,
 * num_splits). Returns 0 for invalid arguments (including Nq > 128). */
size_t fa_decode_grouped_workspace_size(int B, int H, int Nq, int d, int num_splits);

/* Split-KV decode with grouped K/V heads, several new query tokens per
 * sequence and per-sequence KV lengths (the decode variants next to
 * "FlashAttention: Attention Is Limited by Memory, Not Math", section "Where
 * it helps, and where it does not"; the merge as for fa_decode_splitkv).
 * H query heads share Hkv K/V heads: query head h reads K/V head h / (H/Hkv).
 * Sequence b holds L_b = seqlens_k[b] keys (clamped to [0, Nk]; all Nk when
 * seqlens_k is NULL), and its Nq new tokens are its last Nq positions: token t
 * sees key j iff j < L_b and j <= L_b - Nq + t. A token that sees no key gets
 * o = 0 and lse = -inf. The (H/Hkv)*Nq query rows of one (b, K/V head) read
 * the K/V stream together, so each K/V byte is read once per group: up to four
 * rows on the CUDA cores (packed fp32 products), more in one tensor-core tile.
 *   q, o       bf16 [B, H, Nq, d]      k_cache, v_cache  bf16 [B, Hkv, Nk, d]
 *   seqlens_k  int32 [B] in device memory, or NULL
 *   lse        fp32 [B, H, Nq] (may be NULL)
 *   workspace  device memory of at least fa_decode_grouped_workspace_size()
 *              bytes, 256-byte aligned, owned by the caller; overwritten.
 *   Split s covers keys [s*c, min(L_b, (s+1)*c)), c = ceil(Nk / num_splits)
 *   rounded up to a multiple of 128; 1 <= num_splits <= 1024.
 * Errors: FA_ERR_INVALID_ARG for NULL tensors, sizes < 1, H not a multiple of
 * Hkv or a bad scale; FA_ERR_UNSUPPORTED for d not in {64, 128},
 * (H/Hkv)*Nq > 128 or misaligned pointers; FA_ERR_WORKSPACE. Two launches
 * (grouped split kernel, then merge) on `stream`. */
fa_status fa_decode_grouped(const void* q, const void* k_cache, const void* v_cache, const int* seqlens_k, void* o,
                            float* lse, int B, int H, int Hkv, int Nq, int Nk, int d, float scale, int num_splits,
                            void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of device workspace fa_fwd_materialized needs: the bf16 score /
 * probability matrix [B, H, Nq, Nk], rounded up to 256 bytes. 0 for invalid
 * arguments. */
size_t fa_materialized_workspace_size(int B, int H, int Nq, int Nk);

/* The materialising baseline the IO argument compares against ("Explain
 * FlashAttention ...", section "What the byte arithmetic does and does not
 * say"): S = scale * Q K^T is written to HBM in bf16, read back by a row
 * softmax that writes P (bf16, over S), and P is read again for O = P V.
 * Four N^2-sized transfers of 2-byte values, against the fused fa_fwd's
 * none. It computes the same attention as fa_fwd (without a key mask), with
 * S and P rounded to bf16. The two products are cuBLAS GEMMs (the library
 * opens libcublas.so.13 on first use and keeps one cuBLAS handle per device;
 * calls are serialised inside the library); the softmax is this library's
 * kernel.
 *   q, o      bf16 [B, H, Nq, d]       k, v  bf16 [B, H, Nk, d]
 *   lse       fp32 [B, H, Nq] (natural log; may be NULL)
 *   workspace device memory of at least fa_materialized_workspace_size()
 *             bytes, 256-byte aligned, owned by the caller; overwritten.
 * Errors: as for fa_fwd, plus FA_ERR_UNSUPPORTED when Nk is not a multiple of
 * 8 or exceeds the row held in one CTA's shared memory (about 58k keys), or
 * when cuBLAS cannot be loaded; FA_ERR_WORKSPACE. */
fa_status fa_fwd_materialized(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Nq,
                              int Nk, int d, float scale, int causal, void* workspace, size_t workspace_bytes,
                              void* stream);

/* Bytes of device workspace fa_bwd needs: an fp32 dQ accumulator of
 * B*H*ceil(Nq/128)*128*d elements (Nq padded to whole 128-row tiles) and two
 * fp32 per-row statistics [B, H, Nq], each rounded up to 256 bytes. Returns 0
 * for invalid arguments. */
size_t fa_bwd_workspace_size(int B, int H, int Nq, int d);

/* Backward pass of fa_fwd (no key mask): given dout = dL/dO, writes
 * dq = dL/dQ, dk = dL/dK and dv = dL/dV for the same q, k, v, scale and
 * causal flag. The probability tiles are recomputed from the forward's lse
 * instead of being stored ("Flash Attention Optimization", section "Sizing a
 * tile, and why the backward pass recomputes instead of storing"; "Explain
 * FlashAttention ...", section "Exact attention, finite precision and
 * backward"): with P = exp(scale Q K^T - lse) over the visible keys and
 * D_i = sum_c dout_ic o_ic,
 *   dv = P^T dout,  dS = P * (dout V^T - D),  dq = scale dS K,  dk = scale dS^T Q.
 *   q, o, dout, dq  bf16 [B, H, Nq, d]     k, v, dk, dv  bf16 [B, H, Nk, d]
 *   lse             fp32 [B, H, Nq], as written by fa_fwd for these inputs
 *   workspace       device memory of at least fa_bwd_workspace_size() bytes,
 *                   256-byte aligned, owned by the caller; overwritten.
 * Requires B, H, Nq, Nk >= 1, d in {64, 128}, 16-byte aligned bf16 buffers,
 * a finite scale. Keys no visible query reaches get dk = dv = 0. Three
 * launches on `stream` (statistics, the fused tiles, dq conversion); errors
 * as for fa_fwd, plus FA_ERR_WORKSPACE. */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                 void* dq, void* dk, void* dv, int B, int H, int Nq, int Nk, int d, float scale, int causal,
                 void* workspace, size_t workspace_bytes, void* stream);

/* Synchronises `stream`, then returns and clears the device status word of
 * the current device: FA_ERR_TIMEOUT if a bounded wait gave up since the
 * last call, FA_ERR_CUDA if the stream reported an error, else FA_OK. */
fa_status fa_get_device_status(void* stream);

/* Limit, in nanoseconds, on every wait inside the library's kernels
 * (default 2e9). Applies to calls launched afterwards. */
void fa_set_wait_limit_ns(uint64_t ns);
uint64_t fa_get_wait_limit_ns(void);

/* Self-test of the failure path: launches one warp that waits on a barrier
 * nothing ever arrives on, with the given limit; returns what
 * fa_get_device_status() then reports (FA_ERR_TIMEOUT when the bounded wait
 * works). The context stays usable afterwards. */
fa_status fa_selftest_wait_timeout(uint64_t limit_ns, void* stream);

/* Self-test of the device exponential the prefill softmax runs on the FMA
 * pipe for part of each score tile: y[i] = 2^x[i] for x[i] in [-126, 127]
 * (device pointers, fp32, asynchronous on `stream`). Its maximum relative
 * error is 7.5e-5, far below the bf16 rounding applied to P. */
fa_status fa_selftest_exp2(const float* x, float* y, int n, void* stream);

/* Human-readable name of a status code. */
const char* fa_status_string(fa_status s);

/* Detail of the most recent error returned on the calling host thread
 * (empty string if none). */
const char* fa_last_error_detail(void);

/* Number of kernel launches this library issued on the calling host thread
 * since the process started (for accounting in benchmarks). */
uint64_t fa_launch_count(void);

/* Debug build (the pages have no counterpart: this checks the implementation).
 * libfa_gb300_debug.so is the same library compiled with FA_DEBUG=1: its
 * prefill kernels check, before each access, the coordinates of every TMA
 * copy (x on a 16-byte boundary and inside the row, the tile starting inside
 * the tensor, the batch-head index in range), the TMEM lanes and columns of
 * every tensor-memory load, store and product, and at the end of a launch that
 * every barrier completed as many phases as its users counted. A failed check
 * skips the access and records the failure; nothing traps. The release
 * library compiles the checks out.
 *   fa_debug_enabled()   1 in the debug build, 0 in the release build.
 *   fa_debug_record(out) waits for `stream`, copies the current device's
 *                        8-word record to host `out` and clears it: word 0
 *                        bits (1 = TMA coordinate, 2 = TMEM range, 4 =
 *                        barrier phase count), then the first failure's site,
 *                        block, thread and three values, then the number of
 *                        failed checks.
 *   fa_debug_selftest()  launches one warp that runs every check on values it
 *                        must reject, with no access; afterwards the debug
 *                        build's record holds bits 1, 2 and 4. */
int fa_debug_enabled(void);
fa_status fa_debug_record(uint32_t* out, void* stream);
fa_status fa_debug_selftest(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
