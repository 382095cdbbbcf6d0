/*
 * pa.h - C ABI of the GB300 (sm_103a) paged-KV-cache attention library.
 *
 * The operations, as the source pages define them:
 *   pa_store_kv        append new tokens' K/V to their cache slots
 *                      ("tiny-vllm part 05", section "Gathering K/V into a
 *                      batched buffer and scattering into blocks"; the
 *                      store_kvcache step of "Decode Phase Attention Forward
 *                      Pass", section 2).
 *   pa_decode          one query per sequence attending over exactly
 *                      context_len cached keys, read through the block table,
 *                      with GQA head grouping ("Decode Phase Attention Forward
 *                      Pass", sections 2-4 and the zero-padding caveat;
 *                      "Decode Phase" glossary, the q.K^T / softmax / sum-of-V
 *                      steps).
 *   pa_decode_window   pa_decode over a sliding window plus leading sink keys
 *                      ("Decode Phase" glossary, long-context bullets).
 *   pa_decode_append   pa_store_kv of each sequence's new token followed by
 *                      pa_decode, fused into one persistent kernel.
 *   pa_prefill_varlen  packed varlen prefill over a prefix already in the
 *                      paged cache, bottom-right-aligned causal mask
 *                      ("Prefill Forward Prefix Caching Explained", Facts 1-2
 *                      and the mask section).
 *
 * Conventions shared by every call
 *   - Every tensor pointer is a DEVICE pointer owned by the caller. The
 *     library never calls a device allocator: pa_decode's split-K scratch is
 *     passed in as `workspace` (pa_decode_noalloc uses a static buffer).
 *   - All calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *     NULL = the legacy default stream) and never synchronise the host.
 *     Decode launches may start while the previous launch of this library on
 *     the stream is finishing (programmatic dependent launch): they read
 *     context_lens and block_tables before waiting for it, and everything
 *     else after. No kernel of this library writes those two arrays; a
 *     caller's own kernel that writes them and lets its dependents start
 *     early must not directly precede a decode call.
 *   - Argument errors are returned before anything is launched. A launch
 *     failure returns PA_ERR_CUDA. Out-of-range indices found on the device
 *     (a slot beyond the pool, a wait that timed out) never fault: the access
 *     is skipped and a bit is set in a per-device error word, read with
 *     pa_get_device_error().
 *   - Layouts (row-major, contiguous):
 *       k_cache, v_cache  (num_blocks, block_size, num_kv_heads, head_dim)
 *                         bf16, FP8-E4M3 bytes (OCP "e4m3fn") or signed INT8
 *                         codes (the "Decode Phase" glossary names FP8 and
 *                         INT8 KV-cache quantisation);
 *       k_scale, v_scale  (num_blocks, num_kv_heads, block_size) fp32, 8-bit
 *                         caches only: element = code value * scale;
 *       block_tables      (batch, max_blocks_per_seq) int32, physical block
 *                         of logical block j of sequence b;
 *       slot              physical_block * block_size + offset (int64).
 *   - Head map (GQA/MQA): query head h reads kv head h / (num_heads /
 *     num_kv_heads), i.e. the repeat_interleave grouping of the decode page.
 *   - Supported: head_dim 64 or 128 (8-bit caches: 128), block_size 16 or 32,
 *     num_heads a multiple of num_kv_heads with at most 8 query heads per kv
 *     head. Anything else returns PA_ERR_UNSUPPORTED.
 */
#ifndef PA_GB300_H
#define PA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PA_ABI_VERSION 1

typedef enum {
  PA_OK = 0,
  PA_ERR_NULL = 1,        /* a required pointer is NULL */
  PA_ERR_SHAPE = 2,       /* a size is negative/zero where it must not be, or inconsistent */
  PA_ERR_DTYPE = 3,       /* cache dtype / scale pointers do not match */
  PA_ERR_UNSUPPORTED = 4, /* valid but not implemented (head_dim, block_size, group size) */
  PA_ERR_CUDA = 5,        /* a CUDA runtime/driver call or a launch failed */
  PA_ERR_WORKSPACE = 6,   /* workspace missing or smaller than pa_decode_workspace_size() */
  PA_ERR_ALIGN = 7,       /* a pointer is not 16-byte aligned */
  PA_ERR_TOO_LARGE = 8    /* pa_decode_noalloc: the shape needs more scratch than the
                             library's static buffer holds */
} pa_status;

typedef enum { PA_KV_BF16 = 0, PA_KV_FP8_E4M3 = 1, PA_KV_INT8 = 2 } pa_kv_dtype;

/* Device error word bits (pa_get_device_error). */
#define PA_DEVERR_SLOT_RANGE 0x1u   /* store_kv: slot >= num_blocks*block_size, skipped */
#define PA_DEVERR_WAIT_TIMEOUT 0x2u /* a kernel's bounded wait on a copy gave up */
#define PA_DEVERR_BLOCK_RANGE 0x4u  /* block table entry outside [0, num_blocks), zero-filled */

/* A paged KV cache (one layer). Pointers are device pointers; the struct
 * itself is read on the host during the call and may live on the stack. */
typedef struct {
  int32_t num_blocks;   /* physical blocks in the pool */
  int32_t block_size;   /* tokens per block: 16 or 32 */
  int32_t num_kv_heads;
  int32_t head_dim;     /* 64 or 128 */
  int32_t dtype;        /* pa_kv_dtype */
  void* k_cache;        /* (num_blocks, block_size, num_kv_heads, head_dim) */
  void* v_cache;
  float* k_scale;       /* (num_blocks, num_kv_heads, block_size), 8-bit only, else NULL */
  float* v_scale;
} pa_kv_cache;

/* ABI version of the loaded library (PA_ABI_VERSION it was built with). */
int32_t pa_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* pa_status_string(pa_status status);

/*
 * pa_store_kv - write num_tokens new K/V rows into the cache.
 *   k, v           (num_tokens, num_kv_heads, head_dim), cache dtype (bf16, or
 *                  E4M3 / INT8 bytes for an 8-bit cache), device.
 *   k_scale_new,   (num_tokens, num_kv_heads) fp32, 8-bit caches only (else NULL).
 *   v_scale_new
 *   slot_mapping   (num_tokens) int64: destination slot of token t; a negative
 *                  slot skips the token (padding). Slots within one call must
 *                  be distinct (otherwise which write wins is unspecified).
 *   Bytes are copied unchanged (bit-exact). A slot >= num_blocks*block_size is
 *   skipped and flagged PA_DEVERR_SLOT_RANGE. num_tokens == 0 is a no-op.
 */
pa_status pa_store_kv(const void* k, const void* v, const float* k_scale_new,
                      const float* v_scale_new, const int64_t* slot_mapping, int32_t num_tokens,
                      const pa_kv_cache* cache, void* stream);

/*
 * pa_decode_workspace_size - bytes of device scratch pa_decode needs for this
 * shape (split-K partial results). 0 means pa_decode needs no workspace.
 * max_context_len is the same host-side bound that will be passed to
 * pa_decode (<= 0: the block-table capacity max_blocks_per_seq*block_size).
 */
size_t pa_decode_workspace_size(const pa_kv_cache* cache, int32_t batch, int32_t num_heads,
                                int32_t max_blocks_per_seq, int32_t max_context_len);

/*
 * pa_decode - single-query attention over a paged KV cache.
 *   q               (batch, num_heads, head_dim) bf16.
 *   block_tables    (batch, max_blocks_per_seq) int32; only the first
 *                   ceil(context_len/block_size) entries of a row are read.
 *   context_lens    (batch) int32 on the device: keys 0..context_len-1 of each
 *                   sequence are attended (the token stored this step
 *                   included). context_len 0 gives a zero output row.
 *   max_context_len host-side upper bound of every context_len (sizes the
 *                   split-K grid; <= 0 means max_blocks_per_seq*block_size).
 *                   Keys at positions >= this bound are not attended.
 *   scale           softmax scale applied to q.k.
 *   out             (batch, num_heads, head_dim) bf16.
 *   workspace       device scratch of at least pa_decode_workspace_size()
 *                   bytes (may be NULL when that is 0). Contents on entry are
 *                   ignored, up to a 2^-32 chance per stale 64-bit word of
 *                   carrying the call's tag; calls sharing one workspace must
 *                   not overlap.
 *                   The split-K arrival counters in it carry a per-call
 *                   32-bit tag (unrelated from call to call) and each is
 *                   cleared by its last arrival, so a CUDA graph
 *                   that captured the call can be replayed back to back on
 *                   the same workspace (its tag is frozen at capture). After
 *                   a launch that reported PA_DEVERR_WAIT_TIMEOUT, counters
 *                   of unfinished segments stay set: make one uncaptured call
 *                   on the workspace before replaying such a graph again.
 * Arithmetic: bf16 (or E4M3 / INT8 codes widened exactly to f16) operands, fp32 scores,
 * softmax and accumulation, one round to bf16 at the output.
 */
pa_status pa_decode(const void* q, const pa_kv_cache* cache, const int32_t* block_tables,
                    int32_t max_blocks_per_seq, const int32_t* context_lens,
                    int32_t max_context_len, int32_t batch, int32_t num_heads, float scale,
                    void* out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * pa_decode_window - pa_decode restricted to a sliding window with attention
 * sinks ("Decode Phase" glossary, the long-context bullets: sliding window
 * attention over the most recent W tokens; attention sinks as in
 * StreamingLLM, keeping the initial tokens). For a sequence of L =
 * context_len keys the query attends to keys p < sinks and p >= L - window.
 *   window   > 0: window size in keys; <= 0: all keys (same as pa_decode,
 *            sinks ignored).
 *   sinks    >= 0: leading keys always attended (PA_ERR_SHAPE if negative).
 *   other arguments as pa_decode (same workspace size). Blocks that hold no
 *   visible key are not read. Batches above 16384 return PA_ERR_UNSUPPORTED.
 */
pa_status pa_decode_window(const void* q, const pa_kv_cache* cache, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* context_lens,
                           int32_t max_context_len, int32_t batch, int32_t num_heads,
                           float scale, int32_t window, int32_t sinks, void* out, void* workspace,
                           size_t workspace_bytes, void* stream);

/*
 * pa_decode_append - one decode step's store and attention in one call: the
 * store_kvcache step (each sequence's new K/V row written to the cache) then
 * attention over context_len keys, new token included ("Decode Phase
 * Attention Forward Pass", section 2, the store-then-attend order).
 *   k_new, v_new    (batch, num_kv_heads, head_dim), cache dtype, device,
 *                   16-byte aligned: the new token of sequence b.
 *   k_scale_new,    (batch, num_kv_heads) fp32, 8-bit caches only (else NULL).
 *   v_scale_new
 *   other arguments as pa_decode (same workspace size).
 * The row goes to position p = min(context_len, bound) - 1 of its sequence,
 * i.e. slot block_tables[b][p / block_size] * block_size + p % block_size,
 * where bound is max_context_len (or the block-table capacity); a sequence
 * with context_len 0 appends nothing. Result and cache contents are those of
 * pa_store_kv with that slot mapping followed by pa_decode. The block holding
 * position p must not be read by another sequence of the same call. A
 * physical block id out of range skips the write and sets
 * PA_DEVERR_BLOCK_RANGE. With the persistent kernel (batch <= 16384) the warp
 * that attends to a sequence's last block also writes the row; larger batches
 * use a separate store launch first.
 */
pa_status pa_decode_append(const void* q, const void* k_new, const void* v_new,
                           const float* k_scale_new, const float* v_scale_new,
                           const pa_kv_cache* cache, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* context_lens,
                           int32_t max_context_len, int32_t batch, int32_t num_heads,
                           float scale, void* out, void* workspace, size_t workspace_bytes,
                           void* stream);

/*
 * pa_decode_window_append - pa_decode_append with the sliding window and
 * attention sinks of pa_decode_window: the new row is written as by
 * pa_decode_append, then each query attends to the keys pa_decode_window
 * selects (the new token, at position context_len - 1, is always among them).
 * Result and cache contents are those of pa_store_kv followed by
 * pa_decode_window; window 0 is pa_decode_append. Same arguments as
 * pa_decode_append plus window and sinks (as pa_decode_window); batches above
 * 16384 return PA_ERR_UNSUPPORTED, as for pa_decode_window.
 */
pa_status pa_decode_window_append(const void* q, const void* k_new, const void* v_new,
                                  const float* k_scale_new, const float* v_scale_new,
                                  const pa_kv_cache* cache, const int32_t* block_tables,
                                  int32_t max_blocks_per_seq, const int32_t* context_lens,
                                  int32_t max_context_len, int32_t batch, int32_t num_heads,
                                  float scale, int32_t window, int32_t sinks, void* out,
                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * pa_prefill_varlen - prefill attention of packed new tokens over their
 * sequences' paged K/V (cached prefix + the new tokens, which must already be
 * stored with pa_store_kv), with the bottom-right-aligned causal mask: query
 * row i of a sequence (0-based) sees keys j <= i + (kv_len - q_len).
 *   q               (total_q, num_heads, head_dim) bf16, sequences packed.
 *   block_tables    (batch, max_blocks_per_seq) int32.
 *   cu_seqlens_q    (batch+1) int32 on the device, prefix sums of q_len
 *                   (cu_seqlens_q[0] = 0, cu_seqlens_q[batch] = total_q).
 *   cu_seqlens_k    (batch+1) int32 on the device, prefix sums of kv_len.
 *   total_q         packed rows of q/out (host-side).
 *   max_q_len       host-side bound of every q_len (sizes the grid; <= 0 means
 *                   total_q). Rows past this bound are not computed.
 *   scale           softmax scale, > 0.
 *   out             (total_q, num_heads, head_dim) bf16.
 * A sequence with q_len > kv_len is invalid input: its cached length is taken
 * as 0 and keys are clamped to kv_len. Supported: bf16 cache, head_dim 128,
 * block_size 16 or 32, num_heads/num_kv_heads in {1, 2, 4, 8, 16}.
 * Arithmetic: bf16 operands on the tensor cores, fp32 scores and
 * accumulation, probabilities rounded to bf16 for P.V (as two bf16 terms,
 * bf16(p) + bf16(p - bf16(p)), on the first 128 keys of the query tiles that
 * hold rows seeing fewer than 128 keys), bf16 output.
 */
pa_status pa_prefill_varlen(const void* q, const pa_kv_cache* cache, const int32_t* block_tables,
                            int32_t max_blocks_per_seq, const int32_t* cu_seqlens_q,
                            const int32_t* cu_seqlens_k, int32_t batch, int32_t num_heads,
                            int32_t total_q, int32_t max_q_len, float scale, void* out,
                            void* stream);

/*
 * pa_decode_noalloc - pa_decode for callers that cannot allocate device memory.
 * The pages have no counterpart: this entry point exists for callers with no
 * device allocator of their own (a plain C host program handed device
 * pointers by another runtime) or whose device memory is fully reserved (a
 * serving engine's KV-block pool), for whom a scratch cudaMalloc is not an
 * option. Same arguments and result as pa_decode, minus the workspace: the
 * split-K scratch is a static device buffer of
 * PA_DECODE_NOALLOC_SCRATCH_BYTES inside the library, held by every GPU that
 * loads it until the process exits. Allocates nothing per call (no cudaMalloc,
 * cudaFree or allocating library routine).
 *   - Shapes whose pa_decode_workspace_size() exceeds the buffer are rejected
 *     with PA_ERR_TOO_LARGE before anything is launched.
 *   - The first call on a device (with it current) looks up the buffer's
 *     device address; make that first call before any stream capture.
 *   - All calls share the buffer and it keeps the last call's contents (the
 *     kernels write every partial they read, so nothing needs clearing). Calls
 *     that may overlap on the GPU race on it: serialise them.
 */
#define PA_DECODE_NOALLOC_SCRATCH_BYTES (32u << 20) /* 32 MiB */
pa_status pa_decode_noalloc(const void* q, const pa_kv_cache* cache, const int32_t* block_tables,
                            int32_t max_blocks_per_seq, const int32_t* context_lens,
                            int32_t max_context_len, int32_t batch, int32_t num_heads,
                            float scale, void* out, void* stream);

/*
 * pa_get_device_error - synchronise the current device, return its error word
 * (PA_DEVERR_* bits, 0 if none) in *code and clear it.
 */
pa_status pa_get_device_error(uint32_t* code);

/*
 * pa_debug_inject_wait_timeout - test hook for the failure-detection path; the
 * pages have no counterpart. Every wait of a decode kernel on a copy is
 * bounded (2 s by default); after the bound it records PA_DEVERR_WAIT_TIMEOUT,
 * lets the copies it has in flight land (each wait bounded again) and returns,
 * so the context stays usable. This hook makes that happen on purpose without
 * faulting anything: while armed (skip_copy >= 0), decode launches of this
 * process (persistent kernel, batch <= 16384; pa_decode, pa_decode_window,
 * pa_decode_append) wait at most wait_limit_ns (1 .. 2e9) per copy, and in
 * each launch the first warp of the first CTA never issues its skip_copy-th
 * block copy (counted from 0 in its own block order), so its wait for that
 * block runs out. Outputs of such a launch are invalid. skip_copy < 0
 * disarms the hook and restores the 2 s bound (wait_limit_ns ignored).
 * Process-wide, not thread-safe against concurrent decode calls: arm, run
 * one call, disarm. Returns PA_ERR_SHAPE for a bound outside 1 .. 2e9.
 */
pa_status pa_debug_inject_wait_timeout(int32_t skip_copy, uint64_t wait_limit_ns);

#ifdef __cplusplus
}
#endif

#endif /* PA_GB300_H */
