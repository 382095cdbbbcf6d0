// Internal interface between the C-ABI layer (pa_abi.cu) and the kernel
// translation units. Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

struct StoreArgs {
  const void* k;
  const void* v;
  const float* k_scale_new;
  const float* v_scale_new;
  const int64_t* slot_mapping;
  void* k_cache;
  void* v_cache;
  float* k_scale;
  float* v_scale;
  int num_tokens;
  int row_bytes;     // num_kv_heads * head_dim * element size
  int num_kv_heads;
  int block_size;
  long long num_slots;  // num_blocks * block_size
  uint32_t* err;
};

cudaError_t launch_store_kv(const StoreArgs& a, cudaStream_t stream);

// Append each sequence's new token at position context_lens[b]-1 (slot from
// the block table): used by the fused append when the persistent decode does
// not apply. `a.slot_mapping` is ignored; the cache fields of `a` are used.
cudaError_t launch_store_new_tokens(const StoreArgs& a, const int32_t* block_tables,
                                    int max_blocks, const int32_t* context_lens, int len_cap,
                                    cudaStream_t stream);

// Largest batch the persistent decode kernel handles (its per-sequence block
// prefix sums live in shared memory); larger batches use the grid-split kernel.
// KV element kinds (the pa_kv_dtype values): bf16, or 8-bit codes with
// per-(slot, head) scales in E4M3 or INT8.
constexpr int kKvBf16 = 0, kKvE4m3 = 1, kKvInt8 = 2;

constexpr int kMaxPersistentBatch = 16384;

struct DecodeArgs {
  const void* q;              // (B, H, D) bf16
  const int32_t* block_tables;
  const int32_t* context_lens;
  const float* k_scale;       // 8-bit caches: (NB, Hkv, bs)
  const float* v_scale;
  void* out;                  // (B, H, D) bf16
  float* part_o;              // partial slots: (slots, 8, D) fp32
  float* part_ml;             // (slots, 8, 2) fp32: (max, sum) per head
  int* prefix_out;            // persistent path: (B+1) block prefix sums
  unsigned long long* seg_counters;  // persistent path: (B*Hkv) arrival counters
  unsigned long long* grp_counters;  // persistent path: one per partial slot (merge groups)
  uint32_t epoch;             // persistent path: tag of this call in seg_counters
  int slot_rows;              // rows (query heads) of one partial slot
  uint32_t* err;
  // fused append (pa_decode_append): the new token of sequence b, at position
  // context_lens[b]-1, is written to the cache by the warp that attends to it
  const void* k_new;          // (B, Hkv, D) cache dtype, or NULL
  const void* v_new;
  const float* k_scale_new;   // 8-bit caches: (B, Hkv)
  const float* v_scale_new;
  void* k_cache;              // cache base pointers (written when appending)
  void* v_cache;
  int batch, num_heads, num_kv_heads, group, head_dim, block_size;
  int max_blocks, num_blocks, len_cap;
  int window, sinks;          // sliding window (> 0) with leading sink keys; 0 = all keys
  int persistent_ctas;        // > 0: persistent kernel with this many CTAs
  int blocks_per_split, num_splits;  // grid-split path
  int kv;                     // kKvBf16, kKvE4m3 or kKvInt8
  float scale_log2;
  unsigned long long wait_limit_ns;  // bound of every wait on a copy
  // failure-detection test hook (pa_debug_inject_wait_timeout), -1 when off:
  // the first warp of CTA 0 never issues its copy number debug_skip_copy, so
  // its wait for that block runs out
  int debug_skip_copy;
};

// Plan of a decode call: persistent (CTA count, 2 partial slots per CTA) or
// grid-split (blocks per split, number of splits, one slot per split).
struct DecodePlan {
  int persistent_ctas;
  int blocks_per_split;
  int num_splits;
  size_t partial_slots;  // fp32 partials of slot_rows x (head_dim + 2) floats each
  int slot_rows;
  size_t workspace_bytes;
};

DecodePlan plan_decode(int batch, int num_heads, int num_kv_heads, int head_dim, int block_size,
                       int kv, int len_cap, int num_sms);

cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          cudaStream_t stream);

// Bytes of one TMA box row (the innermost box extent): the kernels stage K/V
// as 128-byte-wide, 128B-swizzled tiles.
constexpr int kSwizzleBytes = 128;

}  // namespace pa
