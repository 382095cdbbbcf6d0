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

struct DecodeArgs {
  const void* q;              // (B, H, D) bf16
  const int32_t* block_tables;
  const int32_t* context_lens;
  const float* k_scale;       // FP8: (NB, Hkv, bs)
  const float* v_scale;
  void* out;                  // (B, H, D) bf16
  float* part_o;              // (B, H, S, D) fp32
  float* part_ml;             // (B, H, S, 2) fp32
  uint32_t* err;
  int batch, num_heads, num_kv_heads, group, head_dim, block_size;
  int max_blocks, num_blocks, len_cap;
  int blocks_per_split, num_splits;
  bool fp8;
  float scale_log2;
};

// Split-K plan of a decode call: blocks per split and number of splits.
struct DecodePlan {
  int blocks_per_split;
  int num_splits;
  size_t workspace_bytes;
};

DecodePlan plan_decode(int batch, int num_heads, int num_kv_heads, int head_dim, int block_size,
                       bool fp8, int len_cap, int num_sms);

cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          cudaStream_t stream);

// Bytes of one TMA box row (the innermost box extent): the kernels stage K/V
// as 128-byte-wide, 128B-swizzled tiles.
constexpr int kSwizzleBytes = 128;

}  // namespace pa
