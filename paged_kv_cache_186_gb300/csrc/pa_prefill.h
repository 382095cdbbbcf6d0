// Internal interface of the prefill kernel (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

struct PrefillArgs {
  const int32_t* block_tables;  // (B, max_blocks)
  const int32_t* cu_q;          // (B+1)
  const int32_t* cu_k;          // (B+1)
  void* out;                    // (total_q, H, D) bf16
  uint32_t* err;
  int batch, num_heads, num_kv_heads, group, head_dim, block_size;
  int max_blocks, num_blocks;
  int tokens_per_tile;  // 128 / group query tokens per 128-row tile
  int num_qtiles;       // tiles per sequence in the grid (from the max q_len bound)
  float scale_log2;
};

// Query tokens per 128-row tile for a head group of `group` query heads.
int prefill_tokens_per_tile(int group);

cudaError_t launch_prefill(const PrefillArgs& a, const CUtensorMap& qmap, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, cudaStream_t stream);

}  // namespace pa
