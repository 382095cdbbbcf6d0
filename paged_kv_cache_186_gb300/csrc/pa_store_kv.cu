// store_kv: append new tokens' K/V rows to their paged-cache slots.
//
// "tiny-vllm part 05", section "Gathering K/V into a batched buffer and
// scattering into blocks": the token at position p goes to logical block
// p / BLOCK_SIZE, offset p % BLOCK_SIZE of its sequence; the page's engine
// does this with two device-to-device copies per token. Here the caller
// supplies the resolved slot (physical_block * block_size + offset) and one
// warp moves a token's K and V rows with 16-byte vector accesses, so a whole
// decode batch (or a prefill chunk) is one launch.
#include "pa_device.cuh"
#include "pa_launch.h"

namespace pa {

namespace {

constexpr int kStoreWarps = 4;

// A token's K and V rows (n16 16-byte chunks each) copied by one warp: every
// lane first issues the loads of all its chunks (up to kChunksPerLane each of
// K and V per round), then the stores, so a row costs one load round trip
// instead of one per 512 bytes (the loads of a round could not pass the
// stores of the previous one: the cache may alias the inputs).
constexpr int kChunksPerLane = 8;
__device__ __forceinline__ void copy_rows(const uint4* ks, const uint4* vs, uint4* kd, uint4* vd,
                                          int n16, int lane) {
  for (int base = 0; base < n16; base += 32 * kChunksPerLane) {
    uint4 kb[kChunksPerLane], vb[kChunksPerLane];
#pragma unroll
    for (int j = 0; j < kChunksPerLane; ++j) {
      const int i = base + lane + 32 * j;
      if (i < n16) {
        kb[j] = __ldg(ks + i);
        vb[j] = __ldg(vs + i);
      }
    }
#pragma unroll
    for (int j = 0; j < kChunksPerLane; ++j) {
      const int i = base + lane + 32 * j;
      if (i < n16) {
        kd[i] = kb[j];
        vd[i] = vb[j];
      }
    }
  }
}

__global__ void __launch_bounds__(kStoreWarps * 32) store_kv_kernel(const StoreArgs a) {
  grid_launch_dependents();  // a following decode/prefill may start its prologue
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kStoreWarps + warp;
  if (t >= a.num_tokens) return;
  const long long slot = a.slot_mapping[t];
  if (slot < 0) return;  // padding token
  if (slot >= a.num_slots) {
    if (lane == 0) report_error(a.err, PA_DEVERR_SLOT_RANGE);
    return;
  }
  const int n16 = a.row_bytes >> 4;
  const uint4* ks = reinterpret_cast<const uint4*>(static_cast<const char*>(a.k) +
                                                   static_cast<long long>(t) * a.row_bytes);
  const uint4* vs = reinterpret_cast<const uint4*>(static_cast<const char*>(a.v) +
                                                   static_cast<long long>(t) * a.row_bytes);
  uint4* kd = reinterpret_cast<uint4*>(static_cast<char*>(a.k_cache) + slot * a.row_bytes);
  uint4* vd = reinterpret_cast<uint4*>(static_cast<char*>(a.v_cache) + slot * a.row_bytes);
  copy_rows(ks, vs, kd, vd, n16, lane);
  if (a.k_scale != nullptr) {
    // scales: new (T, Hkv) -> cache (num_blocks, Hkv, block_size)
    const long long blk = slot / a.block_size, off = slot % a.block_size;
    for (int h = lane; h < a.num_kv_heads; h += 32) {
      const long long dst = (blk * a.num_kv_heads + h) * a.block_size + off;
      a.k_scale[dst] = a.k_scale_new[static_cast<long long>(t) * a.num_kv_heads + h];
      a.v_scale[dst] = a.v_scale_new[static_cast<long long>(t) * a.num_kv_heads + h];
    }
  }
}

// One warp per sequence: slot of position context_len-1 from the block table,
// then the same row copies as store_kv_kernel.
__global__ void __launch_bounds__(kStoreWarps * 32)
    store_new_tokens_kernel(const StoreArgs a, const int32_t* block_tables, int max_blocks,
                            const int32_t* context_lens, int len_cap) {
  grid_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kStoreWarps + warp;
  if (t >= a.num_tokens) return;
  const int L = min(context_lens[t], len_cap);
  if (L <= 0) return;
  const int logical = (L - 1) / a.block_size;
  if (logical >= max_blocks) return;
  const long long phys = block_tables[static_cast<long long>(t) * max_blocks + logical];
  const long long slot = phys * a.block_size + (L - 1) % a.block_size;
  if (phys < 0 || slot >= a.num_slots) {
    if (lane == 0) report_error(a.err, PA_DEVERR_BLOCK_RANGE);
    return;
  }
  const int n16 = a.row_bytes >> 4;
  const uint4* ks = reinterpret_cast<const uint4*>(static_cast<const char*>(a.k) +
                                                   static_cast<long long>(t) * a.row_bytes);
  const uint4* vs = reinterpret_cast<const uint4*>(static_cast<const char*>(a.v) +
                                                   static_cast<long long>(t) * a.row_bytes);
  uint4* kd = reinterpret_cast<uint4*>(static_cast<char*>(a.k_cache) + slot * a.row_bytes);
  uint4* vd = reinterpret_cast<uint4*>(static_cast<char*>(a.v_cache) + slot * a.row_bytes);
  copy_rows(ks, vs, kd, vd, n16, lane);
  if (a.k_scale != nullptr) {
    const long long off = slot % a.block_size;
    for (int h = lane; h < a.num_kv_heads; h += 32) {
      const long long dst = (phys * a.num_kv_heads + h) * a.block_size + off;
      a.k_scale[dst] = a.k_scale_new[static_cast<long long>(t) * a.num_kv_heads + h];
      a.v_scale[dst] = a.v_scale_new[static_cast<long long>(t) * a.num_kv_heads + h];
    }
  }
}

}  // namespace

cudaError_t launch_store_new_tokens(const StoreArgs& a, const int32_t* block_tables,
                                    int max_blocks, const int32_t* context_lens, int len_cap,
                                    cudaStream_t stream) {
  if (a.num_tokens <= 0) return cudaSuccess;
  const int grid = (a.num_tokens + kStoreWarps - 1) / kStoreWarps;
  store_new_tokens_kernel<<<grid, kStoreWarps * 32, 0, stream>>>(a, block_tables, max_blocks,
                                                                 context_lens, len_cap);
  return cudaGetLastError();
}

cudaError_t launch_store_kv(const StoreArgs& a, cudaStream_t stream) {
  if (a.num_tokens <= 0) return cudaSuccess;
  const int grid = (a.num_tokens + kStoreWarps - 1) / kStoreWarps;
  store_kv_kernel<<<grid, kStoreWarps * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pa
