// pa_decode_noalloc: pa_decode for callers that cannot allocate device memory.
//
// pa_decode needs split-K scratch (per-split partial max, sum and output) when
// a sequence spans more than one split, and asks the caller for it. Some
// callers cannot provide it: a plain C host program that only receives device
// pointers from another runtime and has no device allocator of its own, or a
// serving engine that has reserved nearly all device memory for its KV-block
// pool, where an extra cudaMalloc would fail or stall the device. This entry
// point takes its scratch from a fixed-size buffer that lives in the library
// itself, so it allocates nothing per call.
//
// The buffer is a file-scope __device__ array: every GPU that loads this part
// of the library holds kNoAllocScratchBytes of device memory until the process
// exits. Host code cannot use the array's name as a device address, so the
// first call on each device (with that device current) looks the address up
// with cudaGetSymbolAddress and keeps it; make that first call before any
// stream capture. All calls share the one buffer and it keeps the previous
// call's contents; the decode kernels write every partial they read, so no
// clearing is needed. Calls whose kernels may overlap on the GPU (different
// streams, or different host threads) race on the buffer and must be
// serialised by the caller.
#include <cuda_runtime.h>

#include <mutex>

#include "pa.h"

namespace {

constexpr size_t kNoAllocScratchBytes = PA_DECODE_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once per
// device, on its first call).
pa_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return PA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_noalloc(const void* q, const pa_kv_cache* cache,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* context_lens, int32_t max_context_len,
                                       int32_t batch, int32_t num_heads, float scale, void* out,
                                       void* stream) {
  if (cache == nullptr) return PA_ERR_NULL;
  if (batch > 0 && num_heads > 0 && max_blocks_per_seq > 0) {
    const size_t need =
        pa_decode_workspace_size(cache, batch, num_heads, max_blocks_per_seq, max_context_len);
    if (need > kNoAllocScratchBytes) return PA_ERR_TOO_LARGE;
  }
  void* scratch = nullptr;
  const pa_status st = scratch_for_current_device(&scratch);
  if (st != PA_OK) return st;
  return pa_decode(q, cache, block_tables, max_blocks_per_seq, context_lens, max_context_len,
                   batch, num_heads, scale, out, scratch, kNoAllocScratchBytes, stream);
}
