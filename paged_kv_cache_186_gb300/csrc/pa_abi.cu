// C-ABI entry points: argument validation, tensor-map encoding, launch.
// Every check happens on the host before any launch; nothing here reads
// device memory or synchronises (except pa_get_device_error).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <atomic>
#include <mutex>

#include "pa.h"
#include "pa_device.cuh"
#include "pa_launch.h"
#include "pa_prefill.h"

namespace {

// Per-device error word (PA_DEVERR_* bits), set by kernels with atomicOr.
__device__ uint32_t g_device_error;

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  uint32_t* err = nullptr;
  int num_sms = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Resolve per-device state (error-word address, SM count) for the current
// device; the first call on a device does the lookup.
pa_status device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return PA_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return PA_ERR_CUDA;
    d.err = static_cast<uint32_t*>(p);
    d.num_sms = sms;
    d.ready = true;
  }
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return PA_ERR_CUDA;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  }
  *out = &d;
  return PA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

pa_status check_cache(const pa_kv_cache* c) {
  if (c == nullptr || c->k_cache == nullptr || c->v_cache == nullptr) return PA_ERR_NULL;
  if (c->num_blocks <= 0 || c->block_size <= 0 || c->num_kv_heads <= 0 || c->head_dim <= 0)
    return PA_ERR_SHAPE;
  if (c->dtype != PA_KV_BF16 && c->dtype != PA_KV_FP8_E4M3 && c->dtype != PA_KV_INT8)
    return PA_ERR_DTYPE;
  const bool q8 = c->dtype != PA_KV_BF16;  // 8-bit codes with scales
  if (q8 && (c->k_scale == nullptr || c->v_scale == nullptr)) return PA_ERR_DTYPE;
  if (!q8 && (c->k_scale != nullptr || c->v_scale != nullptr)) return PA_ERR_DTYPE;
  if (c->block_size != 16 && c->block_size != 32) return PA_ERR_UNSUPPORTED;
  if (q8 ? c->head_dim != 128 : (c->head_dim != 64 && c->head_dim != 128))
    return PA_ERR_UNSUPPORTED;
  if (static_cast<long long>(c->num_blocks) * c->block_size > 0x7fffffffLL) return PA_ERR_SHAPE;
  if (!aligned16(c->k_cache) || !aligned16(c->v_cache)) return PA_ERR_ALIGN;
  if (q8 && (!aligned16(c->k_scale) || !aligned16(c->v_scale))) return PA_ERR_ALIGN;
  return PA_OK;
}

int elem_bytes(const pa_kv_cache* c) { return c->dtype == PA_KV_BF16 ? 2 : 1; }

// Tensor maps over a cache, 128B-swizzled to match the kernels' shared-memory
// layouts. A tile is block_size rows of one kv head, stored as 128-byte-wide
// subtiles one after the other (subtile j holds bytes [128 j, 128 j + 128) of
// every row).
//   kind kSubtileMap (prefill): the cache as 3-D (head_dim, num_kv_heads,
//     num_blocks*block_size); one box is one subtile.
//   kind kRowMap (decode): the cache as 4-D (128 bytes of a row, row,
//     subtile, kv head), box (128 bytes, block_size, all subtiles, 1): one box
//     is a whole tile, one copy instead of one per subtile.
constexpr int kSubtileMap = 0, kRowMap = 1;
pa_status encode_cache_map(CUtensorMap* map, void* base, const pa_kv_cache* c, int kind) {
  const int eb = elem_bytes(c);
  const cuuint64_t row_bytes = static_cast<cuuint64_t>(c->head_dim) * eb;
  const cuuint64_t rows = static_cast<cuuint64_t>(c->num_blocks) * c->block_size;
  const CUtensorMapDataType dt =
      eb == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  // rows are head_dim*elem bytes apart from the next head's: promote L2
  // fills no wider than one row so no neighbouring head is fetched
  const CUtensorMapL2promotion promo =
      eb == 1 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
  CUresult r;
  if (kind == kSubtileMap) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(c->head_dim),
                                static_cast<cuuint64_t>(c->num_kv_heads), rows};
    const cuuint64_t strides[2] = {row_bytes, row_bytes * c->num_kv_heads};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(pa::kSwizzleBytes / eb), 1u,
                               static_cast<cuuint32_t>(c->block_size)};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    r = g_encode(map, dt, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                 CU_TENSOR_MAP_SWIZZLE_128B, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    const cuuint64_t nsub = row_bytes / pa::kSwizzleBytes;
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(pa::kSwizzleBytes / eb), rows, nsub,
                                static_cast<cuuint64_t>(c->num_kv_heads)};
    const cuuint64_t strides[3] = {row_bytes * c->num_kv_heads,
                                   static_cast<cuuint64_t>(pa::kSwizzleBytes), row_bytes};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(pa::kSwizzleBytes / eb),
                               static_cast<cuuint32_t>(c->block_size),
                               static_cast<cuuint32_t>(nsub), 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    r = g_encode(map, dt, 4, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                 CU_TENSOR_MAP_SWIZZLE_128B, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

// Recently encoded cache tensor maps: encoding is pure host work but costs a
// few microseconds, and a decode loop passes the same cache every step.
struct MapEntry {
  void* base;
  int num_blocks, block_size, num_kv_heads, head_dim, dtype, device, kind;
  CUtensorMap map;
};
constexpr int kMapCache = 16;
MapEntry g_maps[kMapCache];
int g_map_count = 0, g_map_next = 0;
std::mutex g_map_mu;

pa_status cached_cache_map(CUtensorMap* out, void* base, const pa_kv_cache* c, int kind) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_map_mu);
  for (int i = 0; i < g_map_count; ++i) {
    const MapEntry& e = g_maps[i];
    if (e.base == base && e.num_blocks == c->num_blocks && e.block_size == c->block_size &&
        e.num_kv_heads == c->num_kv_heads && e.head_dim == c->head_dim && e.dtype == c->dtype &&
        e.device == dev && e.kind == kind) {
      *out = e.map;
      return PA_OK;
    }
  }
  MapEntry e{base, c->num_blocks, c->block_size, c->num_kv_heads, c->head_dim, c->dtype, dev,
             kind, {}};
  const pa_status st = encode_cache_map(&e.map, base, c, kind);
  if (st != PA_OK) return st;
  g_maps[g_map_next] = e;
  g_map_next = (g_map_next + 1) % kMapCache;
  if (g_map_count < kMapCache) ++g_map_count;
  *out = e.map;
  return PA_OK;
}

// Failure-detection test hook (pa_debug_inject_wait_timeout): the copy the
// first warp of decode CTA 0 leaves unissued (-1: none) and the wait bound
// of decode launches (0: kWaitLimitNs).
std::atomic<int> g_debug_skip_copy{-1};
std::atomic<unsigned long long> g_debug_wait_limit_ns{0};

// Tag of one decode call in the workspace's arrival counters: a call counter
// passed through a 64-bit finalising mix (the one of SplitMix64, a bijection
// of 64-bit words), upper half kept, never 0 (a zeroed counter never matches
// the current call). Consecutive calls thus get unrelated tags, and a word of
// arbitrary earlier contents carries the current call's tag with probability
// 2^-32, not "whenever it holds a small integer".
uint32_t next_epoch() {
  static std::atomic<uint64_t> counter{0};
  while (true) {
    uint64_t z = counter.fetch_add(1) + 0x9e3779b97f4a7c15ull;
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    z ^= z >> 31;
    const uint32_t e = static_cast<uint32_t>(z >> 32);
    if (e != 0) return e;
  }
}

int decode_len_cap(const pa_kv_cache* c, int32_t max_blocks_per_seq, int32_t max_context_len) {
  const long long cap = static_cast<long long>(max_blocks_per_seq) * c->block_size;
  long long v = max_context_len > 0 ? std::min<long long>(max_context_len, cap) : cap;
  return static_cast<int>(std::min<long long>(v, 0x7fffffffLL));
}

}  // namespace

extern "C" {

int32_t pa_abi_version(void) { return PA_ABI_VERSION; }

const char* pa_status_string(pa_status s) {
  switch (s) {
    case PA_OK: return "ok";
    case PA_ERR_NULL: return "required pointer is NULL";
    case PA_ERR_SHAPE: return "invalid or inconsistent size";
    case PA_ERR_DTYPE: return "cache dtype and scale pointers do not match";
    case PA_ERR_UNSUPPORTED: return "unsupported head_dim, block_size or head grouping";
    case PA_ERR_CUDA: return "CUDA call or kernel launch failed";
    case PA_ERR_WORKSPACE: return "workspace missing or too small";
    case PA_ERR_ALIGN: return "pointer not 16-byte aligned";
    case PA_ERR_TOO_LARGE: return "shape needs more scratch than the static buffer holds";
  }
  return "unknown status";
}

pa_status pa_store_kv(const void* k, const void* v, const float* k_scale_new,
                      const float* v_scale_new, const int64_t* slot_mapping, int32_t num_tokens,
                      const pa_kv_cache* cache, void* stream) {
  pa_status st = check_cache(cache);
  if (st != PA_OK) return st;
  if (num_tokens < 0) return PA_ERR_SHAPE;
  if (num_tokens == 0) return PA_OK;
  if (k == nullptr || v == nullptr || slot_mapping == nullptr) return PA_ERR_NULL;
  const bool q8 = cache->dtype != PA_KV_BF16;  // 8-bit codes with scales
  if (q8 != (k_scale_new != nullptr) || q8 != (v_scale_new != nullptr)) return PA_ERR_DTYPE;
  if (!aligned16(k) || !aligned16(v)) return PA_ERR_ALIGN;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != PA_OK) return st;
  pa::StoreArgs a{};
  a.k = k;
  a.v = v;
  a.k_scale_new = k_scale_new;
  a.v_scale_new = v_scale_new;
  a.slot_mapping = slot_mapping;
  a.k_cache = cache->k_cache;
  a.v_cache = cache->v_cache;
  a.k_scale = q8 ? cache->k_scale : nullptr;
  a.v_scale = q8 ? cache->v_scale : nullptr;
  a.num_tokens = num_tokens;
  a.row_bytes = cache->num_kv_heads * cache->head_dim * elem_bytes(cache);
  a.num_kv_heads = cache->num_kv_heads;
  a.block_size = cache->block_size;
  a.num_slots = static_cast<long long>(cache->num_blocks) * cache->block_size;
  a.err = dev->err;
  return pa::launch_store_kv(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK
                                                                                  : PA_ERR_CUDA;
}

size_t pa_decode_workspace_size(const pa_kv_cache* cache, int32_t batch, int32_t num_heads,
                                int32_t max_blocks_per_seq, int32_t max_context_len) {
  if (check_cache(cache) != PA_OK || batch <= 0 || num_heads <= 0 || max_blocks_per_seq <= 0)
    return 0;
  DeviceInfo* dev = nullptr;
  if (device_info(&dev) != PA_OK) return 0;
  const int cap = decode_len_cap(cache, max_blocks_per_seq, max_context_len);
  return pa::plan_decode(batch, num_heads, cache->num_kv_heads, cache->head_dim, cache->block_size,
                         static_cast<int>(cache->dtype), cap, dev->num_sms)
      .workspace_bytes;
}

}  // extern "C"

namespace {

// Shared body of pa_decode and pa_decode_append (k_new == NULL: no append).
pa_status decode_common(const void* q, const pa_kv_cache* cache, const int32_t* block_tables,
                        int32_t max_blocks_per_seq, const int32_t* context_lens,
                        int32_t max_context_len, int32_t batch, int32_t num_heads, float scale,
                        void* out, void* workspace, size_t workspace_bytes, void* stream,
                        const void* k_new, const void* v_new, const float* k_scale_new,
                        const float* v_scale_new, int32_t window, int32_t sinks) {
  pa_status st = check_cache(cache);
  if (st != PA_OK) return st;
  if (sinks < 0) return PA_ERR_SHAPE;
  if (batch < 0 || num_heads <= 0 || max_blocks_per_seq <= 0) return PA_ERR_SHAPE;
  if (batch == 0) return PA_OK;
  if (q == nullptr || block_tables == nullptr || context_lens == nullptr || out == nullptr)
    return PA_ERR_NULL;
  if (num_heads % cache->num_kv_heads != 0) return PA_ERR_SHAPE;
  const int group = num_heads / cache->num_kv_heads;
  if (group > 8) return PA_ERR_UNSUPPORTED;
  if (batch > 65535) return PA_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return PA_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(out)) return PA_ERR_ALIGN;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != PA_OK) return st;
  const int cap = decode_len_cap(cache, max_blocks_per_seq, max_context_len);
  const bool q8 = cache->dtype != PA_KV_BF16;  // 8-bit codes with scales
  const pa::DecodePlan plan = pa::plan_decode(batch, num_heads, cache->num_kv_heads,
                                              cache->head_dim, cache->block_size,
                                              static_cast<int>(cache->dtype), cap,
                                              dev->num_sms);
  if (plan.workspace_bytes > 0 &&
      (workspace == nullptr || workspace_bytes < plan.workspace_bytes || !aligned16(workspace)))
    return PA_ERR_WORKSPACE;
  if (window > 0 && plan.persistent_ctas == 0) return PA_ERR_UNSUPPORTED;
  CUtensorMap kmap, vmap;
  if ((st = cached_cache_map(&kmap, cache->k_cache, cache, kRowMap)) != PA_OK) return st;
  if ((st = cached_cache_map(&vmap, cache->v_cache, cache, kRowMap)) != PA_OK) return st;
  const cudaStream_t strm = static_cast<cudaStream_t>(stream);
  const bool fused_append = k_new != nullptr && plan.persistent_ctas > 0;
  if (k_new != nullptr && !fused_append) {
    // grid-split path: append with its own launch first, then attend
    pa::StoreArgs s{};
    s.k = k_new;
    s.v = v_new;
    s.k_scale_new = k_scale_new;
    s.v_scale_new = v_scale_new;
    s.k_cache = cache->k_cache;
    s.v_cache = cache->v_cache;
    s.k_scale = q8 ? cache->k_scale : nullptr;
    s.v_scale = q8 ? cache->v_scale : nullptr;
    s.num_tokens = batch;
    s.row_bytes = cache->num_kv_heads * cache->head_dim * elem_bytes(cache);
    s.num_kv_heads = cache->num_kv_heads;
    s.block_size = cache->block_size;
    s.num_slots = static_cast<long long>(cache->num_blocks) * cache->block_size;
    s.err = dev->err;
    if (pa::launch_store_new_tokens(s, block_tables, max_blocks_per_seq, context_lens, cap,
                                    strm) != cudaSuccess)
      return PA_ERR_CUDA;
  }
  pa::DecodeArgs a{};
  a.q = q;
  if (fused_append) {
    a.k_new = k_new;
    a.v_new = v_new;
    a.k_scale_new = q8 ? k_scale_new : nullptr;
    a.v_scale_new = q8 ? v_scale_new : nullptr;
    a.k_cache = cache->k_cache;
    a.v_cache = cache->v_cache;
  }
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.k_scale = q8 ? cache->k_scale : nullptr;
  a.v_scale = q8 ? cache->v_scale : nullptr;
  a.out = out;
  a.slot_rows = plan.slot_rows;
  if (plan.workspace_bytes > 0) {
    const size_t rows = plan.partial_slots * plan.slot_rows;
    a.part_o = static_cast<float*>(workspace);
    a.part_ml = a.part_o + rows * cache->head_dim;
    a.prefix_out = reinterpret_cast<int*>(a.part_ml + rows * 2);
    // 8-byte aligned arrival counters after the prefix sums
    const uintptr_t cp = reinterpret_cast<uintptr_t>(a.prefix_out + batch + 1);
    a.seg_counters = reinterpret_cast<unsigned long long*>((cp + 15) & ~static_cast<uintptr_t>(15));
    a.grp_counters = a.seg_counters + static_cast<size_t>(batch) * cache->num_kv_heads;
    a.epoch = next_epoch();
  }
  a.err = dev->err;
  a.batch = batch;
  a.num_heads = num_heads;
  a.num_kv_heads = cache->num_kv_heads;
  a.group = group;
  a.head_dim = cache->head_dim;
  a.block_size = cache->block_size;
  a.max_blocks = max_blocks_per_seq;
  a.num_blocks = cache->num_blocks;
  a.len_cap = cap;
  a.window = window > 0 ? window : 0;
  a.sinks = window > 0 ? sinks : 0;
  a.persistent_ctas = plan.persistent_ctas;
  a.blocks_per_split = plan.blocks_per_split;
  a.num_splits = plan.num_splits;
  a.kv = static_cast<int>(cache->dtype);
  a.scale_log2 = scale * 1.4426950408889634f;  // log2(e): scores kept in base-2 units
  const unsigned long long limit = g_debug_wait_limit_ns.load();
  a.wait_limit_ns = limit > 0 ? limit : pa::kWaitLimitNs;
  a.debug_skip_copy = g_debug_skip_copy.load();
  return pa::launch_decode(a, kmap, vmap, strm) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

extern "C" {

pa_status pa_decode(const void* q, const pa_kv_cache* cache, const int32_t* block_tables,
                    int32_t max_blocks_per_seq, const int32_t* context_lens,
                    int32_t max_context_len, int32_t batch, int32_t num_heads, float scale,
                    void* out, void* workspace, size_t workspace_bytes, void* stream) {
  return decode_common(q, cache, block_tables, max_blocks_per_seq, context_lens, max_context_len,
                       batch, num_heads, scale, out, workspace, workspace_bytes, stream, nullptr,
                       nullptr, nullptr, nullptr, 0, 0);
}

pa_status pa_decode_window(const void* q, const pa_kv_cache* cache, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* context_lens,
                           int32_t max_context_len, int32_t batch, int32_t num_heads,
                           float scale, int32_t window, int32_t sinks, void* out, void* workspace,
                           size_t workspace_bytes, void* stream) {
  return decode_common(q, cache, block_tables, max_blocks_per_seq, context_lens, max_context_len,
                       batch, num_heads, scale, out, workspace, workspace_bytes, stream, nullptr,
                       nullptr, nullptr, nullptr, window, sinks);
}

pa_status pa_decode_append(const void* q, const void* k_new, const void* v_new,
                           const float* k_scale_new, const float* v_scale_new,
                           const pa_kv_cache* cache, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* context_lens,
                           int32_t max_context_len, int32_t batch, int32_t num_heads,
                           float scale, void* out, void* workspace, size_t workspace_bytes,
                           void* stream) {
  return pa_decode_window_append(q, k_new, v_new, k_scale_new, v_scale_new, cache, block_tables,
                                 max_blocks_per_seq, context_lens, max_context_len, batch,
                                 num_heads, scale, 0, 0, out, workspace, workspace_bytes, stream);
}

pa_status pa_decode_window_append(const void* q, const void* k_new, const void* v_new,
                                  const float* k_scale_new, const float* v_scale_new,
                                  const pa_kv_cache* cache, const int32_t* block_tables,
                                  int32_t max_blocks_per_seq, const int32_t* context_lens,
                                  int32_t max_context_len, int32_t batch, int32_t num_heads,
                                  float scale, int32_t window, int32_t sinks, void* out,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  pa_status st = check_cache(cache);
  if (st != PA_OK) return st;
  if (batch > 0 && (k_new == nullptr || v_new == nullptr)) return PA_ERR_NULL;
  const bool q8 = cache->dtype != PA_KV_BF16;  // 8-bit codes with scales
  if (q8 != (k_scale_new != nullptr) || q8 != (v_scale_new != nullptr)) return PA_ERR_DTYPE;
  if (batch > 0 && (!aligned16(k_new) || !aligned16(v_new))) return PA_ERR_ALIGN;
  return decode_common(q, cache, block_tables, max_blocks_per_seq, context_lens, max_context_len,
                       batch, num_heads, scale, out, workspace, workspace_bytes, stream, k_new,
                       v_new, k_scale_new, v_scale_new, window, sinks);
}

pa_status pa_prefill_varlen(const void* q, const pa_kv_cache* cache, const int32_t* block_tables,
                            int32_t max_blocks_per_seq, const int32_t* cu_seqlens_q,
                            const int32_t* cu_seqlens_k, int32_t batch, int32_t num_heads,
                            int32_t total_q, int32_t max_q_len, float scale, void* out,
                            void* stream) {
  pa_status st = check_cache(cache);
  if (st != PA_OK) return st;
  if (batch < 0 || num_heads <= 0 || total_q < 0 || max_blocks_per_seq <= 0) return PA_ERR_SHAPE;
  if (batch == 0 || total_q == 0) return PA_OK;
  if (q == nullptr || block_tables == nullptr || cu_seqlens_q == nullptr ||
      cu_seqlens_k == nullptr || out == nullptr)
    return PA_ERR_NULL;
  if (num_heads % cache->num_kv_heads != 0) return PA_ERR_SHAPE;
  const int group = num_heads / cache->num_kv_heads;
  if (cache->dtype != PA_KV_BF16 || cache->head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (group != 1 && group != 2 && group != 4 && group != 8 && group != 16)
    return PA_ERR_UNSUPPORTED;
  if (batch > 65535 || cache->num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;

  if (!std::isfinite(scale) || !(scale > 0.f)) return PA_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(out)) return PA_ERR_ALIGN;
  DeviceInfo* dev = nullptr;
  if ((st = device_info(&dev)) != PA_OK) return st;
  const int tpt = pa::prefill_tokens_per_tile(group);
  const int qbound = max_q_len > 0 ? std::min(max_q_len, total_q) : total_q;
  // the grid's z extent is the number of query-tile pairs of the longest sequence
  if ((static_cast<long long>(qbound) + 2 * tpt - 1) / (2 * tpt) > 65535) return PA_ERR_UNSUPPORTED;
  // Q viewed as (head_dim, num_heads, total_q); one box = the G heads of a kv
  // head for tpt consecutive tokens, 64 dims (128 bytes) wide.
  CUtensorMap qmap, kmap, vmap;
  {
    const cuuint64_t dims[3] = {128u, static_cast<cuuint64_t>(num_heads),
                                static_cast<cuuint64_t>(total_q)};
    const cuuint64_t strides[2] = {128u * 2u, static_cast<cuuint64_t>(num_heads) * 128u * 2u};
    const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(tpt)};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    if (g_encode(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides,
                 box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return PA_ERR_CUDA;
  }
  if ((st = cached_cache_map(&kmap, cache->k_cache, cache, kSubtileMap)) != PA_OK) return st;
  if ((st = cached_cache_map(&vmap, cache->v_cache, cache, kSubtileMap)) != PA_OK) return st;
  pa::PrefillArgs a{};
  a.block_tables = block_tables;
  a.cu_q = cu_seqlens_q;
  a.cu_k = cu_seqlens_k;
  a.out = out;
  a.err = dev->err;
  a.batch = batch;
  a.num_heads = num_heads;
  a.num_kv_heads = cache->num_kv_heads;
  a.group = group;
  a.head_dim = cache->head_dim;
  a.block_size = cache->block_size;
  a.max_blocks = max_blocks_per_seq;
  a.num_blocks = cache->num_blocks;
  a.tokens_per_tile = tpt;
  a.num_qtiles = (qbound + tpt - 1) / tpt;
  a.scale_log2 = scale * 1.4426950408889634f;
  return pa::launch_prefill(a, qmap, kmap, vmap, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

pa_status pa_debug_inject_wait_timeout(int32_t skip_copy, uint64_t wait_limit_ns) {
  if (skip_copy < 0) {
    g_debug_skip_copy.store(-1);
    g_debug_wait_limit_ns.store(0);
    return PA_OK;
  }
  if (wait_limit_ns == 0 || wait_limit_ns > pa::kWaitLimitNs) return PA_ERR_SHAPE;
  g_debug_wait_limit_ns.store(wait_limit_ns);
  g_debug_skip_copy.store(skip_copy);
  return PA_OK;
}

pa_status pa_get_device_error(uint32_t* code) {
  if (code == nullptr) return PA_ERR_NULL;
  DeviceInfo* dev = nullptr;
  pa_status st = device_info(&dev);
  if (st != PA_OK) return st;
  if (cudaDeviceSynchronize() != cudaSuccess) return PA_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, dev->err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return PA_ERR_CUDA;
  const uint32_t zero = 0;
  if (cudaMemcpy(dev->err, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
    return PA_ERR_CUDA;
  *code = v;
  return PA_OK;
}

}  // extern "C"
