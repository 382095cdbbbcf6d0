// Varlen prefix-cached prefill attention on the sm_103a tensor cores.
//
// What is computed ("Prefill Forward Prefix Caching Explained", Facts 1-2,
// branch 1 and the mask section): sequence b owns packed query rows
// cu_q[b] .. cu_q[b+1]-1 (its q_len new tokens) and kv_len = cu_k[b+1] -
// cu_k[b] keys in the paged cache (cached prefix + the new tokens, stored
// there first). With cached = kv_len - q_len, query i (0-based) attends to
// keys j <= i + cached: the causal mask aligned to the bottom-right corner.
//   out[i, h] = sum_j softmax_j(scale * q[i,h] . K[j, h/G]) V[j, h/G]
//
// How (GB300 design):
//   * One CTA per (128-row query tile, kv head, sequence). The 128 rows are
//     128/G tokens x the G query heads of one kv head (GQA packing), so every
//     K/V tile is loaded once for the whole head group.
//   * Warp 0 streams the tile's Q once and then K and V tiles of 128 keys
//     (128/bs physical blocks, one 3-D TMA box per block and 64-dim half,
//     128B-swizzled), resolving logical -> physical blocks through the block
//     table; blocks past the last needed key are fetched out of bounds so TMA
//     fills them with zeros.
//   * Warp 1 issues the tensor-core MMAs (tcgen05, fp32 accumulation in TMEM):
//     S = Q K^T (M=128, N=128, K=128, operands from shared memory) and
//     O += P V (A = P from TMEM, B = V from shared memory, MN-major).
//   * Warps 2-5 own one TMEM lane (= one query row) each: read S, apply the
//     bottom-right mask only on tiles that reach past the row's last visible
//     key, run the online softmax in base 2 (the running max is only raised,
//     and O rescaled, when it grows by more than 2^8, which keeps P <= 256
//     and leaves O/l unchanged), write P as bf16 into the S columns, and in
//     the end normalise O and store bf16 rows.
//   * TMEM: 256 columns per CTA (S/P 128, O 128), two CTAs per SM.
#include <algorithm>

#include "pa_device.cuh"
#include "pa_prefill.h"
#include "pa_tcgen05.cuh"

namespace pa {

namespace {

constexpr int kBM = 128;       // query rows per tile
constexpr int kBN = 128;       // keys per tile
constexpr int kD = 128;        // head_dim
constexpr int kSub = 128 * kBM;  // bytes of one 64-dim (128-byte-wide) half of a 128-row tile
constexpr int kTileBytes = 2 * kSub;  // 32 KB
constexpr int kSmem = 1024 + 3 * kTileBytes;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 256;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

enum { BAR_Q = 0, BAR_KF, BAR_VF, BAR_KE, BAR_VE, BAR_S, BAR_P, BAR_O, BAR_DRAIN, NBAR };

// Bounded wait that also gives up when another role of the CTA has aborted.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag, uint32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      *abort_flag = 1;
      report_error(err, PA_DEVERR_WAIT_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          uint32_t* err) {
  const bool ok = wait_or_abort(bar, parity, abort_flag, err);
  return __all_sync(0xffffffffu, ok);
}

template <int BS>
__global__ void __launch_bounds__(kThreads, 2)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const PrefillArgs a) {
  constexpr int kBlocksPerTile = kBN / BS;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[NBAR];
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z, kvh = blockIdx.y;
  const int qt = a.num_qtiles - 1 - static_cast<int>(blockIdx.x);  // heaviest tiles first
  const int G = a.group, TPT = a.tokens_per_tile;

  const int q0 = a.cu_q[b];
  const int q_len = max(a.cu_q[b + 1] - q0, 0);
  const int kv_len = max(a.cu_k[b + 1] - a.cu_k[b], 0);
  const int cached = max(kv_len - q_len, 0);
  const int t0 = qt * TPT;
  if (t0 >= q_len) return;
  const int t_end = min(t0 + TPT, q_len);
  const int n_keys = min(cached + t_end, kv_len);  // keys the tile's last row can see
  const int T = (n_keys + kBN - 1) / kBN;
  __nv_bfloat16* const out = static_cast<__nv_bfloat16*>(a.out);
  const int H = a.num_heads;

  if (T == 0) {  // no keys at all (invalid q_len > kv_len = 0): zero rows
    for (int e = threadIdx.x; e < (t_end - t0) * G * (kD / 8); e += kThreads) {
      const int row = e / (kD / 8), c = e % (kD / 8);
      const int tok = t0 + row / G, g = row % G;
      reinterpret_cast<uint4*>(out + (static_cast<long long>(q0 + tok) * H + kvh * G + g) * kD)[c] =
          make_uint4(0, 0, 0, 0);
    }
    return;
  }

  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw);
  const uint32_t q_s = base, k_s = base + kTileBytes, v_s = base + 2 * kTileBytes;
  const uint32_t bar0 = smem_addr(&bars[0]);
  auto bar = [&](int i) { return bar0 + 8u * i; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBAR; ++i) mbar_init(bar(i), i == BAR_P ? 4 : 1);
    abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tc::tmem_alloc(smem_addr(&tmem_slot), kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;
  const uint32_t tS = tmem, tO = tmem + 128;  // columns; P overwrites S's first 64 columns

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int k_issued = 0, v_issued = 0;
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(BAR_Q), kTileBytes);
      tma_load_3d(q_s, &qmap, bar(BAR_Q), 0, kvh * G, q0 + t0);
      tma_load_3d(q_s + kSub, &qmap, bar(BAR_Q), 64, kvh * G, q0 + t0);
    }
    const long long bt_row = static_cast<long long>(b) * a.max_blocks;
    const int oob = a.num_blocks * BS;  // first row past the pool: TMA fills zeros
    for (int n = 0; n < T; ++n) {
      int rc = oob;
      if (lane < kBlocksPerTile) {
        const int lb = n * kBlocksPerTile + lane;
        if (lb * BS < n_keys && lb < a.max_blocks) {
          const int phys = a.block_tables[bt_row + lb];
          if (phys >= 0 && phys < a.num_blocks) {
            rc = phys * BS;
          } else {
            report_error(a.err, PA_DEVERR_BLOCK_RANGE);
          }
        }
      }
      if (n > 0 && !warp_wait(bar(BAR_KE), (n - 1) & 1, &abort_flag, a.err)) break;
      if (lane == 0) mbar_arrive_expect_tx(bar(BAR_KF), kTileBytes);
#pragma unroll
      for (int i = 0; i < kBlocksPerTile; ++i) {
        const int c = __shfl_sync(0xffffffffu, rc, i);
        if (lane == 0) {
          tma_load_3d(k_s + i * BS * 128, &kmap, bar(BAR_KF), 0, kvh, c);
          tma_load_3d(k_s + kSub + i * BS * 128, &kmap, bar(BAR_KF), 64, kvh, c);
        }
      }
      ++k_issued;
      if (n > 0 && !warp_wait(bar(BAR_VE), (n - 1) & 1, &abort_flag, a.err)) break;
      if (lane == 0) mbar_arrive_expect_tx(bar(BAR_VF), kTileBytes);
#pragma unroll
      for (int i = 0; i < kBlocksPerTile; ++i) {
        const int c = __shfl_sync(0xffffffffu, rc, i);
        if (lane == 0) {
          tma_load_3d(v_s + i * BS * 128, &vmap, bar(BAR_VF), 0, kvh, c);
          tma_load_3d(v_s + kSub + i * BS * 128, &vmap, bar(BAR_VF), 64, kvh, c);
        }
      }
      ++v_issued;
    }
    if (abort_flag) {
      // let the copies already in flight land before shared memory is released
      if (k_issued > 0) (void)mbar_wait(bar(BAR_KF), (k_issued - 1) & 1);
      if (v_issued > 0) (void)mbar_wait(bar(BAR_VF), (v_issued - 1) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    constexpr uint32_t kIdescQK = tc::idesc_bf16_f32(kBM, kBN, false, false);
    constexpr uint32_t kIdescPV = tc::idesc_bf16_f32(kBM, kD, false, true);
    bool ok = warp_wait(bar(BAR_Q), 0, &abort_flag, a.err);
    for (int n = 0; ok && n < T; ++n) {
      if (!warp_wait(bar(BAR_KF), n & 1, &abort_flag, a.err)) break;
      if (n > 0 && !warp_wait(bar(BAR_O), (n - 1) & 1, &abort_flag, a.err)) break;
      tc::fence_after_sync();
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kSub + (kk & 3) * 32;
          tc::mma_ss(tS, tc::smem_desc_sw128(q_s + off, 16, 1024),
                     tc::smem_desc_sw128(k_s + off, 16, 1024), kIdescQK, kk > 0 ? 1u : 0u);
        }
        tc::commit(bar(BAR_S));
        tc::commit(bar(BAR_KE));
      }
      __syncwarp();
      if (!warp_wait(bar(BAR_P), n & 1, &abort_flag, a.err)) break;
      if (!warp_wait(bar(BAR_VF), n & 1, &abort_flag, a.err)) break;
      // rows of the last, partly filled physical block past kv_len hold
      // whatever the pool had there: zero them so that P = 0 times V stays 0
      const int r0 = kv_len - n * kBN;
      if (r0 > 0 && r0 < kBN && (r0 % BS) != 0) {
        const int r1 = min(kBN, (r0 / BS + 1) * BS);
        for (int e = lane; e < (r1 - r0) * 16; e += 32) {
          const int row = r0 + (e >> 4), c = e & 15;
          *reinterpret_cast<uint4*>(base_ptr + 2 * kTileBytes + (c >> 3) * kSub + row * 128 +
                                    (c & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      tc::fence_after_sync();
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          tc::mma_ts(tO, tS + kk * 8, tc::smem_desc_sw128(v_s + kk * 16 * 128, kSub, 1024),
                     kIdescPV, (n > 0 || kk > 0) ? 1u : 0u);
        tc::commit(bar(BAR_O));
        tc::commit(bar(BAR_VE));
      }
      __syncwarp();
    }
    if (abort_flag) {  // make sure no MMA is still running before TMEM is freed
      if (lane == 0) tc::commit(bar(BAR_DRAIN));
      __syncwarp();
      (void)mbar_wait(bar(BAR_DRAIN), 0);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int wq = warp & 3;
    const int r = 32 * wq + lane;
    const int tok = t0 + r / G, g = r % G;
    const bool row_valid = tok < t_end;
    const int last_key = min(min(tok, q_len - 1) + cached, kv_len - 1);  // last visible key
    const uint32_t trow = static_cast<uint32_t>(32 * wq) << 16;
    const float sl2 = a.scale_log2;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int n = 0; n < T; ++n) {
      if (!warp_wait(bar(BAR_S), n & 1, &abort_flag, a.err)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      const int lim = last_key - n * kBN;  // keys 0..lim of this tile are visible
      uint32_t u[32];
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        tc::tmem_ld32(tS + trow + 32 * c, u);
        tc::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j)
          mx = fmaxf(mx, (32 * c + j <= lim) ? __uint_as_float(u[j]) : -INFINITY);
      }
      const float m_tile = mx * sl2;
      if (n == 0) {
        m_used = m_tile;
      } else if (__any_sync(0xffffffffu, m_tile > m_used + kRescaleThreshold)) {
        if (!warp_wait(bar(BAR_O), (n - 1) & 1, &abort_flag, a.err)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const float m_new = fmaxf(m_used, m_tile);
        const float alpha = fast_exp2(m_used - m_new);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          tc::tmem_ld32(tO + trow + 32 * c, u);
          tc::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) u[j] = __float_as_uint(__uint_as_float(u[j]) * alpha);
          tc::tmem_st32(tO + trow + 32 * c, u);
        }
        tc::tmem_wait_st();
        l *= alpha;
        m_used = m_new;
      }
      // P = 2^(s*scale*log2e - m_used) as bf16, keys 64h..64h+63 -> columns 32h..32h+31
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t u0[32], u1[32], w[32];
        tc::tmem_ld32(tS + trow + 64 * h, u0);
        tc::tmem_ld32(tS + trow + 64 * h + 32, u1);
        tc::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int k0 = 64 * h + 2 * j;
          const float p0 = k0 <= lim ? fast_exp2(fmaf(__uint_as_float(u0[2 * j]), sl2, -m_used)) : 0.f;
          const float p1 =
              k0 + 1 <= lim ? fast_exp2(fmaf(__uint_as_float(u0[2 * j + 1]), sl2, -m_used)) : 0.f;
          l += p0 + p1;
          w[j] = pack_bf16x2(p0, p1);
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int k0 = 64 * h + 32 + 2 * j;
          const float p0 = k0 <= lim ? fast_exp2(fmaf(__uint_as_float(u1[2 * j]), sl2, -m_used)) : 0.f;
          const float p1 =
              k0 + 1 <= lim ? fast_exp2(fmaf(__uint_as_float(u1[2 * j + 1]), sl2, -m_used)) : 0.f;
          l += p0 + p1;
          w[16 + j] = pack_bf16x2(p0, p1);
        }
        tc::tmem_st32(tS + trow + 32 * h, w);
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_P));
    }
    if (ok && warp_wait(bar(BAR_O), (T - 1) & 1, &abort_flag, a.err)) {
      tc::fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* orow = out + (static_cast<long long>(q0 + tok) * H + kvh * G + g) * kD;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t u[32];
        tc::tmem_ld32(tO + trow + 32 * c, u);
        tc::tmem_wait_ld();
        if (row_valid) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            pk[j] = pack_bf16x2(__uint_as_float(u[2 * j]) * inv, __uint_as_float(u[2 * j + 1]) * inv);
          uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
        }
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, const CUtensorMap& qmap, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, cudaStream_t stream) {
  if (a.head_dim != kD || kBM % a.group != 0) return cudaErrorInvalidValue;
  dim3 grid(a.num_qtiles, a.num_kv_heads, a.batch);
  if (a.block_size == 16) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    prefill_kernel<16><<<grid, kThreads, kSmem, stream>>>(qmap, kmap, vmap, a);
  } else if (a.block_size == 32) {
    cudaError_t e = cudaFuncSetAttribute(prefill_kernel<32>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    prefill_kernel<32><<<grid, kThreads, kSmem, stream>>>(qmap, kmap, vmap, a);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

int prefill_tokens_per_tile(int group) { return kBM / group; }

}  // namespace pa
