// Paged decode attention for sm_103a.
//
// What is computed ("Decode Phase Attention Forward Pass", sections 2-4 and
// the zero-padding caveat; "Decode Phase" glossary): for sequence b and query
// head h, with kv head g = h / (H / Hkv),
//     s_p = scale * q[b,h] . K[slot(b,p), g],   p = 0 .. context_len[b]-1
//     out[b,h] = sum_p softmax(s)_p * V[slot(b,p), g]
// where slot(b,p) = block_tables[b][p / bs] * bs + p % bs. Exactly
// context_len keys take part (no padding to a batch maximum).
//
// How (GB300 design):
//   * Work is the list of (sequence, kv head) "segments", each a run of
//     ceil(context_len / bs) physical blocks. The persistent kernel gives every
//     warp a contiguous share of all blocks of all segments, equal in work
//     units (each block one unit, each segment end a fixed number more): long
//     and short sequences cost the same per block, and no CTA is launched
//     without work. A warp writes the bf16 rows of a segment it holds whole;
//     for a segment that straddles warps each writes an fp32 partial and the
//     last to arrive (per-segment counter) merges them.
//   * All G = H/Hkv query heads of a kv head share every K/V tile (GQA).
//   * Each warp streams its blocks through a private ring of shared-memory
//     stages filled by TMA (one tensor copy per K or V tile of one block and
//     kv head, 128B-swizzled; 8-bit-code scales by per-lane 4-byte async
//     copies), tracked by mbarriers with bounded waits. Loads run ahead across segment boundaries;
//     block ids are read 32 at a time, a window ahead of the loads.
//   * The two contractions per block, S = Q K^T (heads x tokens over head_dim)
//     and O^T += V^T P^T (head_dim x heads over tokens), run on the warp-level
//     tensor-core MMA (m16n8k16, fp32 accumulate). The softmax is online
//     ("tiny-vllm part 05", pagedAttentionKernel section): a running max and
//     sum per head, reduced over the 4 lanes that share a head with warp
//     shuffles, accumulators rescaled when the max grows.
//   * 8-bit KV (E4M3 or INT8 codes, flag Q8): codes are widened exactly to
//     f16 in registers; the K scale multiplies the score, the V scale the
//     probability.
//   * A sliding window with sinks (WIN) walks only the blocks that hold a
//     visible key and masks the rest inside them.
//   * Batches above kMaxPersistentBatch use a grid of (kv head, sequence,
//     split) CTAs instead, with the same per-block code.
#include <algorithm>

#include "pa_device.cuh"
#include "pa_launch.h"

namespace pa {

namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kMaxDevices = 64;

template <int D, int BS, int NW, int ST, bool Q8>
struct Cfg {
  static constexpr int kElem = Q8 ? 1 : 2;
  static constexpr int kRowBytes = D * kElem;                  // one (token, kv head) row
  static constexpr int kNSub = kRowBytes / kSwizzleBytes;      // 128-byte-wide subtiles per row
  static constexpr int kSubBytes = BS * kSwizzleBytes;
  static constexpr int kTile = kNSub * kSubBytes;              // K (or V) of one block, one kv head
  static constexpr int kStage = 2 * kTile;
  static constexpr int kTiles = NW * ST * kStage;
  static constexpr int kScaleBytes = Q8 ? NW * ST * 2 * BS * 4 : 0;
  static constexpr int kMoStride = D + 4;                      // padded row of the merge buffer
  static constexpr int kMerge = NW * 8 * kMoStride * 4 + NW * 8 * 2 * 4;
  static constexpr uint32_t kTx = kStage;  // bytes the two tensor copies of a stage bring
  // arrivals per stage phase: the copy issuer's, plus (8-bit) one per lane for
  // its asynchronous copies of the block's scales
  static constexpr uint32_t kArrivals = Q8 ? 33 : 1;
  static_assert(kRowBytes % kSwizzleBytes == 0, "row must be a multiple of 128 bytes");
  static_assert(BS % 16 == 0, "block size must be a multiple of 16");
  static_assert(!Q8 || D == 128, "the 8-bit path is written for head_dim 128");
  static_assert(kMerge % 16 == 0, "merge buffer must keep 16-byte alignment");
};

// Shared-memory byte address of 16-byte chunk `chunk` (0 .. D*elem/16-1) of
// row `row` in a tile stored as 128B-swizzled, 128-byte-wide subtiles.
template <int BS>
__device__ __forceinline__ uint32_t swz(uint32_t tile, int row, int chunk) {
  const int sub = chunk >> 3, c = chunk & 7;
  return tile + sub * (BS * kSwizzleBytes) + row * kSwizzleBytes + ((c ^ (row & 7)) << 4);
}

// The 8-bit scales of one block (BS K scales, then BS V scales, from element
// `off` of k_scale / v_scale) into shared memory at `dst`: one 4-byte
// asynchronous copy per lane and scale (no TMA: a 128-byte bulk copy costs the
// tensor-copy unit as much as a whole tile), then every lane's one arrival on
// the stage barrier for its copies (the barrier counts 32 of them).
template <int BS>
__device__ __forceinline__ void copy_scales(const DecodeArgs& a, uint32_t dst, long long off,
                                            uint32_t bar, int lane) {
#pragma unroll
  for (int i = lane; i < 2 * BS; i += 32) {
    const bool isv = i >= BS;
    const int t = isv ? i - BS : i;
    cp_async_4(dst + 4 * i, (isv ? a.v_scale : a.k_scale) + off + t);
  }
  cp_async_arrive_noinc(bar);
}

// floor(log2 |x|) of a normal float, and 2^k for k in [-126, 127], exactly.
__device__ __forceinline__ int float_exponent(float x) {
  return static_cast<int>((__float_as_uint(x) >> 23) & 0xffu) - 127;
}
__device__ __forceinline__ float pow2i(int k) {
  return __uint_as_float(static_cast<uint32_t>(min(max(k, -126), 127) + 127) << 23);
}

// Q fragments (A operand of S = Q K^T) of kv head `kvh` of sequence b:
// MMA row r = head r of the group (rows >= G are zero).
// bf16: k index of step ks = head_dim ks*16 + {2q4, 2q4+1, 2q4+8, 2q4+9}.
// 8-bit codes (f16 MMA): the head_dim order inside a step is permuted to match how
// the K codes are read (lane quad q4 owns dims [32 q4, 32 q4 + 32)): step ks
// uses dims 32 q4 + 4 ks + {0,1} (k = 2q4, 2q4+1) and + {2,3} (k = 2q4+8, +9).
// The f16 operands of the 8-bit path hold q times a power of two that puts
// the group's largest |q| in [128, 256): any bf16 q keeps its 8 significant
// bits (f16 has 11) and cannot overflow f16. q_inv is the inverse factor, to
// be folded into the score scale (exact: powers of two).
template <int D, bool Q8>
__device__ __forceinline__ void fetch_q(const DecodeArgs& a, int b, int kvh, int lane,
                                        uint32_t (&raw)[D / 16][2]) {
  const int G = a.group, r = lane >> 2, q4 = lane & 3;
  const __nv_bfloat16* qrow = static_cast<const __nv_bfloat16*>(a.q) +
                              (static_cast<long long>(b) * a.num_heads + kvh * G + min(r, G - 1)) * D;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    if (r < G) {
      if constexpr (!Q8) {
        raw[ks][0] = *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 2 * q4);
        raw[ks][1] = *reinterpret_cast<const uint32_t*>(qrow + ks * 16 + 8 + 2 * q4);
      } else {
        const uint2 v = *reinterpret_cast<const uint2*>(qrow + 32 * q4 + 4 * ks);
        raw[ks][0] = v.x;
        raw[ks][1] = v.y;
      }
    } else {
      raw[ks][0] = 0u;
      raw[ks][1] = 0u;
    }
  }
}

template <int D, bool Q8>
__device__ __forceinline__ void finish_q(const uint32_t (&raw)[D / 16][2],
                                         uint32_t (&qa)[D / 16][2], float& q_inv) {
  if constexpr (!Q8) {
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      qa[ks][0] = raw[ks][0];
      qa[ks][1] = raw[ks][1];
    }
    q_inv = 1.f;
  } else {
    uint32_t amax_bits = 0u;  // largest |q| of the lane, as bits (non-negative floats)
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      // |bf16| pairs as bits: clear the sign bits, then compare the 16-bit halves
      const uint32_t x = raw[ks][0] & 0x7fff7fffu, y = raw[ks][1] & 0x7fff7fffu;
      amax_bits = max(amax_bits, max(max(x >> 16, x & 0xffffu), max(y >> 16, y & 0xffffu)));
    }
    amax_bits = __reduce_max_sync(kFull, amax_bits);
    const float amax = __uint_as_float(amax_bits << 16);  // bf16 bits -> float
    const int k = amax > 0.f ? 7 - float_exponent(amax) : 0;
    const float qf = pow2i(k);
    q_inv = pow2i(-k);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      const __nv_bfloat162 lo = *reinterpret_cast<const __nv_bfloat162*>(&raw[ks][0]);
      const __nv_bfloat162 hi = *reinterpret_cast<const __nv_bfloat162*>(&raw[ks][1]);
      qa[ks][0] = pack_f16x2(__low2float(lo) * qf, __high2float(lo) * qf);
      qa[ks][1] = pack_f16x2(__low2float(hi) * qf, __high2float(hi) * qf);
    }
  }
}

template <int D, bool Q8>
__device__ __forceinline__ void load_q(const DecodeArgs& a, int b, int kvh, int lane,
                                       uint32_t (&qa)[D / 16][2], float& q_inv) {
  uint32_t raw[D / 16][2];
  fetch_q<D, Q8>(a, b, kvh, lane, raw);
  finish_q<D, Q8>(raw, qa, q_inv);
}

// One physical block (tokens tok0 .. tok0+BS-1, of which those < L count)
// staged in shared memory at kt (K) / vt (V), 8-bit-code scales at ksc / vsc:
// fold it into the warp's online-softmax state (m_run, l_run for head r of
// lane group r; acc = O^T fragments for heads 2q4, 2q4+1). The whole block is
// one softmax step: S for its BS tokens (BS/8 n-tiles, independent MMA
// chains), one max/sum update, then P.V per 16-token group.
template <int D, int BS, int KV, bool HOLE = false>
__device__ __forceinline__ void attend_block(uint32_t kt, uint32_t vt, const uint8_t* base_ptr,
                                             uint32_t base, const float* ksc, const float* vsc,
                                             int tok0, int L, int hole_lo, int hole_hi,
                                             const uint32_t (&qa)[D / 16][2],
                                             float (&acc)[D / 16][4], float& m_run, float& l_run,
                                             float& vfac, float sl2, int lane) {
  constexpr int NT = BS / 8;  // n-tiles of 8 tokens
  constexpr int NG = BS / 16;  // 16-token groups (k-steps of P.V)
  constexpr bool Q8 = KV != kKvBf16;
  const int r = lane >> 2, q4 = lane & 3;
  // keys t < L outside the window's hole [hole_lo, hole_hi) take part
  auto valid = [&](int t) { return t < L && (!HOLE || t < hole_lo || t >= hole_hi); };
  const bool partial = tok0 + BS > L || (HOLE && hole_lo < tok0 + BS && hole_hi > tok0);
  // ---- S = Q K^T for the block's tokens
  float sc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
  if constexpr (!Q8) {
    const int mi = lane >> 3;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
      for (int hg = 0; hg < NG; ++hg) {
        const int row = hg * 16 + (mi >> 1) * 8 + (lane & 7);
        uint32_t b00, b01, b10, b11;
        ldmatrix_x4(swz<BS>(kt, row, 2 * ks + (mi & 1)), b00, b01, b10, b11);
        mma_bf16(sc[2 * hg], qa[ks][0], 0u, qa[ks][1], 0u, b00, b01);
        mma_bf16(sc[2 * hg + 1], qa[ks][0], 0u, qa[ks][1], 0u, b10, b11);
      }
    }
  } else {
    uint32_t w[NT][8];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int row = nt * 8 + r;
      const uint4 c0 = *reinterpret_cast<const uint4*>(base_ptr + (swz<BS>(kt, row, 2 * q4) - base));
      const uint4 c1 =
          *reinterpret_cast<const uint4*>(base_ptr + (swz<BS>(kt, row, 2 * q4 + 1) - base));
      w[nt][0] = c0.x; w[nt][1] = c0.y; w[nt][2] = c0.z; w[nt][3] = c0.w;
      w[nt][4] = c1.x; w[nt][5] = c1.y; w[nt][6] = c1.z; w[nt][7] = c1.w;
    }
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        uint32_t b0, b1;
        codes8x4_to_f16x2x2<KV>(w[nt][ks], b0, b1);
        mma_f16(sc[nt], qa[ks][0], 0u, qa[ks][1], 0u, b0, b1);
      }
    }
  }
  // ---- one online-softmax step for head r over tokens tok0 + nt*8 + 2q4 + {0,1}
  float x[2 * NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    if constexpr (!Q8) {
      x[2 * nt] = sc[nt][0] * sl2;
      x[2 * nt + 1] = sc[nt][1] * sl2;
    } else {
      const float2 k2 = *reinterpret_cast<const float2*>(ksc + nt * 8 + 2 * q4);
      x[2 * nt] = sc[nt][0] * (k2.x * sl2);
      x[2 * nt + 1] = sc[nt][1] * (k2.y * sl2);
    }
  }
  if (partial) {
#pragma unroll
    for (int j = 0; j < 2 * NT; ++j)
      if (!valid(tok0 + (j >> 1) * 8 + 2 * q4 + (j & 1))) x[j] = -INFINITY;
  }
  float mx = x[0];
#pragma unroll
  for (int j = 1; j < 2 * NT; ++j) mx = fmaxf(mx, x[j]);
  mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
  const float m_new = fmaxf(m_run, mx);
  float pr[2 * NT];
  float psum = 0.f;
#pragma unroll
  for (int j = 0; j < 2 * NT; ++j) {
    pr[j] = fast_exp2(x[j] - m_new);
    psum += pr[j];
  }
  if (__any_sync(kFull, m_new > m_run)) {  // some head's max grew: rescale
    const float alpha = fast_exp2(m_run - m_new);
    l_run *= alpha;
    // accumulator columns are heads 2q4 and 2q4+1: fetch their factors
    const float al0 = __shfl_sync(kFull, alpha, 8 * q4);
    const float al1 = __shfl_sync(kFull, alpha, 8 * q4 + 4);
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      acc[mt][0] *= al0;
      acc[mt][1] *= al1;
      acc[mt][2] *= al0;
      acc[mt][3] *= al1;
    }
  }
  l_run += psum;
  m_run = m_new;
  // ---- 8-bit V: the f16 operand P' = p * v_scale * vfac. vfac is a power of
  // two chosen so that the block's largest V scale times vfac lies in
  // [2^-4, 2^12] (P' <= 4096 since p <= 1: no f16 overflow, and no f16
  // subnormals for any p above 2^-10); when a block falls outside, vfac moves
  // to put it at [128, 256) and acc, which holds sum P' v, is rescaled by the
  // same power of two (exact). The writers divide acc by vfac.
  float vsf[NG][4];
  if constexpr (Q8) {
    float vm = 0.f;
#pragma unroll
    for (int hg = 0; hg < NG; ++hg) {
      const int g0 = tok0 + hg * 16 + 2 * q4;
      const float2 v0 = *reinterpret_cast<const float2*>(vsc + hg * 16 + 2 * q4);
      const float2 v1 = *reinterpret_cast<const float2*>(vsc + hg * 16 + 8 + 2 * q4);
      // masked keys' scales may hold anything: they take no part
      vsf[hg][0] = valid(g0) ? v0.x : 0.f;
      vsf[hg][1] = valid(g0 + 1) ? v0.y : 0.f;
      vsf[hg][2] = valid(g0 + 8) ? v1.x : 0.f;
      vsf[hg][3] = valid(g0 + 9) ? v1.y : 0.f;
      vm = fmaxf(vm, fmaxf(fmaxf(vsf[hg][0], vsf[hg][1]), fmaxf(vsf[hg][2], vsf[hg][3])));
    }
    // the 4 lanes of a quad cover the block's tokens; every quad holds the same
    vm = fmaxf(vm, __shfl_xor_sync(kFull, vm, 1));
    vm = fmaxf(vm, __shfl_xor_sync(kFull, vm, 2));
    const float t = vm * vfac;
    if (vm > 0.f && !(t >= 0.0625f && t <= 4096.f)) {  // warp-uniform
      const float nf = pow2i(7 - float_exponent(vm));
      const float ratio = nf / vfac;  // a power of two
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        acc[mt][0] *= ratio;
        acc[mt][1] *= ratio;
        acc[mt][2] *= ratio;
        acc[mt][3] *= ratio;
      }
      vfac = nf;
    }
#pragma unroll
    for (int hg = 0; hg < NG; ++hg)
#pragma unroll
      for (int j = 0; j < 4; ++j) vsf[hg][j] *= vfac;
  }
  // ---- O^T += V^T P^T, one k-step per 16-token group
#pragma unroll
  for (int hg = 0; hg < NG; ++hg) {
    const int g0 = tok0 + hg * 16 + 2 * q4;  // tokens of this lane's P entries: g0, g0+1, g0+8, g0+9
    if (partial && hg * 16 + tok0 >= L) break;
    uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
    if (partial) {  // V rows of masked keys may hold anything: zero their fragments
      mlo = (valid(g0) ? 0x0000ffffu : 0u) | (valid(g0 + 1) ? 0xffff0000u : 0u);
      mhi = (valid(g0 + 8) ? 0x0000ffffu : 0u) | (valid(g0 + 9) ? 0xffff0000u : 0u);
    }
    const float p0 = pr[4 * hg], p1 = pr[4 * hg + 1], p8 = pr[4 * hg + 2], p9 = pr[4 * hg + 3];
    if constexpr (!Q8) {
      // P as two bf16 terms, p = hi + lo (hi = bf16(p), lo = bf16(p - hi)):
      // one bf16 rounding of P alone (2^-9 relative per weight) can move an
      // output over few keys by more than the tolerance; the sum of two
      // terms carries ~16 significant bits. The second MMA reuses the V
      // fragments; this kernel is HBM-bound, the tensor pipe mostly idle.
      const uint32_t pb0 = pack_bf16x2(p0, p1);
      const uint32_t pb1 = pack_bf16x2(p8, p9);
      const uint32_t pl0 = pack_bf16x2(p0 - __uint_as_float(pb0 << 16),
                                       p1 - __uint_as_float(pb0 & 0xffff0000u));
      const uint32_t pl1 = pack_bf16x2(p8 - __uint_as_float(pb1 << 16),
                                       p9 - __uint_as_float(pb1 & 0xffff0000u));
      const int mi = lane >> 3;
      const int row = hg * 16 + (mi >> 1) * 8 + (lane & 7);
      if (partial) {
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          uint32_t a0, a1, a2, a3;
          ldmatrix_x4_trans(swz<BS>(vt, row, 2 * mt + (mi & 1)), a0, a1, a2, a3);
          a0 &= mlo;
          a1 &= mlo;
          a2 &= mhi;
          a3 &= mhi;
          mma_bf16(acc[mt], a0, a1, a2, a3, pb0, pb1);
          mma_bf16(acc[mt], a0, a1, a2, a3, pl0, pl1);
        }
      } else {
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          uint32_t a0, a1, a2, a3;
          ldmatrix_x4_trans(swz<BS>(vt, row, 2 * mt + (mi & 1)), a0, a1, a2, a3);
          mma_bf16(acc[mt], a0, a1, a2, a3, pb0, pb1);
          mma_bf16(acc[mt], a0, a1, a2, a3, pl0, pl1);
        }
      }
    } else {
      // masked tokens have p = 0 and a zeroed scale
      const uint32_t pb0 = pack_f16x2(p0 * vsf[hg][0], p1 * vsf[hg][1]);
      const uint32_t pb1 = pack_f16x2(p8 * vsf[hg][2], p9 * vsf[hg][3]);
      // lane (r, q4) reads 16-byte chunk r of token rows 2q4, 2q4+1, 2q4+8, 2q4+9:
      // word w gives dims 16r + 4w + {0..3}; output row mapping in the writers.
      const int t0 = hg * 16 + 2 * q4;
      const uint4 W0 = *reinterpret_cast<const uint4*>(base_ptr + (swz<BS>(vt, t0, r) - base));
      const uint4 W1 = *reinterpret_cast<const uint4*>(base_ptr + (swz<BS>(vt, t0 + 1, r) - base));
      const uint4 W8 = *reinterpret_cast<const uint4*>(base_ptr + (swz<BS>(vt, t0 + 8, r) - base));
      const uint4 W9 = *reinterpret_cast<const uint4*>(base_ptr + (swz<BS>(vt, t0 + 9, r) - base));
      const uint32_t w0[4] = {W0.x, W0.y, W0.z, W0.w};
      const uint32_t w1[4] = {W1.x, W1.y, W1.z, W1.w};
      const uint32_t w8[4] = {W8.x, W8.y, W8.z, W8.w};
      const uint32_t w9[4] = {W9.x, W9.y, W9.z, W9.w};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
#pragma unroll
        for (int o = 0; o < 2; ++o) {
          const uint32_t sel = o ? 0x7362u : 0x5140u;
          uint32_t a0, a1, a2, a3;
          codes8x4_to_f16x2x2<KV>(prmt(w0[w], w1[w], sel), a0, a1);
          codes8x4_to_f16x2x2<KV>(prmt(w8[w], w9[w], sel), a2, a3);
          if (partial) {
            a0 &= mlo;
            a1 &= mlo;
            a2 &= mhi;
            a3 &= mhi;
          }
          mma_f16(acc[2 * w + o], a0, a1, a2, a3, pb0, pb1);
        }
      }
    }
  }
}

// Write a warp's (max, sum, O) for its 8 head rows into the merge buffer.
template <int D, int NW, bool Q8>
__device__ __forceinline__ void store_warp_state(float* mo, int warp, int lane, float m_run,
                                                 float l_run, float o_scale,
                                                 const float (&acc)[D / 16][4]) {
  constexpr int S = D + 4;
  const int r = lane >> 2, q4 = lane & 3;
  float l_tot = l_run + __shfl_xor_sync(kFull, l_run, 1);
  l_tot += __shfl_xor_sync(kFull, l_tot, 2);
  float* mm = mo + NW * 8 * S;  // [NW][8] max
  float* ml = mm + NW * 8;      // [NW][8] sum
  if (q4 == 0) {
    mm[warp * 8 + r] = m_run;
    ml[warp * 8 + r] = l_tot;
  }
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) {
    int d0, d1;
    if constexpr (!Q8) {
      d0 = mt * 16 + r;
      d1 = d0 + 8;
    } else {
      d0 = 16 * r + 4 * (mt >> 1) + 2 * (mt & 1);
      d1 = d0 + 1;
    }
    float* row0 = mo + (warp * 8 + 2 * q4) * S;
    float* row1 = row0 + S;
    row0[d0] = acc[mt][0] * o_scale;
    row1[d0] = acc[mt][1] * o_scale;
    row0[d1] = acc[mt][2] * o_scale;
    row1[d1] = acc[mt][3] * o_scale;
  }
}

// Merge the NW warp states of kv head `kvh` of sequence b and write either the
// bf16 output (final) or one fp32 partial (O unnormalised, (max, sum)) to
// partial slot `slot`.
template <int D, int NW>
__device__ __forceinline__ void merge_warps_and_write(const float* mo, const DecodeArgs& a, int b,
                                                      int kvh, bool final_out, long long slot) {
  constexpr int S = D + 4;
  const float* mm = mo + NW * 8 * S;
  const float* ml = mm + NW * 8;
  const int G = a.group;
  for (int e = threadIdx.x; e < G * D; e += NW * 32) {
    const int g = e / D, d = e - g * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, mm[w * 8 + g]);
    float o = 0.f, l = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float f = fast_exp2(mm[w * 8 + g] - M);
        o += f * mo[(w * 8 + g) * S + d];
        l += f * ml[w * 8 + g];
      }
    }
    if (final_out) {
      const long long bh = static_cast<long long>(b) * a.num_heads + kvh * G + g;
      static_cast<__nv_bfloat16*>(a.out)[bh * D + d] = __float2bfloat16_rn(l > 0.f ? o / l : 0.f);
    } else {
      a.part_o[(slot * 8 + g) * D + d] = o;
      if (d == 0) {
        a.part_ml[(slot * 8 + g) * 2 + 0] = M;
        a.part_ml[(slot * 8 + g) * 2 + 1] = l;
      }
    }
  }
}

// Sliding window with sinks: blocks of a sequence of L keys that hold a
// visible key (p < sinks or p >= L - window). They are the first `sb` blocks
// and the blocks from `sb + shift` on, so visible block v is logical block
// v < sb ? v : v + shift; the hole of invisible keys is [hole_lo, hole_hi).
// window <= 0 (or a window reaching back to the sinks) keeps every block.
struct SeqWindow {
  int nvis, sb, shift, hole_lo, hole_hi;
  __device__ __forceinline__ int logical(int v) const { return v < sb ? v : v + shift; }
};

template <int BS>
__device__ __forceinline__ SeqWindow seq_window(int L, int window, int sinks) {
  SeqWindow w;
  const int nblk = (L + BS - 1) / BS;
  w.nvis = nblk;
  w.sb = nblk;
  w.shift = 0;
  w.hole_lo = w.hole_hi = 0;
  if (window > 0 && L > window) {
    const int se = min(sinks, L), lo = L - window;
    if (se < lo) {
      w.hole_lo = se;
      w.hole_hi = lo;
      const int sb = (se + BS - 1) / BS, wb0 = lo / BS;
      if (wb0 > sb) {
        w.sb = sb;
        w.shift = wb0 - sb;
        w.nvis = sb + (nblk - wb0);
      }
    }
  }
  return w;
}

// ============================================================ persistent path
// Flattened work: segment (b, kvh) in b-major order holds nblk(b) blocks; the
// global index of its first block is prefix[b] * Hkv + kvh * nblk(b). Each of
// the W active warps owns a contiguous range of these N = prefix[B] * Hkv
// blocks, cut so that every warp gets the same work counted in blocks plus a
// fixed cost per segment end (block_at_unit below): equal work per warp
// whatever the length mix.
struct Piece {
  int b, kvh, lo, hi;  // segment and its block range owned by this warp
  int nblk;            // blocks of the segment
  long long g;         // global index of block `lo`
  bool valid;
};

__device__ __forceinline__ void piece_first(Piece& p, const int* prefix, int B, int Hkv,
                                            long long r0, long long r1) {
  p.valid = r0 < r1;
  if (!p.valid) return;
  // last b with prefix[b] * Hkv <= r0 (it has nblk > 0 since r0 < prefix[B] * Hkv)
  int lo = 0, hi = B;  // invariant: prefix[lo]*Hkv <= r0 < prefix[hi]*Hkv
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (static_cast<long long>(prefix[mid]) * Hkv <= r0) lo = mid; else hi = mid;
  }
  p.b = lo;
  p.nblk = prefix[lo + 1] - prefix[lo];
  const long long off = r0 - static_cast<long long>(prefix[lo]) * Hkv;
  p.kvh = static_cast<int>(off / p.nblk);
  p.lo = static_cast<int>(off % p.nblk);
  p.hi = static_cast<int>(min(static_cast<long long>(p.nblk), p.lo + (r1 - r0)));
  p.g = r0;
}

__device__ __forceinline__ void piece_next(Piece& p, const int* prefix, int B, int Hkv,
                                           long long r1) {
  p.g += p.hi - p.lo;
  if (p.g >= r1) {
    p.valid = false;
    return;
  }
  if (++p.kvh == Hkv) {
    p.kvh = 0;
    do {
      ++p.b;
    } while (p.b < B && prefix[p.b + 1] == prefix[p.b]);
  }
  p.nblk = prefix[p.b + 1] - prefix[p.b];
  p.lo = 0;
  p.hi = static_cast<int>(min(static_cast<long long>(p.nblk), r1 - p.g));
}

// Write the warp's result for segment (b, kvh): bf16 output rows if the
// segment is entirely this warp's, else an fp32 partial (O unnormalised,
// (max, sum) per head) in `slot`. Lane (r, q4) holds O^T for heads 2q4, 2q4+1
// and the running max/sum of head r.
template <int D, bool Q8>
__device__ __forceinline__ void write_warp_result(const DecodeArgs& a, int b, int kvh,
                                                  bool final_out, long long slot, int lane,
                                                  float m_run, float l_run, float o_scale,
                                                  float (&acc)[D / 16][4]) {
  const int r = lane >> 2, q4 = lane & 3, G = a.group;
  float l_tot = l_run + __shfl_xor_sync(kFull, l_run, 1);
  l_tot += __shfl_xor_sync(kFull, l_tot, 2);
  const int h0 = 2 * q4, h1 = 2 * q4 + 1;  // accumulator heads of this lane
  const float l0 = __shfl_sync(kFull, l_tot, 4 * h0);
  const float l1 = __shfl_sync(kFull, l_tot, 4 * h1);
  if (final_out) {
    const float inv0 = l0 > 0.f ? o_scale / l0 : 0.f, inv1 = l1 > 0.f ? o_scale / l1 : 0.f;
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out) +
                       (static_cast<long long>(b) * a.num_heads + kvh * G) * D;
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) {
      int d0, d1;
      if constexpr (!Q8) { d0 = mt * 16 + r; d1 = d0 + 8; }
      else { d0 = 16 * r + 4 * (mt >> 1) + 2 * (mt & 1); d1 = d0 + 1; }
      if (h0 < G) {
        o[h0 * D + d0] = __float2bfloat16_rn(acc[mt][0] * inv0);
        o[h0 * D + d1] = __float2bfloat16_rn(acc[mt][2] * inv0);
      }
      if (h1 < G) {
        o[h1 * D + d0] = __float2bfloat16_rn(acc[mt][1] * inv1);
        o[h1 * D + d1] = __float2bfloat16_rn(acc[mt][3] * inv1);
      }
    }
    return;
  }
  float* po = a.part_o + slot * a.slot_rows * D;
  if constexpr (Q8) {
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[mt][j] *= o_scale;
  }
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) {
    int d0, d1;
    if constexpr (!Q8) { d0 = mt * 16 + r; d1 = d0 + 8; }
    else { d0 = 16 * r + 4 * (mt >> 1) + 2 * (mt & 1); d1 = d0 + 1; }
    if (h0 < G) {
      po[h0 * D + d0] = acc[mt][0];
      po[h0 * D + d1] = acc[mt][2];
    }
    if (h1 < G) {
      po[h1 * D + d0] = acc[mt][1];
      po[h1 * D + d1] = acc[mt][3];
    }
  }
  if (q4 == 0 && r < G) {
    a.part_ml[(slot * a.slot_rows + r) * 2 + 0] = m_run;
    a.part_ml[(slot * a.slot_rows + r) * 2 + 1] = l_tot;
  }
}

// Warps that take part: about one per 10 blocks of work (N * 51 / 512, a
// multiply and a shift: with a 64-bit divide by 12 here the 8-bit batch-256
// steps, whose warp count it does not change, ran 0.4 % slower), but at
// least one per kMinBlocksPerWarp blocks
// (one per block for short segments) up to one warp per CTA, so that small
// problems keep some parallelism, and at most kMaxPartsPerSegment per
// (sequence, kv head) segment. Problems of more than ~10 blocks per warp of
// the grid use every warp either way. Measured by graph replay on one GB300
// (bf16, 32/8 heads, 16-token blocks), one warp per 16 blocks -> per 10:
// batch 8 x 2048 tokens 21.7 -> 18.2 us, 32 x 1024 27.9 -> 25.0, 64 x 512
// 27.8 -> 24.4, 2 x 12000 27.3 -> 25.7, 8 x 4096 30.0 -> 29.6, 16 x 2048
// 26.4 -> 26.5. One per 12 or 14 blocks was slower overall; one per 8 or 9
// was faster on some of these and slower on the windowed steps.
// Segments of more than kGroupedAbove parts merge in two levels, so no warp
// merges more than max(kGroupedAbove, kMergeGroup + the number of groups)
// partials. (A warp whose share of the work units holds no block has nothing
// to do.)
constexpr long long kWarpsPerBlockNum = 51;  // warps = N * 51 >> 9, about N / 10
constexpr int kWarpsPerBlockShift = 9;
constexpr int kMinBlocksPerWarp = 4;
constexpr int kMaxPartsPerSegment = 1024;
__device__ __forceinline__ long long active_warps(long long N, long long ctas, long long warps,
                                                  long long segments, bool one_block_floor) {
  // (no division by a run-time value: a 64-bit divide here costs registers)
  long long w = max((N * kWarpsPerBlockNum) >> kWarpsPerBlockShift,
                    min(one_block_floor ? N : N / kMinBlocksPerWarp, ctas));
  w = min(w, segments * kMaxPartsPerSegment);
  return max(1LL, min(warps, w));
}

// The floor for a problem whose longest segment has max_blk blocks: when
// every segment is shorter than 8 blocks, one block per warp (the merge of a
// few partials costs less than walking several blocks in turn); otherwise
// kMinBlocksPerWarp. Measured by graph replay on one GB300: the tiny decode
// (7-block segments) 11.7 -> 6.3 us; one 512-token sequence (32-block
// segments) 9.45 us at 4 blocks per warp, 13.0 at 1 and 11.1 at 3 (warp
// ranges then straddle segments unevenly); longer segments unchanged.
constexpr int kShortSegmentBlocks = 8;

// Tiles each warp prefetches into L2 before the dependency wait (bf16).
constexpr int kPrefetchTiles = 4;

// Pieces of a segment that straddles warps: segment (b, kvh) over global
// blocks [s0, s1) is split among warps w0 .. w1 (all with non-empty ranges);
// warp w0 left its piece in slot 2*w0+1, every later one in slot 2*w.
struct SegParts {
  long long w0;
  int n;  // w1 - w0 + 1
  __device__ __forceinline__ long long slot(int j) const {
    return j == 0 ? 2 * w0 + 1 : 2 * (w0 + j);
  }
};

// Segments of more than kGroupedAbove parts merge in two levels: parts
// [16 g, 16 g + 16) form group g; the last arriver of a group merges it into
// the slot of the group's first part, and the last group to finish merges
// the group results. Up to kGroupedAbove parts one merge is faster (one
// level fewer of arrival and partial round trips): 16-17 parts 45.7 us
// against 60.0 us with groups, 57-64 parts 111-112 us against 102-103 us.
constexpr int kMergeGroup = 16;
constexpr int kGroupedAbove = 32;

// Parts j0, j0 + stride, ... (n of them) of a segment, for a merge.
struct PartList {
  SegParts sp;
  int j0, stride, n;
  __device__ __forceinline__ long long slot(int k) const { return sp.slot(j0 + k * stride); }
};

__device__ __forceinline__ SegParts seg_parts(const int* prefix, int B, int Hkv, int b, int kvh,
                                              long long W, int cost) {
  const long long NU = (static_cast<long long>(prefix[B]) + static_cast<long long>(cost) * B) * Hkv;
  const int nblk = prefix[b + 1] - prefix[b];
  // unit of the segment's first block
  const long long u0 = (static_cast<long long>(prefix[b]) + static_cast<long long>(cost) * b) * Hkv +
                       static_cast<long long>(kvh) * (nblk + cost);
  auto owner = [&](long long x) { return ((x + 1) * W - 1) / NU; };
  SegParts sp;
  sp.w0 = owner(u0);
  sp.n = static_cast<int>(owner(u0 + nblk - 1) - sp.w0 + 1);
  return sp;
}

// Fixed work at a segment's end (the new token's append, the piece's result
// or partial, a merge), in blocks of the instantiation's layout. Measured on
// one GB300 by sweeping the value: Llama-3-8B-shaped batch 64 (bf16, 16-token
// blocks) 92.9 us at 2, 90.4 at 6, 91.2 at 12; 70B-shaped batch 256 (32-token
// blocks) best at 4 for E4M3 codes and 3 for INT8 (the widening costs more
// per block, so the fixed work weighs less); 0 would be the equal-block split.
__host__ __device__ constexpr int segment_cost(int kv) {
  return kv == kKvBf16 ? 6 : kv == kKvE4m3 ? 4 : 3;
}

// The split in work units: segment (b, kvh) is its nblk blocks followed by
// `cost` units that stand for the fixed work of a segment's end (the new
// token's append, the piece's result, a merge), so that warps which end many
// segments get fewer blocks. Warp w owns units [w NU / W, (w+1) NU / W), i.e.
// the blocks whose units fall there: a contiguous range of the flattened
// block list. This maps a unit to the index of the first block at or after it.
__device__ __forceinline__ long long block_at_unit(const int* prefix, int B, int Hkv, int cost,
                                                   long long u) {
  const long long NU = (static_cast<long long>(prefix[B]) + static_cast<long long>(cost) * B) * Hkv;
  if (u >= NU) return static_cast<long long>(prefix[B]) * Hkv;
  int lo = 0, hi = B - 1;  // last b whose units start at or before u
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((static_cast<long long>(prefix[mid]) + static_cast<long long>(cost) * mid) * Hkv <= u) lo = mid;
    else hi = mid - 1;
  }
  const int nb = prefix[lo + 1] - prefix[lo];
  const long long off = u - (static_cast<long long>(prefix[lo]) + static_cast<long long>(cost) * lo) * Hkv;
  const int per = nb + cost;
  const int kvh = static_cast<int>(off / per), pos = static_cast<int>(off % per);
  return static_cast<long long>(prefix[lo]) * Hkv + static_cast<long long>(kvh) * nb + min(pos, nb);
}

// Epoch-tagged counters in the caller's workspace (contents on entry are
// arbitrary): the high word holds the call's epoch, the low word the count of
// this call. Every counter is tagged early in the call (tag_counters), so an
// arrival is normally one atomic add. An add that still finds another call's
// epoch tags the word itself with a compare-and-swap (whoever tags first wins;
// only the segment's last arrival clears a tagged word) and counts itself
// again.
__device__ __forceinline__ uint32_t tagged_fetch_add(unsigned long long* counter, uint32_t epoch,
                                                     uint32_t* err) {
  const unsigned long long old = atomicAdd(counter, 1ull);
  if (static_cast<uint32_t>(old >> 32) == epoch) return static_cast<uint32_t>(old);
  unsigned long long cur = old + 1ull;
#pragma unroll 1
  for (int it = 0; it < (1 << 14); ++it) {
    if (static_cast<uint32_t>(cur >> 32) == epoch)
      return static_cast<uint32_t>(atomicAdd(counter, 1ull));
    const unsigned long long prev =
        atomicCAS(counter, cur, (static_cast<unsigned long long>(epoch) << 32) | 1ull);
    if (prev == cur) return 0u;
    cur = prev;
  }
  report_error(err, PA_DEVERR_WAIT_TIMEOUT);
  return 0xffffffffu;
}

// Tag segment counters [lo, hi) and, unless `grp` is null, the two group
// counters grp[0..1] with this call's epoch and a zero count, unless already
// tagged (one lane per counter).
__device__ __forceinline__ void tag_counters(unsigned long long* counters, long long lo,
                                             long long hi, unsigned long long* grp, uint32_t epoch,
                                             int lane) {
  const unsigned long long tagged = static_cast<unsigned long long>(epoch) << 32;
  const int ng = grp != nullptr ? 2 : 0;
  const long long n = ng + max(hi - lo, 0LL);
  for (long long k = lane; k < n; k += 32) {
    unsigned long long* const c = k < ng ? grp + k : counters + lo + (k - ng);
    unsigned long long cur = atomicAdd(c, 0ull);
#pragma unroll 1
    for (int it = 0; it < 8 && static_cast<uint32_t>(cur >> 32) != epoch; ++it) {
      const unsigned long long prev = atomicCAS(c, cur, tagged);
      if (prev == cur) break;
      cur = prev;
    }
  }
}

// Count this warp's arrival at a segment of `parts` pieces; true for the
// last. The last arriver also clears the counter (tag 0 is no call's epoch):
// every other arrival of this call has been counted, so nothing else of this
// call still needs it, and a launch that repeats this call's epoch (a CUDA
// graph replays its captured parameters) finds it untagged and starts the
// count afresh. (A tagging lane of this call that comes later leaves
// (epoch, 0), which is also a correct starting state.)
__device__ __forceinline__ bool arrive_last(unsigned long long* counter, uint32_t epoch,
                                            uint32_t parts, uint32_t* err) {
  const bool last = tagged_fetch_add(counter, epoch, err) + 1u == parts;
  if (last) atomicExch(counter, 0ull);
  return last;
}

// Merge partials of segment (b, kvh): M = max m_j, l = sum l_j 2^(m_j - M),
// o = sum o_j 2^(m_j - M) (scores in base 2), for all G heads at once. With
// `final_out` the bf16 rows o / l are written; otherwise (M, l, o) is stored
// as one partial in the slot of the list's first part. Lane = (head g, slice
// sub of head_dim) with LPH lanes per head (32 / GP, GP = G rounded up to a
// power of two, at most head_dim / 8). The lanes of a head first combine the (max, sum) of the
// parts among themselves (a quarter, an eighth ... of the parts each, then
// shuffles); then every part costs one round of independent loads (its max
// and the lane's head_dim slice of O), two parts in flight at a time.
// Partials are read through L2.
template <int D, int GP>
__device__ __forceinline__ void merge_segment_g(const DecodeArgs& a, const PartList& sp, int b,
                                                int kvh, bool final_out, int lane) {
  // lanes per head (at least 8 dims each, so a slice is whole 16-byte bf16 stores)
  constexpr int LPH = (32 / GP) < (D / 8) ? (32 / GP) : (D / 8);
  constexpr int DL = D / LPH;    // head_dim slice of a lane
  constexpr int V4 = DL / 4;     // float4 of it
  static_assert(DL % 8 == 0 && LPH * GP <= 32, "slices of whole 16-byte stores");
  const int G = a.group;
  const int g = lane / LPH, sub = lane % LPH;
  const bool g_ok = g < G;
  // ---- (max, sum) of head g, online over this lane's parts, then the head's lanes
  float M = -INFINITY, L = 0.f;
  if (g_ok) {
    for (int j = sub; j < sp.n; j += LPH) {
      const float2 ml =
          __ldcg(reinterpret_cast<const float2*>(a.part_ml + (sp.slot(j) * GP + g) * 2));
      const float m2 = fmaxf(M, ml.x);
      if (m2 != -INFINITY) {
        L = L * fast_exp2(M - m2) + ml.y * fast_exp2(ml.x - m2);
        M = m2;
      }
    }
  }
#pragma unroll
  for (int o = LPH / 2; o >= 1; o >>= 1) {
    const float Mo = __shfl_xor_sync(kFull, M, o), Lo = __shfl_xor_sync(kFull, L, o);
    const float m2 = fmaxf(M, Mo);
    if (m2 != -INFINITY) {
      L = L * fast_exp2(M - m2) + Lo * fast_exp2(Mo - m2);
      M = m2;
    }
  }
  // ---- O: the lane's slice of head g, summed over the parts
  float acc[DL];
#pragma unroll
  for (int v = 0; v < DL; ++v) acc[v] = 0.f;
  if (g_ok) {
#pragma unroll 2
    for (int j = 0; j < sp.n; ++j) {
      const long long row = sp.slot(j) * GP + g;
      const float m = __ldcg(a.part_ml + row * 2);
      float4 x[V4];
      const float4* src = reinterpret_cast<const float4*>(a.part_o + row * D + sub * DL);
#pragma unroll
      for (int v = 0; v < V4; ++v) x[v] = __ldcg(src + v);
      const float f = m == -INFINITY ? 0.f : fast_exp2(m - M);
#pragma unroll
      for (int v = 0; v < V4; ++v) {
        acc[4 * v + 0] += f * x[v].x;
        acc[4 * v + 1] += f * x[v].y;
        acc[4 * v + 2] += f * x[v].z;
        acc[4 * v + 3] += f * x[v].w;
      }
    }
  }
  __syncwarp();  // every lane has read the first part's slot before it is overwritten
  if (!g_ok) return;
  if (!final_out) {
    // one partial of the merged parts, in the slot of the first of them
    const long long row = sp.slot(0) * GP + g;
    if (sub == 0) *reinterpret_cast<float2*>(a.part_ml + row * 2) = make_float2(M, L);
    float4* dst = reinterpret_cast<float4*>(a.part_o + row * D + sub * DL);
#pragma unroll
    for (int v = 0; v < V4; ++v)
      dst[v] = make_float4(acc[4 * v], acc[4 * v + 1], acc[4 * v + 2], acc[4 * v + 3]);
    return;
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) +
                       (static_cast<long long>(b) * a.num_heads + kvh * G + g) * D + sub * DL;
#pragma unroll
  for (int v = 0; v < DL; v += 8) {
    uint4 w;
    w.x = pack_bf16x2(acc[v] * inv, acc[v + 1] * inv);
    w.y = pack_bf16x2(acc[v + 2] * inv, acc[v + 3] * inv);
    w.z = pack_bf16x2(acc[v + 4] * inv, acc[v + 5] * inv);
    w.w = pack_bf16x2(acc[v + 6] * inv, acc[v + 7] * inv);
    *reinterpret_cast<uint4*>(dst + v) = w;
  }
}

template <int D>
__device__ __forceinline__ void merge_segment(const DecodeArgs& a, const PartList& sp, int b,
                                              int kvh, bool final_out, int lane) {
  if (a.group <= 1) merge_segment_g<D, 1>(a, sp, b, kvh, final_out, lane);
  else if (a.group <= 2) merge_segment_g<D, 2>(a, sp, b, kvh, final_out, lane);
  else if (a.group <= 4) merge_segment_g<D, 4>(a, sp, b, kvh, final_out, lane);
  else merge_segment_g<D, 8>(a, sp, b, kvh, final_out, lane);
}

// Arrival of one part of a segment of more than kGroupedAbove parts: this
// part's group first (the group's last arriver merges it into the slot of the
// group's first part), then the segment over the group results. Out of line:
// it is rare and must not add registers to the block loop.
template <int D>
__device__ __noinline__ void finish_grouped(const DecodeArgs a, const SegParts sp, int b, int kvh,
                                            long long gw, int lane) {
  const int j = static_cast<int>(gw - sp.w0), g0 = j - j % kMergeGroup;
  const int ng = min(kMergeGroup, sp.n - g0);
  int last = 0;
  if (lane == 0)
    last = arrive_last(a.grp_counters + sp.slot(g0), a.epoch, static_cast<uint32_t>(ng), a.err);
  if (!__shfl_sync(kFull, last, 0)) return;
  __threadfence();
  merge_segment<D>(a, PartList{sp, g0, 1, ng}, b, kvh, false, lane);
  __threadfence();
  __syncwarp();
  const int ngroups = (sp.n + kMergeGroup - 1) / kMergeGroup;
  if (lane == 0)
    last = arrive_last(a.seg_counters + static_cast<long long>(b) * a.num_kv_heads + kvh, a.epoch,
                       static_cast<uint32_t>(ngroups), a.err);
  if (!__shfl_sync(kFull, last, 0)) return;
  __threadfence();
  merge_segment<D>(a, PartList{sp, 0, kMergeGroup, ngroups}, b, kvh, true, lane);
}

template <int D, int BS, int NW, int ST, bool Q8>
struct PCfg {
  using C = Cfg<D, BS, NW, ST, Q8>;
  static constexpr int kScaleOff = C::kTiles;
  static constexpr int kPrefixOff = kScaleOff + C::kScaleBytes;
  static int smem_bytes(int batch) { return 1024 + kPrefixOff + (batch + 1) * 4; }
};

// Fused append (pa_decode_append): the new token of segment (b, kvh) is row t
// of its last block. The warp that attends to that block copies the row from
// k_new / v_new (row `bk` = b * Hkv + kvh) into the staged tile (and the 8-bit
// scales into the staged scales) and into the cache slot. Kept out of line:
// it runs once per segment and must not add registers to the block loop.
template <int D, int BS, bool Q8>
__device__ __noinline__ void append_row(uint8_t* tile, float* stage_scales, const int32_t* bt_entry,
                                        int bk, int t, const DecodeArgs a, int lane) {
  constexpr int kRowBytes = D * (Q8 ? 1 : 2);
  constexpr int kChunks = kRowBytes / 16;
  constexpr int kTile = (kRowBytes / kSwizzleBytes) * BS * kSwizzleBytes;
  const int phys = *bt_entry;
  const bool phys_ok = phys >= 0 && phys < a.num_blocks;
  const int Hkv = a.num_kv_heads, kvh = bk % Hkv;
  if (lane < 2 * kChunks) {
    const bool isv = lane >= kChunks;
    const int c = isv ? lane - kChunks : lane;
    const uint4 val = *reinterpret_cast<const uint4*>(
        static_cast<const uint8_t*>(isv ? a.v_new : a.k_new) +
        static_cast<long long>(bk) * kRowBytes + 16 * c);
    *reinterpret_cast<uint4*>(tile + (isv ? kTile : 0) + (swz<BS>(0, t, c))) = val;
    if (phys_ok)
      *reinterpret_cast<uint4*>(static_cast<uint8_t*>(isv ? a.v_cache : a.k_cache) +
                                ((static_cast<long long>(phys) * BS + t) * Hkv + kvh) * kRowBytes +
                                16 * c) = val;
  }
  if constexpr (Q8) {
    if (lane == 0) {
      const float kn = a.k_scale_new[bk], vn = a.v_scale_new[bk];
      stage_scales[t] = kn;
      stage_scales[BS + t] = vn;
      if (phys_ok) {
        const long long so = (static_cast<long long>(phys) * Hkv + kvh) * BS + t;
        const_cast<float*>(a.k_scale)[so] = kn;
        const_cast<float*>(a.v_scale)[so] = vn;
      }
    }
  }
  if (lane == 0 && !phys_ok) report_error(a.err, PA_DEVERR_BLOCK_RANGE);
  fence_proxy_async_smem();  // generic writes before the stage's next TMA refill
  __syncwarp();
}

template <int D, int BS, int NW, int ST, int KV, bool WIN>
__global__ void __launch_bounds__(NW * 32, 3)
    decode_persistent_kernel(const __grid_constant__ CUtensorMap kmap,
                             const __grid_constant__ CUtensorMap vmap, const DecodeArgs a) {
  constexpr bool Q8 = KV != kKvBf16;
  using C = Cfg<D, BS, NW, ST, Q8>;
  using PC = PCfg<D, BS, NW, ST, Q8>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[NW * ST];
  __shared__ int warp_sums[NW];
  __shared__ int warp_max[NW];

  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw);
  const uint32_t scale_base = base + PC::kScaleOff;
  const float* const scale_ptr = reinterpret_cast<const float*>(base_ptr + PC::kScaleOff);
  int* const prefix = reinterpret_cast<int*>(base_ptr + PC::kPrefixOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int B = a.batch, Hkv = a.num_kv_heads;
  // Launched as a programmatic dependent, and lets the next launch (the next
  // decode step) start early: the prologue below (prefix sums, the split, the
  // first block-id windows) reads only the lengths and the block tables,
  // which no kernel of this library writes, and so overlaps the tail of the
  // previous grid. Everything else (the cache, q, the new rows, the output
  // and the workspace) is touched only after grid_dependency_wait().
  grid_launch_dependents();

  // ---- blocks per sequence and their exclusive prefix sum (whole CTA)
  int carry = 0, vmax = 0;
  for (int base_i = 0; base_i < B; base_i += NW * 32) {
    const int i = base_i + threadIdx.x;
    int v = 0;
    if (i < B)
      v = seq_window<BS>(min(max(a.context_lens[i], 0), a.len_cap), WIN ? a.window : 0, a.sinks)
              .nvis;
    vmax = max(vmax, v);
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) warp_sums[warp] = incl;
    __syncthreads();
    int wbase = 0, total = 0;
    for (int w = 0; w < NW; ++w) {
      if (w < warp) wbase += warp_sums[w];
      total += warp_sums[w];
    }
    if (i < B) prefix[i] = carry + wbase + incl - v;
    carry += total;
    __syncthreads();
  }
  if (threadIdx.x == 0) prefix[B] = carry;
  vmax = __reduce_max_sync(kFull, vmax);
  if (lane == 0) warp_max[warp] = vmax;
  __syncthreads();
  int max_blk = 0;  // blocks of the longest sequence
#pragma unroll
  for (int w = 0; w < NW; ++w) max_blk = max(max_blk, warp_max[w]);

  // ---- this warp's range; from here on warps are independent
  const long long N = static_cast<long long>(prefix[B]) * Hkv;
  const long long W = active_warps(N, gridDim.x, static_cast<long long>(gridDim.x) * NW,
                                   static_cast<long long>(B) * Hkv, max_blk < kShortSegmentBlocks);
  const long long gw = static_cast<long long>(blockIdx.x) * NW + warp;
  // segment-end cost of the split, in blocks; none when every segment is
  // short (one block per warp there)
  const int cost = max_blk < kShortSegmentBlocks ? 0 : segment_cost(KV);
  const long long NU = (static_cast<long long>(prefix[B]) + static_cast<long long>(cost) * B) * Hkv;
  const long long r0 = gw < W ? block_at_unit(prefix, B, Hkv, cost, gw * NU / W) : 0;
  const long long r1 = gw < W ? block_at_unit(prefix, B, Hkv, cost, (gw + 1) * NU / W) : 0;
  const bool active = r0 < r1;  // warps past W, or whose units hold no block, have nothing to do
  // a segment of nblk blocks has at most (nblk - 1) W / N + 2 parts: only
  // with a segment of more than kGroupedAbove parts are the group counters used
  const bool may_group =
      static_cast<long long>(max_blk - 1) * W >= static_cast<long long>(kGroupedAbove - 1) * N;

  const uint32_t bar0 = smem_addr(&bars[warp * ST]);
  const uint32_t stage0 = base + warp * ST * C::kStage;
  // K/V are read once per call: keep them from evicting the block tables,
  // lengths, q and split partials that later reads want from L2
  const uint64_t l2_policy = l2_evict_first_policy();
  if (active && lane == 0) {
    for (int s = 0; s < ST; ++s) mbar_init(bar0 + 8 * s, C::kArrivals);
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  __syncwarp();

  // ---- producer: this warp's blocks in order. Block ids come 32 at a time:
  // lane i holds the kv head and physical block of the warp's block
  // win_base + i; the next window's table reads are in flight while the
  // current window is used, so no TMA issue waits for a block-table read.
  const long long nmine = r1 - r0;
  auto load_window = [&](long long wbase, int& kvh_o, int& phys_o) {
    kvh_o = 0;
    phys_o = 0;
    const long long r = r0 + wbase + lane;
    if (r < r1) {
      int lo = 0, hi = B - 1;  // last b with prefix[b] * Hkv <= r (it has blocks)
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (static_cast<long long>(prefix[mid]) * Hkv <= r) lo = mid;
        else hi = mid - 1;
      }
      const int nb = prefix[lo + 1] - prefix[lo];
      const long long off = r - static_cast<long long>(prefix[lo]) * Hkv;
      kvh_o = static_cast<int>(off / nb);
      int blk = static_cast<int>(off % nb);
      if (WIN)
        blk = seq_window<BS>(min(max(a.context_lens[lo], 0), a.len_cap), a.window, a.sinks)
                  .logical(blk);
      phys_o = a.block_tables[static_cast<long long>(lo) * a.max_blocks + blk];
    }
  };
  int cur_kvh, cur_phys, nxt_kvh, nxt_phys;
  load_window(0, cur_kvh, cur_phys);
  load_window(32, nxt_kvh, nxt_phys);
  // bf16: the warp's first kPrefetchTiles tiles into L2 while the previous
  // grid drains. A prefetch consumes nothing (a line the previous grid still
  // writes is served from L2 as written), so it may precede the dependency
  // wait. Measured on the Llama-3-8B-shaped batch 64 (same box each line): no
  // prefetch 92.0 us per step, the first 2 tiles 89.4, 4 tiles 88.0; on
  // another box 3 / 4 / 5 / 6 tiles 85.3 / 84.6 / 85.5 / 87.1, 8 tiles worse
  // again (the prefetches then compete with the previous grid's tail); the
  // windowed steps gain 0.4-1 us more. The 8-bit instantiations, bound by
  // instruction latency, gain nothing (4 tiles: E4M3 1 % slower).
  if constexpr (!Q8) {
    if (lane < kPrefetchTiles && lane < nmine) {
      const int pp = cur_phys >= 0 && cur_phys < a.num_blocks ? cur_phys : 0;
      tma_prefetch_4d(&kmap, 0, pp * BS, 0, cur_kvh);
      tma_prefetch_4d(&vmap, 0, pp * BS, 0, cur_kvh);
    }
  }

  // ---- from here on: memory the previous launch may write
  grid_dependency_wait();
  // sequences without keys: zero output rows (no warp owns any of their
  // blocks). Sequence b is checked by CTA b mod gridDim.x, so no CTA scans
  // more than ceil(B / gridDim.x) of them.
  for (int b = blockIdx.x; b < B; b += gridDim.x) {
    if (prefix[b + 1] != prefix[b]) continue;  // uniform over the CTA
    uint4* const row = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) +
                                                static_cast<long long>(b) * a.num_heads * D);
    for (int i = threadIdx.x; i < a.num_heads * (D / 8); i += NW * 32) row[i] = make_uint4(0, 0, 0, 0);
  }
  if (!active) return;

  long long win_base = 0;
  int issued = 0;
  // test hook (off: -1): this warp leaves one copy unissued, so that its
  // bounded wait for the block runs out; nothing is in flight on that stage
  const int skip_copy = (blockIdx.x == 0 && warp == 0) ? a.debug_skip_copy : -1;
  auto issue_pending = [&]() {
    if (issued >= nmine) return;
    if (issued - win_base == 32) {
      win_base += 32;
      cur_kvh = nxt_kvh;
      cur_phys = nxt_phys;
      load_window(win_base + 32, nxt_kvh, nxt_phys);
    }
    const int i = static_cast<int>(issued - win_base);
    const int kvh = __shfl_sync(kFull, cur_kvh, i);
    int phys = __shfl_sync(kFull, cur_phys, i);
    if (phys < 0 || phys >= a.num_blocks) {
      if (lane == 0) report_error(a.err, PA_DEVERR_BLOCK_RANGE);
      phys = 0;  // stay inside the pool; the result is flagged as invalid
    }
    if (issued != skip_copy) {
      const int s = issued % ST;
      const uint32_t bar = bar0 + 8 * s;
      if constexpr (Q8)
        copy_scales<BS>(a, scale_base + ((warp * ST + s) * 2) * BS * 4,
                        (static_cast<long long>(phys) * Hkv + kvh) * BS, bar, lane);
      if (lane == 0) {
        // the K and V tiles, one tensor copy each (all 128-byte subtiles)
        const uint32_t kt = stage0 + s * C::kStage;
        mbar_arrive_expect_tx(bar, C::kTx);
        tma_load_4d(kt, &kmap, bar, 0, phys * BS, 0, kvh, l2_policy);
        tma_load_4d(kt + C::kTile, &vmap, bar, 0, phys * BS, 0, kvh, l2_policy);
      }
    }
    ++issued;
  };
  for (int s = 0; s < ST; ++s) issue_pending();
  // This warp's share of the segment arrival counters is tagged with the
  // call's epoch once its first block has been attended to (off the path to
  // the first block; an arrival that comes earlier tags the word itself).
  auto tag_my_counters = [&]() {
    const long long nctr = static_cast<long long>(B) * Hkv;
    const long long per = (nctr + W - 1) / W;
    tag_counters(a.seg_counters, gw * per, min(nctr, (gw + 1) * per),
                 may_group ? a.grp_counters + 2 * gw : nullptr, a.epoch, lane);
  };

  // ---- consumer: pieces in order. The next piece's q is fetched before the
  // current piece's result is written, so its latency overlaps the write,
  // the arrival and any merge.
  Piece cp;
  piece_first(cp, prefix, B, Hkv, r0, r1);
  const float sl2 = a.scale_log2;
  int consumed = 0;
  bool ok = true;
  uint32_t qraw[D / 16][2];
  if (cp.valid) fetch_q<D, Q8>(a, cp.b, cp.kvh, lane, qraw);
  while (ok && cp.valid) {
    uint32_t qa[D / 16][2];
    float q_inv;
    finish_q<D, Q8>(qraw, qa, q_inv);
    const float sl2p = sl2 * q_inv;
    const int L = min(max(a.context_lens[cp.b], 0), a.len_cap);
    const SeqWindow sw = seq_window<BS>(L, WIN ? a.window : 0, a.sinks);
    float acc[D / 16][4];
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
    float m_run = -INFINITY, l_run = 0.f, vfac = 1.f;
    const bool whole = cp.lo == 0 && cp.hi == cp.nblk;
    unsigned long long seen = 0ull;  // the segment's arrival counter near the piece's end
    for (int vb = cp.lo; vb < cp.hi; ++vb) {
      const int blk = sw.logical(vb);  // visible block -> logical block
      const int s = consumed % ST;
      const bool got = mbar_wait(bar0 + 8 * s, (consumed / ST) & 1, a.wait_limit_ns);
      if (!__all_sync(kFull, got)) {
        ok = false;
        if (lane == 0) report_error(a.err, PA_DEVERR_WAIT_TIMEOUT);
        break;
      }
      const uint32_t kt = stage0 + s * C::kStage;
      const float* ksc = scale_ptr + ((warp * ST + s) * 2) * BS;
      if (a.k_new != nullptr && vb == cp.nblk - 1)
        append_row<D, BS, Q8>(base_ptr + (kt - base),
                               const_cast<float*>(scale_ptr) + ((warp * ST + s) * 2) * BS,
                               a.block_tables + static_cast<long long>(cp.b) * a.max_blocks + blk,
                               cp.b * Hkv + cp.kvh, (L - 1) - blk * BS, a, lane);
      attend_block<D, BS, KV, WIN>(kt, kt + C::kTile, base_ptr, base, ksc, ksc + BS, blk * BS, L,
                                    sw.hole_lo, sw.hole_hi, qa, acc, m_run, l_run, vfac, sl2p,
                                    lane);
      if (!whole && vb == cp.hi - 1 && lane == 0)
        seen = ld_relaxed_gpu(a.seg_counters + static_cast<long long>(cp.b) * Hkv + cp.kvh);
      ++consumed;
      __syncwarp();
      issue_pending();
      if (consumed == 1) tag_my_counters();
    }
    if (!ok) break;
    Piece nx = cp;
    piece_next(nx, prefix, B, Hkv, r1);
    if (nx.valid) fetch_q<D, Q8>(a, nx.b, nx.kvh, lane, qraw);
    write_warp_result<D, Q8>(a, cp.b, cp.kvh, whole, 2 * gw + (cp.lo == 0 ? 1 : 0), lane, m_run,
                              l_run, 1.f / vfac, acc);
    if (!whole) {
      const SegParts sp = seg_parts(prefix, B, Hkv, cp.b, cp.kvh, W, cost);
      // Every other part already arrived (counted after publishing its
      // partial): this warp is the segment's last. Its own partial is read
      // only by its own lanes, so it needs neither a fence nor an arrival:
      // the counter is cleared for the next call, a fence orders the other
      // parts' partials before the merge reads them.
      const bool all_others = sp.n <= kGroupedAbove &&
                              __shfl_sync(kFull, static_cast<uint32_t>(seen >> 32) == a.epoch &&
                                                     static_cast<uint32_t>(seen) + 1u ==
                                                         static_cast<uint32_t>(sp.n), 0);
      if (all_others) {
        if (lane == 0) atomicExch(a.seg_counters + static_cast<long long>(cp.b) * Hkv + cp.kvh, 0ull);
        __threadfence();
        __syncwarp();
        merge_segment<D>(a, PartList{sp, 0, 1, sp.n}, cp.b, cp.kvh, true, lane);
        cp = nx;
        continue;
      }
      // publish the partial, count the arrival; the last warp merges the segment
      __threadfence();
      __syncwarp();
      if (sp.n > kGroupedAbove) {
        finish_grouped<D>(a, sp, cp.b, cp.kvh, gw, lane);
      } else {
        int last = 0;
        if (lane == 0)
          last = arrive_last(a.seg_counters + static_cast<long long>(cp.b) * Hkv + cp.kvh, a.epoch,
                             static_cast<uint32_t>(sp.n), a.err);
        if (__shfl_sync(kFull, last, 0)) {
          __threadfence();
          merge_segment<D>(a, PartList{sp, 0, 1, sp.n}, cp.b, cp.kvh, true, lane);
        }
      }
    }
    cp = nx;
  }
  if (!ok) {
    // give copies still in flight a bounded chance to land before exit
    for (int i = consumed; i < issued; ++i)
      (void)mbar_wait(bar0 + 8 * (i % ST), (i / ST) & 1, a.wait_limit_ns);
  }
}

// ============================================================ grid-split path
// Grid (Hkv, B, S): CTA = (kv head, sequence, split of blocks_per_split
// blocks). Used for batches too large for the persistent kernel's prefix.
template <int D, int BS, int NW, int ST, int KV>
__global__ void __launch_bounds__(NW * 32)
    decode_split_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const DecodeArgs a) {
  constexpr bool Q8 = KV != kKvBf16;
  using C = Cfg<D, BS, NW, ST, Q8>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[NW * ST];

  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw);
  const uint32_t scale_base = base + C::kTiles;
  const float* const scale_ptr = reinterpret_cast<const float*>(base_ptr + C::kTiles);
  float* const merge_buf = reinterpret_cast<float*>(base_ptr + C::kTiles + C::kScaleBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kvh = blockIdx.x, b = blockIdx.y, split = blockIdx.z;

  const int L = min(max(a.context_lens[b], 0), a.len_cap);
  const int nblk = (L + BS - 1) / BS;
  const int CB = a.blocks_per_split;
  const int nsplit_seq = (nblk + CB - 1) / CB;
  if (split > 0 && split >= nsplit_seq) return;
  const int blk0 = split * CB;
  const int blk1 = min(nblk, blk0 + CB);
  const int n_my = max(0, (blk1 - blk0 - warp + NW - 1) / NW);

  // Physical block ids of this warp's blocks (lane i holds the i-th).
  int my_phys = 0;
  if (lane < n_my) {
    my_phys = a.block_tables[static_cast<long long>(b) * a.max_blocks + blk0 + warp + lane * NW];
    if (my_phys < 0 || my_phys >= a.num_blocks) {
      report_error(a.err, PA_DEVERR_BLOCK_RANGE);
      my_phys = 0;
    }
  }

  const uint32_t bar0 = smem_addr(&bars[warp * ST]);
  const uint32_t stage0 = base + warp * ST * C::kStage;
  if (lane == 0) {
    for (int s = 0; s < ST; ++s) mbar_init(bar0 + 8 * s, C::kArrivals);
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  __syncwarp();

  auto issue = [&](int i) {
    const int phys = __shfl_sync(kFull, my_phys, i);
    const int s = i % ST;
    const uint32_t bar = bar0 + 8 * s;
    if constexpr (Q8)
      copy_scales<BS>(a, scale_base + ((warp * ST + s) * 2) * BS * 4,
                      (static_cast<long long>(phys) * a.num_kv_heads + kvh) * BS, bar, lane);
    if (lane == 0) {
      const uint32_t kt = stage0 + s * C::kStage;
      mbar_arrive_expect_tx(bar, C::kTx);
      tma_load_4d(kt, &kmap, bar, 0, phys * BS, 0, kvh);
      tma_load_4d(kt + C::kTile, &vmap, bar, 0, phys * BS, 0, kvh);
    }
  };

  const int n_pre = min(ST, n_my);
  for (int i = 0; i < n_pre; ++i) issue(i);

  uint32_t qa[D / 16][2];
  float q_inv;
  load_q<D, Q8>(a, b, kvh, lane, qa, q_inv);
  const float sl2p = a.scale_log2 * q_inv;
  float acc[D / 16][4];
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
  float m_run = -INFINITY, l_run = 0.f, vfac = 1.f;

  bool ok = true;
  int consumed = 0;
  for (int i = 0; i < n_my; ++i) {
    const int s = i % ST;
    const bool got = mbar_wait(bar0 + 8 * s, (i / ST) & 1, a.wait_limit_ns);
    if (!__all_sync(kFull, got)) {
      ok = false;
      break;
    }
    consumed = i + 1;
    const uint32_t kt = stage0 + s * C::kStage;
    const float* ksc = scale_ptr + ((warp * ST + s) * 2) * BS;
    attend_block<D, BS, KV>(kt, kt + C::kTile, base_ptr, base, ksc, ksc + BS,
                             (blk0 + warp + i * NW) * BS, L, 0, 0, qa, acc, m_run, l_run, vfac,
                             sl2p, lane);
    __syncwarp();
    if (i + ST < n_my) issue(i + ST);
  }
  if (!ok) {
    if (lane == 0) report_error(a.err, PA_DEVERR_WAIT_TIMEOUT);
    for (int i = consumed; i < min(n_my, consumed + ST); ++i)
      (void)mbar_wait(bar0 + 8 * (i % ST), (i / ST) & 1, a.wait_limit_ns);
  }
  store_warp_state<D, NW, Q8>(merge_buf, warp, lane, m_run, l_run, 1.f / vfac, acc);
  const bool any_fail = __syncthreads_or(!ok);
  if (any_fail) return;
  // partial slot of (b, kvh, split): the merge kernel below reads these
  const long long slot = (static_cast<long long>(b) * a.num_kv_heads + kvh) * a.num_splits + split;
  merge_warps_and_write<D, NW>(merge_buf, a, b, kvh, nsplit_seq <= 1, slot);
}

// Merge the splits of sequences that needed more than one (grid-split path).
// One warp per (sequence, query head).
template <int D, int BS>
__global__ void __launch_bounds__(128) decode_split_merge_kernel(const DecodeArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long gw = static_cast<long long>(blockIdx.x) * 4 + warp;
  if (gw >= static_cast<long long>(a.batch) * a.num_heads) return;
  const int b = static_cast<int>(gw / a.num_heads);
  const int h = static_cast<int>(gw % a.num_heads);
  const int kvh = h / a.group, g = h % a.group;
  const int L = min(max(a.context_lens[b], 0), a.len_cap);
  const int nblk = (L + BS - 1) / BS;
  const int ns = (nblk + a.blocks_per_split - 1) / a.blocks_per_split;
  if (ns <= 1) return;
  const long long slot0 = (static_cast<long long>(b) * a.num_kv_heads + kvh) * a.num_splits;
  float M = -INFINITY;
  for (int j = lane; j < ns; j += 32) M = fmaxf(M, a.part_ml[((slot0 + j) * 8 + g) * 2]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
  float l = 0.f;
  for (int j = lane; j < ns; j += 32)
    l += a.part_ml[((slot0 + j) * 8 + g) * 2 + 1] * fast_exp2(a.part_ml[((slot0 + j) * 8 + g) * 2] - M);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(kFull, l, o);
  constexpr int V = D / 32;
  float acc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = 0.f;
  for (int j = 0; j < ns; ++j) {
    const float f = fast_exp2(a.part_ml[((slot0 + j) * 8 + g) * 2] - M);
    const float* src = a.part_o + ((slot0 + j) * 8 + g) * D + lane * V;
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] += f * src[v];
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) + gw * D + lane * V;
#pragma unroll
  for (int v = 0; v < V; v += 2)
    *reinterpret_cast<__nv_bfloat162*>(dst + v) = __floats2bfloat162_rn(acc[v] * inv, acc[v + 1] * inv);
}

// ============================================================ host side
constexpr int kWarps = 4;
// Shared-memory budget of one CTA's stage rings (the CTA count per SM follows
// from it); each warp gets kStageBudget / (kWarps * stage) stages, 2 to 8.
constexpr int kStageBudget = 64 * 1024;

constexpr int stages_for(int stage_bytes) {
  return kStageBudget / (kWarps * stage_bytes) < 2 ? 2
         : kStageBudget / (kWarps * stage_bytes) > 8 ? 8
                                                     : kStageBudget / (kWarps * stage_bytes);
}

template <int D, int BS, int KV>
struct Inst {
  static constexpr bool Q8 = KV != kKvBf16;
  static constexpr int kStages = stages_for(Cfg<D, BS, kWarps, 2, Q8>::kStage);
  using C = Cfg<D, BS, kWarps, kStages, Q8>;
  using PC = PCfg<D, BS, kWarps, kStages, Q8>;
  static constexpr int kSplitSmem = 1024 + C::kTiles + C::kScaleBytes + C::kMerge;
  static_assert(kSplitSmem <= 227 * 1024, "shared memory over the per-CTA limit");
  static_assert(PC::kPrefixOff + 1024 + (kMaxPersistentBatch + 1) * 4 <= 227 * 1024,
                "shared memory over the per-CTA limit");

  // Shared memory grows with the batch (its block prefix sums): batches are
  // bucketed by 256 sequences. Per device and bucket, once: allow the
  // largest size any batch needs and record how many CTAs fit on an SM (the
  // persistent grid is that times the SM count, the same for every call with
  // a batch in the bucket).
  static constexpr int kBucket = 256;
  static constexpr int kBuckets = kMaxPersistentBatch / kBucket;
  static int bucket_batch(int batch) {
    return std::max(1, (batch + kBucket - 1) / kBucket) * kBucket;
  }
  static int ctas_per_sm(int batch) {
    static int cached[kMaxDevices][kBuckets] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
    const int bb = bucket_batch(std::min(std::max(batch, 1), kMaxPersistentBatch));
    int& slot = cached[dev][bb / kBucket - 1];
    if (slot > 0) return slot;
    // both variants (with and without a sliding window) get the attribute;
    // the grid is sized by the one with fewer resident CTAs
    auto* k0 = decode_persistent_kernel<D, BS, kWarps, kStages, KV, false>;
    auto* k1 = decode_persistent_kernel<D, BS, kWarps, kStages, KV, true>;
    const int smem_max = PC::smem_bytes(kMaxPersistentBatch);
    const int smem = PC::smem_bytes(bb);
    int n0 = 0, n1 = 0;
    if (cudaFuncSetAttribute(k0, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max) !=
            cudaSuccess ||
        cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n0, k0, kWarps * 32, smem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n1, k1, kWarps * 32, smem) != cudaSuccess)
      return 1;
    slot = std::max(1, std::min(n0, n1));
    return slot;
  }

  static cudaError_t launch(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                            cudaStream_t stream) {
    cudaError_t e;
    const long long rows = static_cast<long long>(a.batch) * a.num_heads;
    if (a.persistent_ctas > 0) {
      auto* k = a.window > 0 ? decode_persistent_kernel<D, BS, kWarps, kStages, KV, true>
                             : decode_persistent_kernel<D, BS, kWarps, kStages, KV, false>;
      (void)ctas_per_sm(a.batch);  // makes sure the shared-memory attribute is set
      // programmatic dependent launch: the prologue may overlap the kernel
      // before this one on the stream (the kernel waits before reading K/V)
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(a.persistent_ctas);
      cfg.blockDim = dim3(kWarps * 32);
      cfg.dynamicSmemBytes = PC::smem_bytes(bucket_batch(a.batch));  // the size the grid assumed
      cfg.stream = stream;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[0].val.programmaticStreamSerializationAllowed = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      return cudaLaunchKernelEx(&cfg, k, kmap, vmap, a);
    }
    auto* k = decode_split_kernel<D, BS, kWarps, kStages, KV>;
    static bool attr_set[kMaxDevices] = {};
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSplitSmem);
      if (e != cudaSuccess) return e;
      attr_set[dev] = true;
    }
    dim3 grid(a.num_kv_heads, a.batch, a.num_splits);
    k<<<grid, kWarps * 32, kSplitSmem, stream>>>(kmap, vmap, a);
    if ((e = cudaGetLastError()) != cudaSuccess || a.num_splits <= 1) return e;
    decode_split_merge_kernel<D, BS><<<static_cast<unsigned>((rows + 3) / 4), 128, 0, stream>>>(a);
    return cudaGetLastError();
  }
};

// Tokens per split of the grid-split path.
constexpr int kSplitTokens = 512;

template <typename F>
auto dispatch(int head_dim, int block_size, int kv, F&& f)
    -> decltype(f(Inst<128, 16, kKvBf16>{})) {
  if (kv == kKvE4m3) {
    if (block_size == 16) return f(Inst<128, 16, kKvE4m3>{});
    return f(Inst<128, 32, kKvE4m3>{});
  }
  if (kv == kKvInt8) {
    if (block_size == 16) return f(Inst<128, 16, kKvInt8>{});
    return f(Inst<128, 32, kKvInt8>{});
  }
  if (head_dim == 128 && block_size == 16) return f(Inst<128, 16, kKvBf16>{});
  if (head_dim == 128 && block_size == 32) return f(Inst<128, 32, kKvBf16>{});
  if (head_dim == 64 && block_size == 16) return f(Inst<64, 16, kKvBf16>{});
  return f(Inst<64, 32, kKvBf16>{});
}

}  // namespace

DecodePlan plan_decode(int batch, int num_heads, int num_kv_heads, int head_dim, int block_size,
                       int kv, int len_cap, int num_sms) {
  DecodePlan p{};
  if (batch <= kMaxPersistentBatch) {
    const int per_sm = dispatch(head_dim, block_size, kv,
                                [&](auto inst) { return decltype(inst)::ctas_per_sm(batch); });
    // No more CTAs than blocks the call can hold (the host-side length
    // bound): at most one warp per block ever gets work, and a CTA without
    // any only runs its prologue. Small problems thus launch a small grid.
    const long long nblk_max = (std::max(len_cap, 0) + block_size - 1) / block_size;
    const long long blocks_max = static_cast<long long>(batch) * nblk_max * num_kv_heads;
    const long long ctas_needed = std::max(1LL, blocks_max);
    p.persistent_ctas = static_cast<int>(std::min<long long>(static_cast<long long>(per_sm) * num_sms,
                                                             ctas_needed));
    p.blocks_per_split = 0;
    p.num_splits = 0;
    // two partial slots per warp, one row per query head of a group (rounded
    // up to a power of two, the merge's lane layout)
    p.partial_slots = 2 * static_cast<size_t>(p.persistent_ctas) * kWarps;
    const int group = std::max(1, num_heads / std::max(1, num_kv_heads));
    p.slot_rows = group <= 1 ? 1 : group <= 2 ? 2 : group <= 4 ? 4 : 8;
    const size_t slot_floats = static_cast<size_t>(p.slot_rows) * (head_dim + 2);
    // partials, prefix sums, 16-byte pad, segment and group arrival counters
    p.workspace_bytes = p.partial_slots * slot_floats * sizeof(float) +
                        (static_cast<size_t>(batch) + 1) * sizeof(int) + 16 +
                        static_cast<size_t>(batch) * num_kv_heads * sizeof(unsigned long long) +
                        p.partial_slots * sizeof(unsigned long long) + 256;
    return p;
  }
  p.persistent_ctas = 0;
  const int max_nblk = (std::max(len_cap, 0) + block_size - 1) / block_size;
  int cb = std::max(1, kSplitTokens / block_size);
  cb = std::min(cb, 32 * kWarps);  // a warp holds its block ids in one register per lane
  p.blocks_per_split = cb;
  p.num_splits = std::max(1, (max_nblk + cb - 1) / cb);
  if (p.num_splits > 65535) {  // grid z limit: widen the splits
    p.blocks_per_split = (max_nblk + 65534) / 65535;
    p.num_splits = (max_nblk + p.blocks_per_split - 1) / p.blocks_per_split;
  }
  p.slot_rows = 8;
  if (p.num_splits <= 1) {
    p.partial_slots = 0;
    p.workspace_bytes = 0;
  } else {
    p.partial_slots = static_cast<size_t>(batch) * num_kv_heads * p.num_splits;
    p.workspace_bytes = p.partial_slots * 8 * (head_dim + 2) * sizeof(float) + 256;
  }
  return p;
}

cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          cudaStream_t stream) {
  if (a.kv != kKvBf16 && a.head_dim != 128) return cudaErrorInvalidValue;
  if ((a.head_dim != 64 && a.head_dim != 128) || (a.block_size != 16 && a.block_size != 32))
    return cudaErrorInvalidValue;
  return dispatch(a.head_dim, a.block_size, a.kv,
                  [&](auto inst) { return decltype(inst)::launch(a, kmap, vmap, stream); });
}

}  // namespace pa
