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
//   * A query tile is 128 rows = 128/G tokens x the G query heads of one kv
//     head (GQA packing: every K/V tile serves the whole head group). One CTA
//     per SM holds TWO consecutive query tiles of a (sequence, kv head) and
//     walks the K/V tiles (128 keys) they need, so every K/V byte brought in
//     serves 256 query rows.
//   * Warp 8 streams the two Q tiles once and the K tiles, warp 10 the V
//     tiles, each through its own 2-stage ring (one 3-D TMA box per physical
//     block and 64-dim half, 128B-swizzled). Block ids are read 32 at a
//     time, a window ahead, so no copy waits for a block-table read; blocks
//     past the last needed key are fetched out of bounds so TMA fills them
//     with zeros.
//   * Warp 9 issues the tensor-core MMAs (tcgen05, fp32 accumulation in TMEM)
//     per key tile n: P_0 V(n), S_0 = Q_0 K(n+1)^T, P_1 V(n), S_1 = Q_1
//     K(n+1)^T. P_i is stored over S_i, so S_i(n+1) waits for P_i V(n) to
//     finish; while one tile's softmax runs, the tensor pipe works on the
//     other's. Its waits suspend in mbarrier try_wait: a spinning warp would
//     take issue slots from the softmax warps that share its scheduler.
//   * Warps 0-3 (tile 0) and 4-7 (tile 1) own one TMEM lane (= query row)
//     each: read the S row, apply the bottom-right mask only on tiles that
//     reach past the row's last visible key, run the online softmax in base 2
//     (the running max is only raised, and O rescaled, when it grows by more
//     than 2^8, which keeps P <= 256 and leaves O/l unchanged), write P as
//     bf16 into the S columns, and at the end normalise O and store bf16 rows.
//   * P precision: one bf16 rounding of P is 2^-9 relative per weight. Over
//     many keys the errors average out (worst |error| ~4e-3 at 128 keys in
//     20k random rows, falling with more keys), but a row that sees only a
//     few keys keeps its weights' rounding whole: 2-4 keys reached 1.0-1.1e-2
//     before the output's own bf16 rounding. So on key tile 0 of a query tile
//     whose first row sees fewer than 128 keys (all of such a row's keys lie
//     in tile 0), P goes in as two bf16 terms, bf16(p) in columns 0..63 and
//     bf16(p - bf16(p)) in columns 64..127 of S, and that P.V takes 16 MMAs
//     instead of 8. Tiles of rows with longer prefixes are unchanged; the
//     code's presence costs ~3 % there (measured 124.2 -> 128.4 us on the
//     8-sequence benchmark, whose prefixes are all >= 250 tokens).
//   * TMEM: 512 columns (S0, S1, O0, O1, 128 each); shared memory: Q0, Q1,
//     two K and two V stages (192 KB).
#include <algorithm>
#include <type_traits>

#include "pa_device.cuh"
#include "pa_prefill.h"
#include "pa_tcgen05.cuh"

namespace pa {

namespace {

constexpr int kBM = 128;               // query rows per tile
constexpr int kBN = 128;               // keys per tile
constexpr int kD = 128;                // head_dim
constexpr int kSub = 128 * kBM;        // bytes of one 64-dim (128-byte-wide) half of a 128-row tile
constexpr int kTileBytes = 2 * kSub;   // 32 KB
constexpr int kKStages = 2;            // K ring depth
constexpr int kVStages = 2;            // V ring depth
constexpr int kSmem = 1024 + (2 + kKStages + kVStages) * kTileBytes;
static_assert(kSmem <= 227 * 1024, "shared memory over the per-CTA limit");
static_assert(32 % (kBN / 16) == 0 && 32 % (kBN / 32) == 0, "tiles must not straddle a block-id window");
constexpr int kThreads = 384;          // 2 x 4 softmax warps, K producer, MMA, V producer, idle
// Register split (setmaxnreg): launched at 65536/384 -> 168 per thread; the
// producer/MMA warpgroup drops to 88 so the two softmax warpgroups can hold a
// whole 128-key score row: 2*128*208 + 128*88 = 384*168. (216/72 left the
// MMA warp no room for the two-term P.V below: it spilled or ran slower.)
constexpr int kSoftmaxRegs = 208;
constexpr int kControlRegs = 88;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kControlRegs <= kThreads * 168,
              "register split exceeds the launch allocation");
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// barrier indices
enum {
  BAR_Q = 0,
  BAR_KF = 1,                  // + stage: K tile landed
  BAR_KE = BAR_KF + kKStages,  // + stage: K stage free (the S MMAs reading it done)
  BAR_VF = BAR_KE + kKStages,  // + stage: V tile landed
  BAR_VE = BAR_VF + kVStages,  // + stage: V stage free (the P.V MMAs reading it done)
  BAR_S = BAR_VE + kVStages,   // + tile: S_i ready
  BAR_P = BAR_S + 2,           // + tile: P_i written (4 warps)
  BAR_O = BAR_P + 2,           // + tile: P_i.V done
  BAR_DRAIN = BAR_O + 2,
  NBAR = BAR_DRAIN + 1
};

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
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const PrefillArgs a) {
  constexpr int kBlocksPerTile = kBN / BS;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t bars[NBAR];
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int abort_flag;

  // launched as a programmatic dependent of the store that wrote the new
  // tokens' K/V: wait for it before reading anything
  grid_dependency_wait();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // grid (kv head, sequence, tile pair counted from each sequence's end): CTAs
  // are dispatched x fastest, so every sequence's last pair (its most keys)
  // starts in the first wave
  const int kvh = blockIdx.x, b = blockIdx.y;
  const int G = a.group, TPT = a.tokens_per_tile;

  const int q0 = a.cu_q[b];
  const int q_len = max(a.cu_q[b + 1] - q0, 0);
  const int kv_len = max(a.cu_k[b + 1] - a.cu_k[b], 0);
  const int cached = max(kv_len - q_len, 0);
  const int pair = (q_len + 2 * TPT - 1) / (2 * TPT) - 1 - static_cast<int>(blockIdx.z);
  if (pair < 0) return;
  const int t00 = 2 * pair * TPT;  // first token of query tile 0
  if (t00 >= q_len) return;
  const bool has1 = t00 + TPT < q_len;
  // K/V tiles each query tile needs (keys its last row can see)
  int Tq[2];
  Tq[0] = (min(cached + min(t00 + TPT, q_len), kv_len) + kBN - 1) / kBN;
  Tq[1] = has1 ? (min(cached + min(t00 + 2 * TPT, q_len), kv_len) + kBN - 1) / kBN : 0;
  const int T = max(Tq[0], Tq[1]);
  // P.V takes P as two bf16 terms on key tile 0 of a query tile whose first
  // row sees fewer than kBN keys (every key of such a row lies in tile 0)
  auto two_term = [&](int i) { return cached + t00 + i * TPT < kBN; };
  __nv_bfloat16* const out = static_cast<__nv_bfloat16*>(a.out);
  const int H = a.num_heads;

  if (T == 0) {  // no keys at all (invalid q_len > kv_len = 0): zero rows
    const int rows = (min(t00 + 2 * TPT, q_len) - t00) * G;
    for (int e = threadIdx.x; e < rows * (kD / 8); e += kThreads) {
      const int row = e / (kD / 8), c = e % (kD / 8);
      const int tok = t00 + row / G, g = row % G;
      reinterpret_cast<uint4*>(out + (static_cast<long long>(q0 + tok) * H + kvh * G + g) * kD)[c] =
          make_uint4(0, 0, 0, 0);
    }
    return;
  }

  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const base_ptr = smem_raw + (base - raw);
  auto q_s = [&](int i) { return base + i * kTileBytes; };
  auto k_s = [&](int s) { return base + (2 + s) * kTileBytes; };
  auto v_s = [&](int s) { return base + (2 + kKStages + s) * kTileBytes; };
  const uint32_t bar0 = smem_addr(&bars[0]);
  auto bar = [&](int i) { return bar0 + 8u * i; };

  if (threadIdx.x == 0) {
    for (int i = 0; i < NBAR; ++i) mbar_init(bar(i), (i == BAR_P || i == BAR_P + 1) ? 4 : 1);
    abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 9) {
    tc::tmem_alloc(smem_addr(&tmem_slot), kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;
  auto tS = [&](int i) { return tmem + 128u * i; };        // S_i, P_i in its first 64 columns
  auto tO = [&](int i) { return tmem + 256u + 128u * i; };  // O_i

  if (warp >= 8) {
   asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kControlRegs));
   if (warp == 8 || warp == 10) {
    // ------------------------------------------------------------ producers
    // warp 8 streams Q and the K tiles, warp 10 the V tiles, each as far
    // ahead as its own ring allows
    const bool is_k = warp == 8;
    const CUtensorMap* map = is_k ? &kmap : &vmap;
    const int full0 = is_k ? BAR_KF : BAR_VF, empty0 = is_k ? BAR_KE : BAR_VE;
    const int NS = is_k ? kKStages : kVStages;
    int issued = 0;
    if (is_k && lane == 0) {
      mbar_arrive_expect_tx(bar(BAR_Q), (has1 ? 2 : 1) * kTileBytes);
      for (int i = 0; i < (has1 ? 2 : 1); ++i) {
        tma_load_3d(q_s(i), &qmap, bar(BAR_Q), 0, kvh * G, q0 + t00 + i * TPT);
        tma_load_3d(q_s(i) + kSub, &qmap, bar(BAR_Q), 64, kvh * G, q0 + t00 + i * TPT);
      }
    }
    const long long bt_row = static_cast<long long>(b) * a.max_blocks;
    const int n_keys = min(cached + min(t00 + 2 * TPT, q_len), kv_len);
    const int oob = a.num_blocks * BS;  // first row past the pool: TMA fills zeros
    // Block ids come 32 at a time (lane l: logical block wb + l, as the pool
    // row of its first key), the next window's table reads in flight while
    // the current one is used.
    auto load_ids = [&](int wb) {
      const int lb = wb + lane;
      int rc = oob;
      if (lb * BS < n_keys && lb < a.max_blocks) {
        const int phys = a.block_tables[bt_row + lb];
        if (phys >= 0 && phys < a.num_blocks) {
          rc = phys * BS;
        } else if (is_k) {
          report_error(a.err, PA_DEVERR_BLOCK_RANGE);
        }
      }
      return rc;
    };
    int wbase = 0;
    int cur_ids = load_ids(0), nxt_ids = load_ids(32);
    for (int n = 0; n < T; ++n) {
      const int s = n % NS;
      if (n * kBlocksPerTile - wbase == 32) {  // tiles never straddle a window
        wbase += 32;
        cur_ids = nxt_ids;
        nxt_ids = load_ids(wbase + 32);
      }
      const int id0 = n * kBlocksPerTile - wbase;
      if (n >= NS && !warp_wait(bar(empty0 + s), ((n - NS) / NS) & 1, &abort_flag, a.err)) break;
      const uint32_t dst = is_k ? k_s(s) : v_s(s);
      if (lane == 0) mbar_arrive_expect_tx(bar(full0 + s), kTileBytes);
#pragma unroll
      for (int i = 0; i < kBlocksPerTile; ++i) {
        const int c = __shfl_sync(0xffffffffu, cur_ids, id0 + i);
        if (lane == 0) {
          tma_load_3d(dst + i * BS * 128, map, bar(full0 + s), 0, kvh, c);
          tma_load_3d(dst + kSub + i * BS * 128, map, bar(full0 + s), 64, kvh, c);
        }
      }
      ++issued;
    }
    if (abort_flag) {
      // let the copies already in flight land before shared memory is released
      for (int n = max(0, issued - NS); n < issued; ++n)
        (void)mbar_wait(bar(full0 + n % NS), (n / NS) & 1);
    }
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issue
    constexpr uint32_t kIdescQK = tc::idesc_bf16_f32(kBM, kBN, false, false);
    constexpr uint32_t kIdescPV = tc::idesc_bf16_f32(kBM, kD, false, true);
    auto issue_s = [&](int i, int n) {  // S_i = Q_i K(n)^T
      const int ks = n % kKStages;
      tc::fence_after_sync();
      if (lane == 0) {
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kSub + (kk & 3) * 32;
          tc::mma_ss(tS(i), tc::smem_desc_sw128(q_s(i) + off, 16, 1024),
                     tc::smem_desc_sw128(k_s(ks) + off, 16, 1024), kIdescQK, kk > 0 ? 1u : 0u);
        }
        tc::commit(bar(BAR_S + i));
      }
      __syncwarp();
    };
    auto issue_pv = [&](int i, int n) {  // O_i += P_i V(n)
      const int vs = n % kVStages;
      const int terms = n == 0 && two_term(i) ? 2 : 1;
      tc::fence_after_sync();
      if (lane == 0) {
#pragma unroll 1
        for (int t = 0; t < terms; ++t) {  // P = hi (columns 0..63) + lo (64..127)
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            tc::mma_ts(tO(i), tS(i) + 64 * t + kk * 8,
                       tc::smem_desc_sw128(v_s(vs) + kk * 16 * 128, kSub, 1024), kIdescPV,
                       (n > 0 || kk > 0 || t > 0) ? 1u : 0u);
        }
        tc::commit(bar(BAR_O + i));
      }
      __syncwarp();
    };
    bool ok = warp_wait(bar(BAR_Q), 0, &abort_flag, a.err) &&
              warp_wait(bar(BAR_KF + 0), 0, &abort_flag, a.err);
    if (ok) {
      for (int i = 0; i < 2; ++i)
        if (Tq[i] > 0) issue_s(i, 0);
      if (lane == 0) tc::commit(bar(BAR_KE + 0));
      __syncwarp();
    }
    for (int n = 0; ok && n < T; ++n) {
      const int s = n % kVStages;
      if (!warp_wait(bar(BAR_VF + s), (n / kVStages) & 1, &abort_flag, a.err)) break;
      const int r0 = kv_len - n * kBN;
      if (r0 > 0 && r0 < kBN && (r0 % BS) != 0) {
        const int r1 = min(kBN, (r0 / BS + 1) * BS);
        uint8_t* vp = base_ptr + (v_s(s) - base);
        for (int e = lane; e < (r1 - r0) * 16; e += 32) {
          const int row = r0 + (e >> 4), c = e & 15;
          *reinterpret_cast<uint4*>(vp + (c >> 3) * kSub + row * 128 + (c & 7) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      const bool more = n + 1 < T;
      const int s1 = (n + 1) % kKStages;
      if (more && !warp_wait(bar(BAR_KF + s1), ((n + 1) / kKStages) & 1, &abort_flag, a.err))
        break;
      for (int i = 0; i < 2; ++i) {
        if (n >= Tq[i]) continue;
        if (!warp_wait(bar(BAR_P + i), n & 1, &abort_flag, a.err)) {
          ok = false;
          break;
        }
        issue_pv(i, n);
        if (n + 1 < Tq[i]) {
          if (!warp_wait(bar(BAR_O + i), n & 1, &abort_flag, a.err)) {
            ok = false;
            break;
          }
          issue_s(i, n + 1);
        }
      }
      if (!ok) break;
      if (lane == 0) {
        tc::commit(bar(BAR_VE + s));
        if (more) tc::commit(bar(BAR_KE + s1));
      }
      __syncwarp();
    }
    if (abort_flag) {  // make sure no MMA is still running before TMEM is freed
      if (lane == 0) tc::commit(bar(BAR_DRAIN));
      __syncwarp();
      (void)mbar_wait(bar(BAR_DRAIN), 0);
    }
   }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
    // ------------------------------------------------------------ softmax
    const int ti = warp / 4;        // query tile of this warpgroup
    const int Tn = Tq[ti];
    const int wq = warp & 3;        // TMEM lane quarter this warp may access
    const int r = 32 * wq + lane;
    const int tok = t00 + ti * TPT + r / G, g = r % G;
    const bool row_valid = tok < q_len;
    const int last_key = min(min(tok, q_len - 1) + cached, kv_len - 1);  // last visible key
    const uint32_t trow = static_cast<uint32_t>(32 * wq) << 16;
    const float sl2 = a.scale_log2;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int n = 0; n < Tn; ++n) {
      if (!warp_wait(bar(BAR_S + ti), n & 1, &abort_flag, a.err)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      const int lim = last_key - n * kBN;  // keys 0..lim of this tile are visible
      // the whole score row in registers: one TMEM round trip
      uint32_t u[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tc::tmem_ld32(tS(ti) + trow + 32 * c, u[c]);
      tc::tmem_wait_ld();
      // most tiles lie wholly left of every row's diagonal: no mask there
      if (!__all_sync(0xffffffffu, lim >= kBN - 1)) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (32 * c + j > lim) u[c][j] = __float_as_uint(-INFINITY);
      }
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        mx = fmaxf(mx, fmaxf(fmaxf(__uint_as_float(u[0][j]), __uint_as_float(u[1][j])),
                             fmaxf(__uint_as_float(u[2][j]), __uint_as_float(u[3][j]))));
      const float m_tile = mx * sl2;
      if (n == 0) {
        m_used = m_tile;
      } else if (__any_sync(0xffffffffu, m_tile > m_used + kRescaleThreshold)) {
        if (!warp_wait(bar(BAR_O + ti), (n - 1) & 1, &abort_flag, a.err)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const float m_new = fmaxf(m_used, m_tile);
        const float alpha = fast_exp2(m_used - m_new);
        uint32_t w[32];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          tc::tmem_ld32(tO(ti) + trow + 32 * c, w);
          tc::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) w[j] = __float_as_uint(__uint_as_float(w[j]) * alpha);
          tc::tmem_st32(tO(ti) + trow + 32 * c, w);
        }
        tc::tmem_wait_st();
        l *= alpha;
        m_used = m_new;
      }
      // P = 2^(s*scale*log2e - m_used) as bf16, keys 64h..64h+63 -> columns 32h..32h+31
      // (masked keys hold -inf: P = 0); pairs of keys share one packed FMA for
      // the exponent argument and one packed add for the row sum
      const uint64_t sl2x2 = tc::f32x2(sl2, sl2), nmx2 = tc::f32x2(-m_used, -m_used);
      uint64_t lsum = tc::f32x2(0.f, 0.f);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t w[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int c = 2 * h + (j >> 4), e = 2 * (j & 15);
          const uint64_t xa = tc::fma_f32x2(
              tc::f32x2(__uint_as_float(u[c][e]), __uint_as_float(u[c][e + 1])), sl2x2, nmx2);
          float x0, x1;
          tc::f32x2_split(xa, x0, x1);
          const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
          lsum = tc::add_f32x2(lsum, tc::f32x2(p0, p1));
          w[j] = pack_bf16x2(p0, p1);
        }
        tc::tmem_st32(tS(ti) + trow + 32 * h, w);
      }
      if (n == 0 && two_term(ti)) {
        // second term of P, p - bf16(p) as bf16, into columns 64..127: P is
        // computed again from the scores (the same operations, the same values)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t w[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int c = 2 * h + (j >> 4), e = 2 * (j & 15);
            const uint64_t xa = tc::fma_f32x2(
                tc::f32x2(__uint_as_float(u[c][e]), __uint_as_float(u[c][e + 1])), sl2x2, nmx2);
            float x0, x1;
            tc::f32x2_split(xa, x0, x1);
            const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
            const uint32_t hi = pack_bf16x2(p0, p1);
            w[j] = pack_bf16x2(p0 - __uint_as_float(hi << 16), p1 - __uint_as_float(hi & 0xffff0000u));
          }
          tc::tmem_st32(tS(ti) + trow + 64 + 32 * h, w);
        }
      }
      {
        float la, lb;
        tc::f32x2_split(lsum, la, lb);
        l += la + lb;
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(BAR_P + ti));
    }
    if (ok && Tn > 0 && warp_wait(bar(BAR_O + ti), (Tn - 1) & 1, &abort_flag, a.err)) {
      tc::fence_after_sync();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      __nv_bfloat16* orow = out + (static_cast<long long>(q0 + tok) * H + kvh * G + g) * kD;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t w[32];
        tc::tmem_ld32(tO(ti) + trow + 32 * c, w);
        tc::tmem_wait_ld();
        if (row_valid) {
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            pk[j] = pack_bf16x2(__uint_as_float(w[2 * j]) * inv, __uint_as_float(w[2 * j + 1]) * inv);
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
  if (warp == 9) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int BS>
cudaError_t launch_bs(const PrefillArgs& a, const CUtensorMap& qmap, const CUtensorMap& kmap,
                      const CUtensorMap& vmap, cudaStream_t stream) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(prefill_kernel<BS>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  // programmatic dependent launch: may start while the preceding store runs
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.num_kv_heads, a.batch, (a.num_qtiles + 1) / 2);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_kernel<BS>, qmap, kmap, vmap, a);
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, const CUtensorMap& qmap, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, cudaStream_t stream) {
  if (a.head_dim != kD || kBM % a.group != 0) return cudaErrorInvalidValue;
  if (a.block_size == 16) return launch_bs<16>(a, qmap, kmap, vmap, stream);
  if (a.block_size == 32) return launch_bs<32>(a, qmap, kmap, vmap, stream);
  return cudaErrorInvalidValue;
}

int prefill_tokens_per_tile(int group) { return kBM / group; }

}  // namespace pa
