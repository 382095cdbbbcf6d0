/*
 * Plain, slow CPU oracle for paged-KV-cache attention.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the ground truth that the CUDA path
 * is compared against. Only the test-suite, the smoke check and the bench's
 * CPU-baseline leg may load it. It shares no code, header, table or helper
 * with the CUDA library, and the CUDA library never calls it.
 *
 * Everything is computed in IEEE double precision with straight loops, in the
 * order the definitions are written, with no blocking or fusion. OpenMP only
 * distributes independent (sequence, head) problems over host cores.
 *
 * Sources (web pages on paged KV-cache decode/prefill):
 *   [DEC]  "Decode Phase Attention Forward Pass" (lzwjava.github.io),
 *          sections 2-4: context_lens counts the token just stored; keys are
 *          read per position through block_tables as k_cache[block, offset];
 *          GQA repeats each KV head num_heads/num_kv_heads times
 *          (repeat_interleave on the head axis); no causal mask in decode;
 *          caveat section: zero-padding to max_len distorts the softmax, so
 *          exactly context_len keys are used.
 *   [GLO]  "Decode Phase" glossary (inferensys.com): q.K^T scores, softmax,
 *          weighted sum of V; FP8 / INT8 KV-cache quantisation; for long
 *          contexts, sliding window attention (only the most recent W tokens)
 *          and attention sinks as in StreamingLLM (the initial tokens kept).
 *   [TVL]  "tiny-vllm part 05" (jaehun.me), section "Gathering K/V into a
 *          batched buffer and scattering into blocks": a token at position p
 *          lives in logical block p / BLOCK_SIZE at offset p % BLOCK_SIZE.
 *          Section "Attention is finished off by pagedAttentionKernel":
 *          online softmax over the blocks of a sequence.
 *   [PRE]  "Prefill Forward Prefix Caching Explained" (lzwjava.github.io):
 *          packed varlen q with cu_seqlens (Fact 1), cached_len = kv_len -
 *          q_len (key bookkeeping line), bottom-right causal mask: query i
 *          sees key j iff j <= i + cached_len (the 2x5 example).
 *
 * Readings where the pages are silent (each is also listed in the design
 * notes): slot = physical_block * block_size + offset, negative slot = skip;
 * cache layout (num_blocks, block_size, num_kv_heads, head_dim) row-major for
 * both K and V; FP8 is OCP E4M3 with one fp32 scale per (slot, kv head) in a
 * (num_blocks, num_kv_heads, block_size) array (one head's scales for one
 * block are contiguous); INT8 is a signed byte times the same kind of scale
 * (symmetric, no zero point); a sliding window of W tokens with S sinks
 * keeps keys p < S and p >= context_len - W; context_len 0 gives a zero
 * output row; a prefill sequence with q_len > kv_len is invalid input.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_OK = 0, OR_ERR_ARG = 1, OR_ERR_RANGE = 2, OR_ERR_NOMEM = 3 };
enum { OR_KV_BF16 = 0, OR_KV_E4M3 = 1, OR_KV_INT8 = 2 };

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* OCP 8-bit floating point, E4M3 flavour ("fn": finite, no infinities):
 * 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits.
 * exponent field 0 -> subnormal  (-1)^s * (m/8) * 2^(1-7)
 * S.1111.111       -> NaN (the only non-finite encoding)
 * otherwise        -> (-1)^s * (1 + m/8) * 2^(e-7)                      */
double oracle_e4m3_to_double(uint8_t code) {
  int s = (code >> 7) & 1;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double mag;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, 1 - 7);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -mag : mag;
}

void oracle_e4m3_decode_array(const uint8_t* codes, int64_t n, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_to_double(codes[i]);
}

/* ------------------------------------------------------------------------ */
/* store_kvcache: write each new token's K and V rows into its cache slot.
 * [TVL] scatter section: block = slot / block_size, offset = slot % block_size.
 * Bytes are copied verbatim.
 * k, v: (T, row_bytes); caches: (num_slots, row_bytes) where
 * num_slots = num_blocks * block_size and row_bytes = Hkv * D * elem_size.
 * Optional FP8 scales (T, Hkv) go to scale caches (num_blocks, Hkv, block_size):
 * head h of the token lands at [block][h][offset]. */
int oracle_store_kv(const uint8_t* k, const uint8_t* v, const int64_t* slot_mapping,
                    int64_t T, int64_t row_bytes, int64_t num_slots, int64_t block_size,
                    uint8_t* k_cache, uint8_t* v_cache,
                    const float* k_scale_new, const float* v_scale_new,
                    float* k_scale_cache, float* v_scale_cache, int64_t hkv) {
  if (!k || !v || !slot_mapping || !k_cache || !v_cache || row_bytes <= 0 || block_size <= 0)
    return OR_ERR_ARG;
  for (int64_t t = 0; t < T; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue; /* padding token: nothing is written */
    if (slot >= num_slots) return OR_ERR_RANGE;
    int64_t block = slot / block_size, offset = slot % block_size;
    memcpy(k_cache + slot * row_bytes, k + t * row_bytes, (size_t)row_bytes);
    memcpy(v_cache + slot * row_bytes, v + t * row_bytes, (size_t)row_bytes);
    for (int64_t h = 0; h < hkv; ++h) {
      if (k_scale_new && k_scale_cache)
        k_scale_cache[(block * hkv + h) * block_size + offset] = k_scale_new[t * hkv + h];
      if (v_scale_new && v_scale_cache)
        v_scale_cache[(block * hkv + h) * block_size + offset] = v_scale_new[t * hkv + h];
    }
  }
  return OR_OK;
}

/* ------------------------------------------------------------------------ */
typedef struct {
  const void* k_cache;
  const void* v_cache;
  const float* k_scale;
  const float* v_scale;
  int dtype;
  int64_t num_blocks;
  int block_size, hkv, d;
} or_cache;

/* Element (slot, kv head, dim) of a cache, widened to double (times the
 * per-(slot, head) scale for E4M3 and INT8, stored at [block][head][offset]). */
static double cache_elem(const or_cache* c, const void* base, const float* scale,
                         int64_t slot, int g, int dim) {
  int64_t idx = (slot * c->hkv + g) * c->d + dim;
  if (c->dtype == OR_KV_BF16) return bf16_to_double(((const uint16_t*)base)[idx]);
  int64_t block = slot / c->block_size, offset = slot % c->block_size;
  double sc = (double)scale[(block * c->hkv + g) * c->block_size + offset];
  if (c->dtype == OR_KV_INT8) return (double)((const int8_t*)base)[idx] * sc;
  return oracle_e4m3_to_double(((const uint8_t*)base)[idx]) * sc;
}

/* Whether key position p is attended by the query of a sequence of n_keys
 * tokens ([GLO], long-context bullets): with a sliding window (window > 0)
 * only the last `window` keys and the first `sinks` keys; otherwise all. */
static int key_visible(int64_t p, int64_t n_keys, int64_t window, int64_t sinks) {
  if (window <= 0) return 1;
  return p < sinks || p >= n_keys - window;
}

/* Slot of logical position p of sequence b, through the block table
 * ([TVL]: logical block p / block_size, offset p % block_size;
 *  [DEC] section 2: k_cache[block, offset]). Returns -1 if out of range. */
static int64_t slot_of(const or_cache* c, const int32_t* block_tables, int max_blocks,
                       int b, int64_t p) {
  int64_t logical = p / c->block_size;
  int64_t offset = p % c->block_size;
  if (logical >= max_blocks) return -1;
  int64_t phys = block_tables[(int64_t)b * max_blocks + logical];
  if (phys < 0 || phys >= c->num_blocks) return -1;
  return phys * c->block_size + offset;
}

/* Softmax attention of one query row over keys 0..n_keys-1 of sequence b,
 * kv head g: out[d] = sum_p softmax(s)_p * V[p][d], s_p = scale * q.K[p].
 * The softmax subtracts the maximum before exponentiating (exact in real
 * arithmetic, avoids overflow). n_keys == 0 yields a zero row. */
static int attend_row(const or_cache* c, const int32_t* block_tables, int max_blocks, int b,
                      int g, const uint16_t* qrow, int64_t n_keys, double scale,
                      int64_t window, int64_t sinks, double* s /* scratch n_keys */,
                      double* out) {
  const int D = c->d;
  for (int dd = 0; dd < D; ++dd) out[dd] = 0.0;
  if (n_keys <= 0) return OR_OK;
  double m = -INFINITY;
  for (int64_t p = 0; p < n_keys; ++p) {
    if (!key_visible(p, n_keys, window, sinks)) continue;
    int64_t slot = slot_of(c, block_tables, max_blocks, b, p);
    if (slot < 0) return OR_ERR_RANGE;
    double dot = 0.0;
    for (int dd = 0; dd < D; ++dd)
      dot += bf16_to_double(qrow[dd]) * cache_elem(c, c->k_cache, c->k_scale, slot, g, dd);
    s[p] = scale * dot;
    if (s[p] > m) m = s[p];
  }
  double l = 0.0;
  for (int64_t p = 0; p < n_keys; ++p) {
    if (!key_visible(p, n_keys, window, sinks)) continue;
    s[p] = exp(s[p] - m);
    l += s[p];
  }
  for (int64_t p = 0; p < n_keys; ++p) {
    if (!key_visible(p, n_keys, window, sinks)) continue;
    int64_t slot = slot_of(c, block_tables, max_blocks, b, p);
    double w = s[p] / l;
    for (int dd = 0; dd < D; ++dd)
      out[dd] += w * cache_elem(c, c->v_cache, c->v_scale, slot, g, dd);
  }
  return OR_OK;
}

static int check_cache(const or_cache* c) {
  if (!c->k_cache || !c->v_cache) return OR_ERR_ARG;
  if (c->block_size <= 0 || c->hkv <= 0 || c->d <= 0 || c->num_blocks <= 0) return OR_ERR_ARG;
  if (c->dtype != OR_KV_BF16 && c->dtype != OR_KV_E4M3 && c->dtype != OR_KV_INT8)
    return OR_ERR_ARG;
  if (c->dtype != OR_KV_BF16 && (!c->k_scale || !c->v_scale)) return OR_ERR_ARG;
  return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Single-query decode ([DEC] sections 2-4, [GLO]): for every sequence b and
 * query head h, attend over exactly context_lens[b] keys (no padding), using
 * kv head g = h / (num_heads / num_kv_heads). q: (B, H, D) bf16 bits;
 * out: (B, H, D) double. window > 0 restricts the keys to the last `window`
 * and the first `sinks` positions ([GLO]); window <= 0 attends to all. */
int oracle_decode_window(const uint16_t* q, const void* k_cache, const void* v_cache,
                         int dtype, const float* k_scale, const float* v_scale,
                         int64_t num_blocks, int block_size, int hkv, int d,
                         const int32_t* block_tables, int max_blocks,
                         const int32_t* context_lens, int batch, int num_heads, double scale,
                         int64_t window, int64_t sinks, double* out, int nthreads) {
  or_cache c = {k_cache, v_cache, k_scale, v_scale, dtype, num_blocks, block_size, hkv, d};
  int st = check_cache(&c);
  if (st) return st;
  if (!q || !block_tables || !context_lens || !out || batch < 0 || num_heads <= 0) return OR_ERR_ARG;
  if (num_heads % hkv) return OR_ERR_ARG;
  const int group = num_heads / hkv;
  int64_t max_len = 0;
  for (int b = 0; b < batch; ++b) {
    if (context_lens[b] < 0 || (int64_t)context_lens[b] > (int64_t)max_blocks * block_size)
      return OR_ERR_RANGE;
    if (context_lens[b] > max_len) max_len = context_lens[b];
  }
  int err = OR_OK;
  const int64_t n_rows = (int64_t)batch * num_heads;
#pragma omp parallel num_threads(nthreads > 0 ? nthreads : 1)
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
    if (!s) {
#pragma omp atomic write
      err = OR_ERR_NOMEM;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; ++r) {
      if (!s) continue;
      int b = (int)(r / num_heads), h = (int)(r % num_heads);
      int g = h / group;
      int e = attend_row(&c, block_tables, max_blocks, b, g, q + r * d, context_lens[b], scale,
                         window, sinks, s, out + r * d);
      if (e) {
#pragma omp atomic write
        err = e;
      }
    }
    free(s);
  }
  return err;
}

/* ------------------------------------------------------------------------ */
/* Split-K form of the same decode (flash-decoding): keys of each sequence are
 * cut into consecutive chunks of split_tokens; chunk j yields its own maximum
 * m_j, sum l_j = sum exp(s - m_j) and unnormalised o_j = sum exp(s - m_j) V;
 * then M = max_j m_j, l = sum_j l_j exp(m_j - M), o = sum_j o_j exp(m_j - M) / l.
 * This is the online-softmax rescaling that [TVL] describes for
 * pagedAttentionKernel, applied once per chunk. Used to pin the merge step. */
/* Decode over all context_len keys: the window-free case. */
int oracle_decode(const uint16_t* q, const void* k_cache, const void* v_cache, int dtype,
                  const float* k_scale, const float* v_scale, int64_t num_blocks,
                  int block_size, int hkv, int d, const int32_t* block_tables, int max_blocks,
                  const int32_t* context_lens, int batch, int num_heads, double scale,
                  double* out, int nthreads) {
  return oracle_decode_window(q, k_cache, v_cache, dtype, k_scale, v_scale, num_blocks,
                              block_size, hkv, d, block_tables, max_blocks, context_lens, batch,
                              num_heads, scale, 0, 0, out, nthreads);
}

int oracle_decode_split(const uint16_t* q, const void* k_cache, const void* v_cache, int dtype,
                        const float* k_scale, const float* v_scale, int64_t num_blocks,
                        int block_size, int hkv, int d, const int32_t* block_tables,
                        int max_blocks, const int32_t* context_lens, int batch, int num_heads,
                        double scale, int split_tokens, double* out) {
  or_cache c = {k_cache, v_cache, k_scale, v_scale, dtype, num_blocks, block_size, hkv, d};
  int st = check_cache(&c);
  if (st) return st;
  if (split_tokens <= 0 || num_heads % hkv) return OR_ERR_ARG;
  const int group = num_heads / hkv;
  double* oj = (double*)malloc(sizeof(double) * (size_t)d);
  if (!oj) return OR_ERR_NOMEM;
  for (int b = 0; b < batch; ++b) {
    int64_t L = context_lens[b];
    for (int h = 0; h < num_heads; ++h) {
      const uint16_t* qrow = q + ((int64_t)b * num_heads + h) * d;
      double* o = out + ((int64_t)b * num_heads + h) * d;
      int g = h / group;
      int64_t n_split = (L + split_tokens - 1) / split_tokens;
      double M = -INFINITY, lsum = 0.0;
      double* ms = (double*)malloc(sizeof(double) * (size_t)(n_split > 0 ? n_split : 1));
      double* ls = (double*)malloc(sizeof(double) * (size_t)(n_split > 0 ? n_split : 1));
      double* os = (double*)malloc(sizeof(double) * (size_t)(n_split > 0 ? n_split : 1) * d);
      if (!ms || !ls || !os) {
        free(ms); free(ls); free(os); free(oj);
        return OR_ERR_NOMEM;
      }
      for (int64_t j = 0; j < n_split; ++j) {
        int64_t p0 = j * split_tokens, p1 = p0 + split_tokens < L ? p0 + split_tokens : L;
        double m = -INFINITY, l = 0.0;
        for (int dd = 0; dd < d; ++dd) oj[dd] = 0.0;
        for (int64_t p = p0; p < p1; ++p) {
          int64_t slot = slot_of(&c, block_tables, max_blocks, b, p);
          double dot = 0.0;
          for (int dd = 0; dd < d; ++dd)
            dot += bf16_to_double(qrow[dd]) * cache_elem(&c, c.k_cache, c.k_scale, slot, g, dd);
          double sc = scale * dot;
          if (sc > m) m = sc;
        }
        for (int64_t p = p0; p < p1; ++p) {
          int64_t slot = slot_of(&c, block_tables, max_blocks, b, p);
          double dot = 0.0;
          for (int dd = 0; dd < d; ++dd)
            dot += bf16_to_double(qrow[dd]) * cache_elem(&c, c.k_cache, c.k_scale, slot, g, dd);
          double w = exp(scale * dot - m);
          l += w;
          for (int dd = 0; dd < d; ++dd) oj[dd] += w * cache_elem(&c, c.v_cache, c.v_scale, slot, g, dd);
        }
        ms[j] = m;
        ls[j] = l;
        memcpy(os + j * d, oj, sizeof(double) * (size_t)d);
        if (m > M) M = m;
      }
      for (int dd = 0; dd < d; ++dd) o[dd] = 0.0;
      for (int64_t j = 0; j < n_split; ++j) {
        double f = exp(ms[j] - M);
        lsum += ls[j] * f;
        for (int dd = 0; dd < d; ++dd) o[dd] += os[j * d + dd] * f;
      }
      if (n_split > 0)
        for (int dd = 0; dd < d; ++dd) o[dd] /= lsum;
      free(ms); free(ls); free(os);
    }
  }
  free(oj);
  return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Bottom-right-aligned causal mask ([PRE], "how the causal mask handles the
 * prefix"): query row i of q_len rows may see key j of kv_len keys iff
 * j <= i + (kv_len - q_len). mask: (q_len, kv_len) bytes, 1 = visible. */
int oracle_causal_mask(int q_len, int kv_len, uint8_t* mask) {
  if (q_len < 0 || kv_len < 0 || q_len > kv_len || !mask) return OR_ERR_ARG;
  int cached = kv_len - q_len;
  for (int i = 0; i < q_len; ++i)
    for (int j = 0; j < kv_len; ++j) mask[(int64_t)i * kv_len + j] = (j <= i + cached) ? 1 : 0;
  return OR_OK;
}

/* Varlen prefix-cached prefill ([PRE] Facts 1-2, branch 1, the mask): the
 * new tokens of sequence b are packed rows cu_q[b] .. cu_q[b+1]-1 of q; the
 * keys are kv positions 0 .. kv_len-1 read from the paged cache (the new
 * tokens' K/V were stored there first); query row i (0-based within the
 * sequence) attends to keys 0 .. i + cached_len with cached_len = kv_len -
 * q_len. q: (total_q, H, D) bf16 bits; out: (total_q, H, D) double. */
int oracle_prefill(const uint16_t* q, const void* k_cache, const void* v_cache, int dtype,
                   const float* k_scale, const float* v_scale, int64_t num_blocks,
                   int block_size, int hkv, int d, const int32_t* block_tables, int max_blocks,
                   const int32_t* cu_q, const int32_t* cu_k, int batch, int num_heads,
                   double scale, double* out, int nthreads) {
  or_cache c = {k_cache, v_cache, k_scale, v_scale, dtype, num_blocks, block_size, hkv, d};
  int st = check_cache(&c);
  if (st) return st;
  if (!q || !block_tables || !cu_q || !cu_k || !out || batch < 0 || num_heads <= 0) return OR_ERR_ARG;
  if (num_heads % hkv) return OR_ERR_ARG;
  if (cu_q[0] != 0 || cu_k[0] != 0) return OR_ERR_ARG;
  const int group = num_heads / hkv;
  int64_t max_k = 0;
  for (int b = 0; b < batch; ++b) {
    int64_t ql = (int64_t)cu_q[b + 1] - cu_q[b], kl = (int64_t)cu_k[b + 1] - cu_k[b];
    if (ql < 0 || kl < 0 || ql > kl) return OR_ERR_RANGE;
    if (kl > (int64_t)max_blocks * block_size) return OR_ERR_RANGE;
    if (kl > max_k) max_k = kl;
  }
  const int64_t total_q = cu_q[batch];
  const int64_t n_rows = total_q * num_heads;
  int err = OR_OK;
#pragma omp parallel num_threads(nthreads > 0 ? nthreads : 1)
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(max_k > 0 ? max_k : 1));
    if (!s) {
#pragma omp atomic write
      err = OR_ERR_NOMEM;
    }
#pragma omp for schedule(dynamic, 4)
    for (int64_t r = 0; r < n_rows; ++r) {
      if (!s) continue;
      int64_t row = r / num_heads;
      int h = (int)(r % num_heads);
      int b = 0;
      while (b + 1 < batch && cu_q[b + 1] <= row) ++b;
      int64_t i = row - cu_q[b];
      int64_t kv_len = (int64_t)cu_k[b + 1] - cu_k[b];
      int64_t q_len = (int64_t)cu_q[b + 1] - cu_q[b];
      int64_t cached = kv_len - q_len;
      /* visible keys: j = 0 .. i + cached, i.e. i + cached + 1 of them */
      int e = attend_row(&c, block_tables, max_blocks, b, h / group,
                         q + (row * num_heads + h) * d, i + cached + 1, scale, 0, 0, s,
                         out + (row * num_heads + h) * d);
      if (e) {
#pragma omp atomic write
        err = e;
      }
    }
    free(s);
  }
  return err;
}
