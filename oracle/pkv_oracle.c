/*
 * Test infrastructure: a plain, slow, float64 CPU oracle for paged decode
 * attention and for the KV-cache append.  Only tests, the smoke check and the
 * benchmark's CPU-baseline leg may load it; the product path never does.  It
 * shares no code, header or table with the CUDA library.
 *
 * What it restates (page = "KV Cache Engineering: PagedAttention, Continuous
 * Batching, Attention Variants, and the Bandwidth Wall", unless noted):
 *   - "What the KV Cache Stores and Why": each step keeps K,V of earlier
 *     tokens, computes K,V of the new token only, and attends the new query
 *     over all cached K,V.  Attention itself is scaled dot-product attention:
 *     out = softmax(q . K^T * scale) . V over the sequence's tokens.
 *   - "PagedAttention": the cache is a pool of fixed-size physical blocks;
 *     a per-sequence block table maps logical block j to a physical block;
 *     only the last block may be partly filled.
 *   - "Attention Variants": grouped-query attention, query heads partitioned
 *     into groups that share one K/V head (head h uses KV head h / G).
 *   - "Quantized KV Cache / FP8 KV cache": E4M3 storage with a scale,
 *     dequantised on read.  The E4M3 format is the OCP 8-bit floating point
 *     "E4M3FN" encoding: 1 sign, 4 exponent (bias 7), 3 mantissa bits, no
 *     infinities, NaN = S.1111.111, largest finite 448, subnormals down to
 *     2^-9.
 *   - page "KV-Cache Engineering: Paged Attention, Prefix Cache,
 *     Disaggregation (2026)", Q&A on cross-layer KV sharing: every logical
 *     layer has a shared-with pointer naming the cache its group reads.
 *
 * Cache layout (a reading; the pages draw blocks as opaque boxes): K and V
 * are separate arrays [S][NB][Hkv][bs][D], S = cache slots (layer groups).
 * FP8 scales are fp32 [S][NB][Hkv], one per (slot, block, KV head).
 *
 * Everything is computed in double precision, in logical token order, with
 * no blocking, fusion or reordering.  Parallelism (OpenMP, when compiled
 * with it) is only across independent (sequence, head) pairs.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_BAD_ARG (-1)
#define ORACLE_BAD_BLOCK (-2)
#define ORACLE_BAD_SLOT (-3)
#define ORACLE_BAD_CTX (-4)

/* bf16 bit pattern -> double: bf16 is the upper half of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static float bf16_bits_to_float(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* ------------------------------------------------------------------------ */
/* E4M3 (OCP E4M3FN) codec                                                  */
/* ------------------------------------------------------------------------ */

/* Value of one E4M3 code, straight from the field definitions. */
double pkv_oracle_e4m3_decode(uint8_t code) {
  int sign = (code >> 7) & 1;
  int exponent = (code >> 3) & 0xF;
  int mantissa = code & 0x7;
  double mag;
  if (exponent == 0xF && mantissa == 0x7) return NAN; /* the only NaN codes */
  if (exponent == 0)
    mag = ldexp((double)mantissa / 8.0, 1 - 7); /* subnormal: 0.m * 2^(1-bias) */
  else
    mag = ldexp(1.0 + (double)mantissa / 8.0, exponent - 7);
  return sign ? -mag : mag;
}

/* Sorted magnitudes of the 127 non-negative finite codes 0x00..0x7E
 * (the code order is the value order for non-negative codes). */
static double g_e4m3_mag[127];
static int g_e4m3_ready = 0;

static void e4m3_table_init(void) {
  if (g_e4m3_ready) return;
  for (int c = 0; c < 127; ++c) g_e4m3_mag[c] = pkv_oracle_e4m3_decode((uint8_t)c);
  g_e4m3_ready = 1;
}

/* Round a float to E4M3 with round-to-nearest, ties to the even code, and
 * saturation to +-448 for finite values beyond the range (the "satfinite"
 * rule); NaN maps to the canonical NaN 0x7F.  The nearest code is found by
 * searching the sorted magnitude list; a tie goes to the code whose
 * mantissa LSB (= code LSB) is zero. */
uint8_t pkv_oracle_e4m3_encode(float x) {
  e4m3_table_init();
  if (isnan(x)) return 0x7F;
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs((double)x);
  if (a >= g_e4m3_mag[126]) return (uint8_t)(sign | 126); /* 448 and above, incl. inf */
  /* largest code with magnitude <= a */
  int lo = 0, hi = 126;
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (g_e4m3_mag[mid] <= a) lo = mid; else hi = mid;
  }
  if (g_e4m3_mag[hi] <= a) lo = hi;
  int code;
  if (g_e4m3_mag[lo] == a || lo == 126) {
    code = lo;
  } else {
    double dlo = a - g_e4m3_mag[lo];
    double dhi = g_e4m3_mag[lo + 1] - a;
    if (dlo < dhi) code = lo;
    else if (dhi < dlo) code = lo + 1;
    else code = (lo % 2 == 0) ? lo : lo + 1;
  }
  return (uint8_t)(sign | code);
}

void pkv_oracle_e4m3_decode_array(const uint8_t* codes, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = pkv_oracle_e4m3_decode(codes[i]);
}

/* Quantise bf16 values with one float scale each: e4m3(float(x) / scale),
 * the division in IEEE binary32. */
void pkv_oracle_e4m3_quantize_array(const uint16_t* x_bf16, const float* scale_per_elem,
                                    uint8_t* out, int64_t n) {
  e4m3_table_init();
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
  for (int64_t i = 0; i < n; ++i) {
    volatile float q = bf16_bits_to_float(x_bf16[i]) / scale_per_elem[i];
    out[i] = pkv_oracle_e4m3_encode(q);
  }
}

/* ------------------------------------------------------------------------ */
/* INT8 codec ("KV Cache Engineering ...", "INT8 KV cache": symmetric or     */
/* asymmetric integer quantisation with a scale and a zero point)           */
/* ------------------------------------------------------------------------ */

/* Code of x: q = rne(x / scale) + zero, clamped to [lo, 127] with lo = -127
 * for a symmetric page (zero == 0) and -128 otherwise; x / scale in IEEE
 * binary32; NaN gives the zero point. */
int8_t pkv_oracle_int8_encode(float x, float scale, float zero) {
  volatile float t = x / scale;
  if (isnan(t)) return (int8_t)zero;
  double q = nearbyint((double)t) + (double)zero; /* default rounding: to nearest, ties to even */
  double lo = (zero == 0.0f) ? -127.0 : -128.0;
  if (q < lo) q = lo;
  if (q > 127.0) q = 127.0;
  return (int8_t)q;
}

/* Value of a code: (q - zero) * scale. */
double pkv_oracle_int8_decode(int8_t q, float scale, float zero) {
  return ((double)q - (double)zero) * (double)scale;
}

/* ------------------------------------------------------------------------ */
/* KV append: write each new token's K and V into its physical slot         */
/* ------------------------------------------------------------------------ */

/*
 * k_new, v_new: bf16 bits [N][Hkv][D]; slot_mapping[i] = physical block *
 * bs + offset within the block, -1 = padding (skipped).  The token's row
 * [Hkv][D] lands at cache[slot][blk][h][off][:].  bf16 caches receive the
 * bits unchanged; E4M3 caches receive e4m3(float(x) / scale[slot][blk][h]).
 * Returns ORACLE_BAD_SLOT (and writes nothing) if any slot is out of range.
 */
int pkv_oracle_kv_append(const uint16_t* k_new, const uint16_t* v_new,
                         const int64_t* slot_mapping, int32_t N,
                         void* k_cache, void* v_cache, int32_t kind /* 0 bf16, 1 E4M3, 2 INT8 */,
                         const float* k_scale, const float* v_scale,
                         int32_t S, int32_t NB, int32_t Hkv, int32_t bs, int32_t D,
                         int32_t slot) {
  if (slot < 0 || slot >= S || N < 0 || bs <= 0 || D <= 0 || Hkv <= 0) return ORACLE_BAD_ARG;
  const int64_t nslots = (int64_t)NB * bs;
  for (int32_t i = 0; i < N; ++i)
    if (slot_mapping[i] < -1 || slot_mapping[i] >= nslots) return ORACLE_BAD_SLOT;
  e4m3_table_init();
  for (int32_t i = 0; i < N; ++i) {
    int64_t s = slot_mapping[i];
    if (s == -1) continue;
    int64_t blk = s / bs, off = s % bs;
    for (int32_t h = 0; h < Hkv; ++h) {
      int64_t src = ((int64_t)i * Hkv + h) * D;
      int64_t page = (((int64_t)slot * NB + blk) * Hkv + h);
      int64_t dst = (page * bs + off) * D;
      if (kind == 0) {
        memcpy((uint16_t*)k_cache + dst, k_new + src, (size_t)D * 2);
        memcpy((uint16_t*)v_cache + dst, v_new + src, (size_t)D * 2);
      } else if (kind == 2) {
        /* scales are (scale, zero) pairs per page */
        float ks = k_scale[2 * page], kz = k_scale[2 * page + 1];
        float vs = v_scale[2 * page], vz = v_scale[2 * page + 1];
        for (int32_t d = 0; d < D; ++d) {
          ((int8_t*)k_cache)[dst + d] = pkv_oracle_int8_encode(bf16_bits_to_float(k_new[src + d]), ks, kz);
          ((int8_t*)v_cache)[dst + d] = pkv_oracle_int8_encode(bf16_bits_to_float(v_new[src + d]), vs, vz);
        }
      } else {
        float ks = k_scale[page], vs = v_scale[page];
        for (int32_t d = 0; d < D; ++d) {
          volatile float kq = bf16_bits_to_float(k_new[src + d]) / ks;
          volatile float vq = bf16_bits_to_float(v_new[src + d]) / vs;
          ((uint8_t*)k_cache)[dst + d] = pkv_oracle_e4m3_encode(kq);
          ((uint8_t*)v_cache)[dst + d] = pkv_oracle_e4m3_encode(vq);
        }
      }
    }
  }
  return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* Paged decode attention                                                   */
/* ------------------------------------------------------------------------ */

/* Value of cache element (slot, blk, g, row, d), dequantised for E4M3
 * (code * scale) and INT8 ((code - zero) * scale). */
static double cache_value(const void* cache, int32_t kind, const float* scales,
                          int64_t page, int32_t bs, int32_t D, int32_t row, int32_t d) {
  int64_t idx = (page * bs + row) * D + d;
  if (kind == 0) return bf16_bits_to_double(((const uint16_t*)cache)[idx]);
  if (kind == 2) return pkv_oracle_int8_decode(((const int8_t*)cache)[idx], scales[2 * page], scales[2 * page + 1]);
  return pkv_oracle_e4m3_decode(((const uint8_t*)cache)[idx]) * (double)scales[page];
}

/*
 * One decode step for one layer, T >= 1 new query tokens per sequence.
 *   q            bf16 bits [B][T][Hq][D]
 *   k/v_cache    [S][NB][Hkv][bs][D], bf16 bits, E4M3 codes or INT8 codes
 *   k/v_scale    fp32 [S][NB][Hkv] (E4M3) or [S][NB][Hkv][2] (INT8: scale, zero)
 *   block_tables int32 [B][MB]; context_lens int32 [B]
 *   kv_group_ptr int32 [L]: cache slot read by layer l (shared-with pointer)
 *   out          double [B][T][Hq][D]
 *   pairs        optional int32 [npairs][2] list of distinct (b, r), r = t*Hq + h,
 *                to compute (the others are left untouched); NULL computes all.
 * The T new tokens are the last T of the n = context_lens[b] cached tokens
 * (already appended): query token t sits at position n - T + t and attends
 * to positions 0 .. n - T + t (causal among the new tokens).  Row (b, t, h)
 * with m = n - T + t + 1 keys (m <= 0 gives zeros):
 *   K_j = K[slot][table[b][j / bs]][h / G][j % bs][:], j = 0 .. m-1 (V alike)
 *   s_j = double(scale) * sum_d double(q[b][t][h][d]) * K_j[d]
 *   out = sum_j exp(s_j - max s) V_j / sum_j exp(s_j - max s)
 * T = 1 is single-token decode.  Sources: "KV Cache Engineering:
 * PagedAttention, Continuous Batching, Attention Variants, and the Bandwidth
 * Wall", "What the KV Cache Stores and Why" and "PagedAttention"; the T > 1
 * reading follows "KV-Cache Engineering: Paged Attention, Prefix Cache,
 * Disaggregation (2026)", speculative decoding (the target checks the
 * draft's proposed tokens in one parallel pass over the shared cache).
 * Returns ORACLE_BAD_BLOCK / ORACLE_BAD_CTX if a table entry that would be
 * read or a context length is out of range (nothing is read out of bounds).
 */
int pkv_oracle_paged_decode_multi(const uint16_t* q, int32_t B, int32_t T, int32_t Hq,
                                  const void* k_cache, const void* v_cache,
                                  int32_t fp8 /* element kind: 0 bf16, 1 E4M3, 2 INT8 */,
                                  const float* k_scale, const float* v_scale,
                                  int32_t S, int32_t NB, int32_t Hkv, int32_t bs, int32_t D,
                                  const int32_t* block_tables, int32_t MB,
                                  const int32_t* context_lens,
                                  const int32_t* kv_group_ptr, int32_t L, int32_t layer,
                                  float scale, double* out,
                                  const int32_t* pairs, int32_t npairs) {
  if (B < 0 || T <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || bs <= 0 || D <= 0 || MB <= 0)
    return ORACLE_BAD_ARG;
  if (layer < 0 || layer >= L) return ORACLE_BAD_ARG;
  const int32_t slot = kv_group_ptr[layer];
  if (slot < 0 || slot >= S) return ORACLE_BAD_ARG;
  const int32_t G = Hq / Hkv;
  for (int32_t b = 0; b < B; ++b) {
    int32_t n = context_lens[b];
    if (n < 0 || (int64_t)n > (int64_t)MB * bs) return ORACLE_BAD_CTX;
    for (int32_t j = 0; j < (n + bs - 1) / bs; ++j) {
      int32_t blk = block_tables[(int64_t)b * MB + j];
      if (blk < 0 || blk >= NB) return ORACLE_BAD_BLOCK;
    }
  }
  const int32_t rows = T * Hq; /* query rows per sequence */
  const int64_t total = (pairs != NULL) ? npairs : (int64_t)B * rows;
  int32_t maxn = 0;
  for (int32_t b = 0; b < B; ++b) if (context_lens[b] > maxn) maxn = context_lens[b];

#ifdef _OPENMP
#pragma omp parallel
#endif
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(maxn > 0 ? maxn : 1));
    double* acc = (double*)malloc(sizeof(double) * (size_t)D);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int64_t w = 0; w < total; ++w) {
      int32_t b = (pairs != NULL) ? pairs[2 * w] : (int32_t)(w / rows);
      int32_t r = (pairs != NULL) ? pairs[2 * w + 1] : (int32_t)(w % rows);
      int32_t t = r / Hq, h = r % Hq;
      int32_t g = h / G;
      int32_t m = context_lens[b] - T + t + 1; /* keys this query token sees */
      double* o = out + ((int64_t)b * rows + r) * D;
      const uint16_t* qv = q + ((int64_t)b * rows + r) * D;
      for (int32_t d = 0; d < D; ++d) acc[d] = 0.0;
      if (m <= 0) {
        for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
        continue;
      }
      /* logits over the gathered logical sequence */
      double smax = -INFINITY;
      for (int32_t j = 0; j < m; ++j) {
        int32_t blk = block_tables[(int64_t)b * MB + j / bs];
        int64_t page = ((int64_t)slot * NB + blk) * Hkv + g;
        double dot = 0.0;
        for (int32_t d = 0; d < D; ++d)
          dot += bf16_bits_to_double(qv[d]) * cache_value(k_cache, fp8, k_scale, page, bs, D, j % bs, d);
        s[j] = (double)scale * dot;
        if (s[j] > smax) smax = s[j];
      }
      /* softmax weights and the weighted sum of values */
      double z = 0.0;
      for (int32_t j = 0; j < m; ++j) {
        s[j] = exp(s[j] - smax);
        z += s[j];
      }
      for (int32_t j = 0; j < m; ++j) {
        int32_t blk = block_tables[(int64_t)b * MB + j / bs];
        int64_t page = ((int64_t)slot * NB + blk) * Hkv + g;
        double p = s[j] / z;
        for (int32_t d = 0; d < D; ++d)
          acc[d] += p * cache_value(v_cache, fp8, v_scale, page, bs, D, j % bs, d);
      }
      /* the row is stored once, so a (b, r) listed twice cannot interleave */
      for (int32_t d = 0; d < D; ++d) o[d] = acc[d];
    }
    free(acc);
    free(s);
  }
  return ORACLE_OK;
}

/* Single-token decode: T = 1, pairs are (b, h). */
int pkv_oracle_paged_decode(const uint16_t* q, int32_t B, int32_t Hq,
                            const void* k_cache, const void* v_cache, int32_t fp8,
                            const float* k_scale, const float* v_scale,
                            int32_t S, int32_t NB, int32_t Hkv, int32_t bs, int32_t D,
                            const int32_t* block_tables, int32_t MB,
                            const int32_t* context_lens,
                            const int32_t* kv_group_ptr, int32_t L, int32_t layer,
                            float scale, double* out,
                            const int32_t* pairs, int32_t npairs) {
  return pkv_oracle_paged_decode_multi(q, B, 1, Hq, k_cache, v_cache, fp8, k_scale, v_scale, S, NB,
                                       Hkv, bs, D, block_tables, MB, context_lens, kv_group_ptr, L,
                                       layer, scale, out, pairs, npairs);
}

/* ------------------------------------------------------------------------ */
/* Block copy between two pools (copy-on-write of a shared block; moving a  */
/* sequence's blocks to host memory and back)                               */
/* ------------------------------------------------------------------------ */

/*
 * Pools are [num_blocks][block_bytes] for K and V (and [num_blocks][Hkv]
 * fp32 scales for E4M3 pools, NULL otherwise).  Pairs are applied in order:
 * dst[pairs[i][1]] = src[pairs[i][0]].  Returns ORACLE_BAD_BLOCK (copying
 * nothing) if an id is out of range.
 */
int pkv_oracle_copy_blocks(const uint8_t* src_k, const uint8_t* src_v, const float* src_ks,
                           const float* src_vs, int32_t src_nb, uint8_t* dst_k, uint8_t* dst_v,
                           float* dst_ks, float* dst_vs, int32_t dst_nb, const int32_t* pairs,
                           int32_t count, int64_t block_bytes, int32_t scales_per_block) {
  for (int32_t i = 0; i < count; ++i)
    if (pairs[2 * i] < 0 || pairs[2 * i] >= src_nb || pairs[2 * i + 1] < 0 || pairs[2 * i + 1] >= dst_nb)
      return ORACLE_BAD_BLOCK;
  for (int32_t i = 0; i < count; ++i) {
    const int64_t s = pairs[2 * i], d = pairs[2 * i + 1];
    memcpy(dst_k + d * block_bytes, src_k + s * block_bytes, (size_t)block_bytes);
    memcpy(dst_v + d * block_bytes, src_v + s * block_bytes, (size_t)block_bytes);
    if (src_ks != NULL) {
      memcpy(dst_ks + d * scales_per_block, src_ks + s * scales_per_block, sizeof(float) * (size_t)scales_per_block);
      memcpy(dst_vs + d * scales_per_block, src_vs + s * scales_per_block, sizeof(float) * (size_t)scales_per_block);
    }
  }
  return ORACLE_OK;
}

/* Number of threads the OpenMP runtime would use (1 without OpenMP). */
int pkv_oracle_num_threads(void) {
#ifdef _OPENMP
  int n = 1;
#pragma omp parallel
  {
#pragma omp single
    n = omp_get_num_threads();
  }
  return n;
#else
  return 1;
#endif
}
