/*
 * oracle.c — plain, slow, double-precision CPU reference for paged GQA decode
 * attention.  TEST INFRASTRUCTURE ONLY: it exists to check the CUDA library,
 * is called by the tests, by the smoke check and by the benchmark's CPU
 * baseline, and is never linked into or called by the library itself.  It
 * shares no code, header or table with the CUDA path.
 *
 * Every function states the passage it follows.  Page titles used below:
 *   [P2] 大模型推理加速核心KV Cache 复用机制与内存布局优化 (mlqm.cn)
 *   [P3] LLM推理优化实战：从KV-Cache到Continuous Batching的技术演进与代码实现 (tbr8.org)
 *   [P4] 大模型推理加速——KV Cache篇 (AiGC面试宝典)
 *   [P5] 苦猿的大模型日记 · Day45 · 大模型推理加速 (devpress.csdn.net)
 *
 * Number formats are decoded from their public definitions (IEEE 754
 * binary16, bfloat16 = the top half of binary32, OCP 8-bit floating point
 * E4M3 "fn" variant), not through any CUDA or compiler intrinsic.
 *
 * Build: cc -O2 -fopenmp -ffp-contract=off -shared -fPIC oracle.c -lm
 * (no -ffast-math: the fp32 division in the fp8 quantiser must be IEEE).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Element type codes of the oracle's own interface. */
enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2, OR_E4M3 = 3 };

/* ---------------------------------------------------------------------- */
/* Number formats                                                          */
/* ---------------------------------------------------------------------- */

/* IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double oracle_f16_to_double(uint16_t h) {
  int s = h >> 15, e = (h >> 10) & 0x1f, m = h & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)m / 1024.0, -14);
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp(1.0 + (double)m / 1024.0, e - 15);
  return s ? -v : v;
}

/* bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits. */
double oracle_bf16_to_double(uint16_t h) {
  int s = h >> 15, e = (h >> 7) & 0xff, m = h & 0x7f;
  double v;
  if (e == 0)
    v = ldexp((double)m / 128.0, -126);
  else if (e == 255)
    v = m ? NAN : INFINITY;
  else
    v = ldexp(1.0 + (double)m / 128.0, e - 127);
  return s ? -v : v;
}

/* OCP FP8 E4M3 ("fn"): 1 sign, 4 exponent (bias 7), 3 fraction bits; no
 * infinities; S.1111.111 is NaN; exponent field 0 is subnormal 2^-6 * 0.m.
 * Largest finite magnitude 1.75 * 2^8 = 448.  The FP8 KV cache is named in
 * [P2] §四 (FP8/E4M3 KV Cache) and [P5] PART 02 (FP8 KV Cache). */
double oracle_e4m3_to_double(uint8_t byte) {
  int s = byte >> 7, e = (byte >> 3) & 0xf, m = byte & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

/* Nearest E4M3 code to x, ties to the even code (fraction LSB 0), magnitudes
 * beyond 448 saturating to 448, NaN -> 0x7f.  Brute force over the 127
 * non-negative finite codes, which are increasing in value. */
uint8_t oracle_e4m3_from_float(float x) {
  if (isnan(x)) return 0x7f;
  int neg = signbit(x) ? 1 : 0;
  double a = fabs((double)x);
  int best = 0;
  double bestd = INFINITY;
  for (int code = 0; code <= 126; ++code) {
    double d = fabs(oracle_e4m3_to_double((uint8_t)code) - a);
    if (d < bestd || (d == bestd && (code & 1) == 0)) {
      bestd = d;
      best = code;
    }
  }
  return (uint8_t)((neg << 7) | best);
}

static double load_elem(const void *base, int dtype, size_t i) {
  switch (dtype) {
    case OR_F32: {
      float f;
      memcpy(&f, (const char *)base + 4 * i, 4);
      return (double)f;
    }
    case OR_F16: {
      uint16_t h;
      memcpy(&h, (const char *)base + 2 * i, 2);
      return oracle_f16_to_double(h);
    }
    case OR_BF16: {
      uint16_t h;
      memcpy(&h, (const char *)base + 2 * i, 2);
      return oracle_bf16_to_double(h);
    }
    case OR_E4M3:
      return oracle_e4m3_to_double(((const uint8_t *)base)[i]);
  }
  return NAN;
}

static size_t elem_size(int dtype) {
  return dtype == OR_F32 ? 4 : (dtype == OR_E4M3 ? 1 : 2);
}

/* Exact fp32 value of a 16/32-bit element (all of them are representable). */
static float load_as_float(const void *base, int dtype, size_t i) {
  return (float)load_elem(base, dtype, i);
}

/* ---------------------------------------------------------------------- */
/* KV bytes per token: 2 * num_layers * num_kv_heads * head_dim * bytes     */
/* ([P5] PART 02, "一行公式，算出单个 token 吃多少显存").                        */
/* ---------------------------------------------------------------------- */
double oracle_kv_bytes_per_token(int num_layers, int num_kv_heads, int head_dim,
                                 double dtype_bytes) {
  return 2.0 * num_layers * num_kv_heads * head_dim * dtype_bytes;
}

/* ---------------------------------------------------------------------- */
/* Append: write the new token's K and V into its slot.                     */
/* [P4] §3.1 (Attention.forward step 2: cache_k[:, start_pos] = xk),          */
/* [P5] PART 02 (new_k appended to k_cache), [P3] §2.2 (logical block =       */
/* num_tokens // BLOCK_SIZE).  Cache layout [num_blocks][Hkv][bs][D].          */
/* FP8: q8 = e4m3_rne_sat((float)x / scale) with an fp32 division; a token    */
/* at offset 0 of its block opens the block and sets scale = amax/448 (1 if   */
/* amax is 0).  Returns 0, or -1 for an unsupported dtype pair.               */
/* ---------------------------------------------------------------------- */
static void append_one(const void *src, int new_dtype, size_t src_off,
                       void *cache, int cache_dtype, float *scales,
                       size_t tile_elem, size_t scale_idx, int off, int D) {
  if (cache_dtype == OR_E4M3) {
    float sc;
    if (off == 0) {
      float amax = 0.0f;
      for (int d = 0; d < D; ++d) {
        float a = fabsf(load_as_float(src, new_dtype, src_off + d));
        if (a > amax) amax = a;
      }
      sc = amax > 0.0f ? amax / 448.0f : 1.0f;
      scales[scale_idx] = sc;
    } else {
      sc = scales[scale_idx];
    }
    for (int d = 0; d < D; ++d) {
      float x = load_as_float(src, new_dtype, src_off + d);
      float r = x / sc;
      ((uint8_t *)cache)[tile_elem + d] = oracle_e4m3_from_float(r);
    }
  } else {
    size_t es = elem_size(cache_dtype);
    memcpy((char *)cache + es * tile_elem, (const char *)src + es * src_off, es * D);
  }
}

int oracle_append(void *k_cache, void *v_cache, int cache_dtype, float *k_scale,
                  float *v_scale, const void *k_new, const void *v_new, int new_dtype,
                  const int64_t *slot_mapping, int B, int Hkv, int D,
                  int64_t num_blocks, int block_size) {
  if (cache_dtype != OR_E4M3 && new_dtype != cache_dtype) return -1;
  if (cache_dtype == OR_E4M3 && new_dtype == OR_E4M3) return -1;
  for (int b = 0; b < B; ++b) {
    int64_t slot = slot_mapping[b];
    if (slot < 0) continue;
    int64_t blk = slot / block_size;
    int off = (int)(slot % block_size);
    if (blk >= num_blocks) continue;
    for (int h = 0; h < Hkv; ++h) {
      size_t tile = ((size_t)(blk * Hkv + h) * block_size + off) * D;
      size_t src = ((size_t)b * Hkv + h) * D;
      size_t sidx = (size_t)blk * Hkv + h;
      append_one(k_new, new_dtype, src, k_cache, cache_dtype, k_scale, tile, sidx, off, D);
      append_one(v_new, new_dtype, src, v_cache, cache_dtype, v_scale, tile, sidx, off, D);
    }
  }
  return 0;
}

/* ---------------------------------------------------------------------- */
/* Calibrated FP8 append.  [P2] §四 and [P5] PART 02 (first advanced          */
/* direction) warn that an FP8 cache's quality depends on how its scales are  */
/* calibrated.  Here a block's scale follows the running maximum of its       */
/* tokens and is a power of two: cand(x) = the smallest 2^k with              */
/* max|x| <= 448 * 2^k (1 if x is all zero).  A token at offset 0 sets        */
/* scale = cand; a later token with cand > scale first raises the scale to    */
/* cand and re-quantises the block's earlier tokens,                          */
/*   q' = e4m3_rne_sat( fp32( decode(q) * scale_old ) / scale_new ),           */
/* then every token is stored as e4m3_rne_sat(x / scale) (fp32 ops).  No      */
/* stored value saturates, and since scales are powers of two the            */
/* re-quantisation only shifts exponents: exact for values that stay in the   */
/* e4m3 normal range.  Tokens are applied in order b = 0 .. B-1.  Other       */
/* cache types: the plain append.                                             */
/* ---------------------------------------------------------------------- */
static float pow2_scale(float amax) {
  if (!(amax > 0.0f)) return 1.0f;
  int e;
  float m = frexpf(amax, &e); /* amax = m * 2^e, 0.5 <= m < 1 */
  /* amax <= 448 * 2^k = 0.875 * 2^(9 + k) */
  int k = (m <= 0.875f) ? e - 9 : e - 8;
  return ldexpf(1.0f, k);
}

static void append_one_calibrated(const void *src, int new_dtype, size_t src_off,
                                  uint8_t *cache, float *scales, size_t tile_elem,
                                  size_t scale_idx, int off, int D) {
  float amax = 0.0f;
  for (int d = 0; d < D; ++d) {
    float a = fabsf(load_as_float(src, new_dtype, src_off + d));
    if (a > amax) amax = a;
  }
  float cand = pow2_scale(amax);
  float sc;
  if (off == 0) {
    sc = cand;
  } else {
    sc = scales[scale_idx];
    if (cand > sc) {
      /* earlier tokens of the block: rows off-1 .. 0 of the same tile */
      for (int t = 0; t < off; ++t) {
        uint8_t *row = cache + tile_elem - (size_t)(off - t) * D;
        for (int d = 0; d < D; ++d) {
          float v = (float)oracle_e4m3_to_double(row[d]);
          float y = v * sc;
          float r = y / cand;
          row[d] = oracle_e4m3_from_float(r);
        }
      }
      sc = cand;
    }
  }
  scales[scale_idx] = sc;
  for (int d = 0; d < D; ++d) {
    float x = load_as_float(src, new_dtype, src_off + d);
    float r = x / sc;
    cache[tile_elem + d] = oracle_e4m3_from_float(r);
  }
}

int oracle_append_calibrated(void *k_cache, void *v_cache, int cache_dtype, float *k_scale,
                             float *v_scale, const void *k_new, const void *v_new, int new_dtype,
                             const int64_t *slot_mapping, int B, int Hkv, int D,
                             int64_t num_blocks, int block_size) {
  if (cache_dtype != OR_E4M3)
    return oracle_append(k_cache, v_cache, cache_dtype, k_scale, v_scale, k_new, v_new, new_dtype,
                         slot_mapping, B, Hkv, D, num_blocks, block_size);
  if (new_dtype == OR_E4M3) return -1;
  for (int b = 0; b < B; ++b) {
    int64_t slot = slot_mapping[b];
    if (slot < 0) continue;
    int64_t blk = slot / block_size;
    int off = (int)(slot % block_size);
    if (blk >= num_blocks) continue;
    for (int h = 0; h < Hkv; ++h) {
      size_t tile = ((size_t)(blk * Hkv + h) * block_size + off) * D;
      size_t src = ((size_t)b * Hkv + h) * D;
      size_t sidx = (size_t)blk * Hkv + h;
      append_one_calibrated(k_new, new_dtype, src, (uint8_t *)k_cache, k_scale, tile, sidx, off, D);
      append_one_calibrated(v_new, new_dtype, src, (uint8_t *)v_cache, v_scale, tile, sidx, off, D);
    }
  }
  return 0;
}

/* ---------------------------------------------------------------------- */
/* Decode attention over the paged cache.                                   */
/* out[b,hq,:] = sum_t softmax_t(scale * q.K_t) V_t  ([P5] PART 02 formula     */
/* Attention = softmax(QK^T/sqrt(d))V; [P3] §1.1 attention_step; [P4] §3.1     */
/* scores = xq.keys^T / sqrt(d), softmax, .values).  For a single new query    */
/* the causal mask of [P4] §2.1 admits every cached position, so it is empty. */
/* K_t is gathered through the block table ([P3] §2.2; [P2] §三):              */
/*   K_t = k_cache[block_table[b][t / bs]][h][t % bs][:],  h = hq / (Hq/Hkv)  */
/* ([P4] §6.2 GQA: a group of query heads shares one K/V head).               */
/* FP8 elements are decode(byte) * scale[block][h].  Positions t run over     */
/* [t_begin[b], context_lens[b]) (t_begin NULL means 0), which lets tests      */
/* build partial results over a sub-range.  lse_out (may be NULL) receives     */
/* log(sum_t exp(s_t)) = m + log(l); a row with no positions gives out = 0    */
/* and lse = -inf.                                                              */
/*                                                                          */
/* Several new queries per sequence (q_len > 1, the verify step of           */
/* speculative decoding, [P3] §4): the q_len newest positions are the new     */
/* tokens, and new token i (0-based) sees positions up to its own, i.e. the   */
/* first ctx - (q_len - 1 - i) of them — the causal mask                      */
/* tril(diagonal = kv_len - q_len) of [P5] PART 04 naive_attention.           */
/* q and out are then [B][q_len][Hq][D], lse [B][q_len][Hq].                  */
/*                                                                          */
/* Sliding window (window W > 0; 0 means none): a row sees only the W most    */
/* recent positions up to its own, [lim - W, lim) with lim its causal limit   */
/* above — the fixed-size visible history of [P5] PART 02 (third advanced     */
/* direction, sliding window / KV eviction).  Positions no row can see are    */
/* not gathered at all, so their blocks may have been released.              */
/*                                                                          */
/* Prefill (q_start != NULL): sequence b has its own number of new tokens,    */
/* n_b = q_start[b+1] - q_start[b], packed in q / out from row q_start[b]     */
/* ([total][Hq][D]); they are the n_b newest of its ctx_b positions and       */
/* attend causally as above — the masked attention of a prompt over itself    */
/* and any cached prefix ([P3] §3.2 flash_attention over Q, K, V blocks;      */
/* [P5] PART 04 causal naive_attention).                                     */
/* ---------------------------------------------------------------------- */
static int decode_impl(double *out, double *lse_out, const void *q, int q_dtype,
                       const void *k_cache, const void *v_cache, int cache_dtype,
                       const float *k_scale, const float *v_scale,
                       const int32_t *block_table, int max_blocks,
                       const int32_t *context_lens, const int32_t *t_begin,
                       const int32_t *q_start,
                       int B, int q_len, int window, int Hq, int Hkv, int D, int64_t num_blocks,
                       int block_size, double scale, int nthreads) {
  if (Hkv <= 0 || Hq % Hkv != 0 || (!q_start && q_len <= 0) || window < 0) return -1;
  int G = Hq / Hkv;
  int err = 0;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int b = 0; b < B; ++b) {
    for (int h = 0; h < Hkv; ++h) {
      int t0 = t_begin ? t_begin[b] : 0;
      int t1 = context_lens[b];
      /* this sequence's new tokens and its first row in q / out */
      const int nl = q_start ? q_start[b + 1] - q_start[b] : q_len;
      const size_t row0 = q_start ? (size_t)q_start[b] : (size_t)b * q_len;
      /* the earliest position any row sees: row 0's window start */
      if (window > 0 && t1 - (nl - 1) - window > t0) t0 = t1 - (nl - 1) - window;
      int n = t1 > t0 ? t1 - t0 : 0;
      double *K = NULL, *V = NULL, *s = NULL, *qv = NULL;
      if (n > 0) {
        K = (double *)malloc(sizeof(double) * (size_t)n * D);
        V = (double *)malloc(sizeof(double) * (size_t)n * D);
        s = (double *)malloc(sizeof(double) * (size_t)n);
      }
      qv = (double *)malloc(sizeof(double) * D);
      /* gather this (sequence, kv head)'s K and V contiguously */
      for (int i = 0; i < n; ++i) {
        int t = t0 + i;
        int logical = t / block_size;
        int64_t blk = logical < max_blocks ? block_table[(size_t)b * max_blocks + logical] : -1;
        if (blk < 0 || blk >= num_blocks) {
#pragma omp atomic write
          err = -2;
          blk = 0;
        }
        size_t base = ((size_t)(blk * Hkv + h) * block_size + (t % block_size)) * D;
        double ks = 1.0, vs = 1.0;
        if (cache_dtype == OR_E4M3) {
          ks = k_scale[blk * Hkv + h];
          vs = v_scale[blk * Hkv + h];
        }
        for (int d = 0; d < D; ++d) {
          K[(size_t)i * D + d] = load_elem(k_cache, cache_dtype, base + d) * ks;
          V[(size_t)i * D + d] = load_elem(v_cache, cache_dtype, base + d) * vs;
        }
      }
      for (int qi = 0; qi < nl; ++qi) {
        /* new token qi sees gathered positions [lo, hi) */
        int hi = n - (nl - 1 - qi);
        if (hi < 0) hi = 0;
        int lo = (window > 0 && hi - window > 0) ? hi - window : 0;
        int nq = hi - lo;
        size_t row = row0 + qi;
        for (int g = 0; g < G; ++g) {
          int hq = h * G + g;
          double *o = out + (row * Hq + hq) * D;
          for (int d = 0; d < D; ++d) qv[d] = load_elem(q, q_dtype, (row * Hq + hq) * D + d);
          if (nq == 0) {
            for (int d = 0; d < D; ++d) o[d] = 0.0;
            if (lse_out) lse_out[row * Hq + hq] = -INFINITY;
            continue;
          }
          double m = -INFINITY;
          for (int i = lo; i < hi; ++i) {
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += qv[d] * K[(size_t)i * D + d];
            s[i] = scale * acc;
            if (s[i] > m) m = s[i];
          }
          double l = 0.0;
          for (int i = lo; i < hi; ++i) {
            s[i] = exp(s[i] - m);
            l += s[i];
          }
          for (int d = 0; d < D; ++d) {
            double acc = 0.0;
            for (int i = lo; i < hi; ++i) acc += s[i] * V[(size_t)i * D + d];
            o[d] = acc / l;
          }
          if (lse_out) lse_out[row * Hq + hq] = m + log(l);
        }
      }
      free(K);
      free(V);
      free(s);
      free(qv);
    }
  }
  return err;
}

int oracle_decode(double *out, double *lse_out, const void *q, int q_dtype,
                  const void *k_cache, const void *v_cache, int cache_dtype,
                  const float *k_scale, const float *v_scale,
                  const int32_t *block_table, int max_blocks,
                  const int32_t *context_lens, const int32_t *t_begin,
                  int B, int Hq, int Hkv, int D, int64_t num_blocks,
                  int block_size, double scale, int nthreads) {
  return decode_impl(out, lse_out, q, q_dtype, k_cache, v_cache, cache_dtype, k_scale, v_scale,
                     block_table, max_blocks, context_lens, t_begin, NULL, B, 1, 0, Hq, Hkv, D,
                     num_blocks, block_size, scale, nthreads);
}

int oracle_decode_multi(double *out, double *lse_out, const void *q, int q_dtype,
                        const void *k_cache, const void *v_cache, int cache_dtype,
                        const float *k_scale, const float *v_scale,
                        const int32_t *block_table, int max_blocks,
                        const int32_t *context_lens, const int32_t *t_begin,
                        int B, int q_len, int window, int Hq, int Hkv, int D, int64_t num_blocks,
                        int block_size, double scale, int nthreads) {
  return decode_impl(out, lse_out, q, q_dtype, k_cache, v_cache, cache_dtype, k_scale, v_scale,
                     block_table, max_blocks, context_lens, t_begin, NULL, B, q_len, window, Hq, Hkv, D,
                     num_blocks, block_size, scale, nthreads);
}

int oracle_prefill(double *out, double *lse_out, const void *q, int q_dtype,
                   const void *k_cache, const void *v_cache, int cache_dtype,
                   const float *k_scale, const float *v_scale,
                   const int32_t *block_table, int max_blocks,
                   const int32_t *context_lens, const int32_t *q_start,
                   int B, int window, int Hq, int Hkv, int D, int64_t num_blocks,
                   int block_size, double scale, int nthreads) {
  return decode_impl(out, lse_out, q, q_dtype, k_cache, v_cache, cache_dtype, k_scale, v_scale,
                     block_table, max_blocks, context_lens, NULL, q_start, B, 0, window, Hq, Hkv, D,
                     num_blocks, block_size, scale, nthreads);
}

/* ---------------------------------------------------------------------- */
/* Merge of partial results over disjoint position ranges.                  */
/* From the online-softmax rescaling of [P3] §3.2 (O and l rescaled by        */
/* exp(m_old - m_new) when the running max grows): with per-part lse_s and    */
/* normalised o_s, out = sum_s exp(lse_s - M) o_s / sum_s exp(lse_s - M),     */
/* M = max_s lse_s.  o_parts [R][S][D], lse_parts [R][S]; -inf = empty part.  */
/* ---------------------------------------------------------------------- */
void oracle_merge(double *out, const double *o_parts, const double *lse_parts,
                  int R, int S, int D) {
  for (int r = 0; r < R; ++r) {
    double M = -INFINITY;
    for (int s = 0; s < S; ++s)
      if (lse_parts[(size_t)r * S + s] > M) M = lse_parts[(size_t)r * S + s];
    double *o = out + (size_t)r * D;
    if (M == -INFINITY) {
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      continue;
    }
    double wsum = 0.0;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    for (int s = 0; s < S; ++s) {
      double lse = lse_parts[(size_t)r * S + s];
      if (lse == -INFINITY) continue;
      double w = exp(lse - M);
      wsum += w;
      for (int d = 0; d < D; ++d) o[d] += w * o_parts[((size_t)r * S + s) * D + d];
    }
    for (int d = 0; d < D; ++d) o[d] /= wsum;
  }
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
