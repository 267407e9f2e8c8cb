/*
 * pa_oracle.c — plain fp64 CPU oracle for paged attention in a
 * speculative-decoding verify step.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the correctness reference that the
 * CUDA path is checked against.  Only the test suite, the package smoke test
 * and the benchmark's CPU-baseline leg may load it.  The product library never
 * links, loads or calls it, and it shares no code, header, table or helper
 * with the CUDA path: the storage layouts below are restated here from their
 * definitions, not included.
 *
 * What it computes (the plain definition; the method reaches exactly this
 * result up to rounding order):
 *
 *   For every sequence b, every new token i < T_b and every query head h
 *   (any T_b: a verify step brings a few tokens, a prefill chunk many)
 *     p   = past_len_b + i                       absolute position of token i
 *     g   = h / (Hq / Hkv)                       KV head shared by the GQA group
 *     lo  = W > 0 ? max(0, p - W + 1) : 0         first visible key
 *     for j in [lo, p]:  K_j, V_j = stored key / value of position j, read
 *                         through the block table page bt[b][j / ps], slot j % ps
 *     s_j = scale * sum_d q[t, h, d] * K_j[d]
 *     out[t, h, :] = sum_j exp(s_j - max s) V_j / sum_j exp(s_j - max s)
 *   with t = subsequence_begins[b] + i.
 *
 *   Tree-mask verify (pa_oracle_forward_tree): the draft tokens form a tree
 *   (DDTree; OpenVINO issue 34644, cited by the OpenVINO issue 38153 page):
 *   token i sees every past key j < past_len_b inside its window as above, and
 *   the new token k (key past_len_b + k) only if bit k of tree_mask[t] is set.
 *   The causal chain (bits 0..i) gives back the definition above exactly.
 *
 * Sources (web pages on paged attention for speculative verification):
 *  - OpenVINO issue 38153, "Performance issue description" and "Cause":
 *    a verify step sends k+1 query tokens of one sequence against a long
 *    past_len; the suggested single-token handling gives query token i the key
 *    limit past_len + i + 1 (i.e. keys 0 .. past_len + i), and GQA heads share
 *    one KV head ("GQA read-once").
 *  - OpenVINO issue 38153, "Step-by-step reproduction", step 3: the operation's
 *    inputs are past_lens, subsequence_begins, max_context_len and a block
 *    table; u8 KV cache precision (step 1).
 *  - SGLang discussion 36314, "Observation 3", and the dual-radeon-vllm
 *    article's per-call section: sliding-window layers attend only the last
 *    window of keys (window 1024 on those pages).
 *
 * Readings where the pages are silent (each restated in the design notes):
 *  - GQA groups are contiguous: query head h uses KV head h / G, G = Hq / Hkv.
 *  - A window W admits exactly W keys ending at the token itself (j > p - W).
 *    W = 0 means no window.
 *  - The new tokens' own K/V already sit in the cache at positions
 *    past_len .. past_len + T - 1.
 *  - u8 dequantisation is (u8 - zp) * scale with fp16 scale and zero-point,
 *    one pair per token per KV head, separately for K and for V.
 *  - scale multiplies q.k before the softmax; no soft-cap, no bias.
 *
 * Storage layouts read here (restated, not shared):
 *  - q   [total_tokens, Hq, D] in q_dtype (0 f32, 1 f16, 2 bf16).
 *  - float KV cache  [num_blocks, Hkv, ps, D] in kv_dtype (0, 1 or 2).
 *  - u8 KV cache (kv_dtype 3): per (block, KV head) one record of
 *    ps*D bytes of codes, then ps fp16 scales, then ps fp16 zero-points;
 *    records are ps*(D+4) bytes, [num_blocks, Hkv, record].  K records hold
 *    their codes slot-major (code of slot j, element d at j*D + d), V
 *    records dim-major (at d*ps + j).
 *  - block_tables [num_seqs, max_blocks_per_seq] int32 physical block ids.
 *
 * Every stored value is converted exactly to double; all arithmetic is fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2, OR_U8 = 3 };

/* IEEE binary16 -> double, exact (normals, subnormals, inf, nan). */
static double half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int expo = (h >> 10) & 0x1f;
  int mant = h & 0x3ff;
  double v;
  if (expo == 0) {
    v = ldexp((double)mant, -24); /* subnormal: mant * 2^-14 * 2^-10 */
  } else if (expo == 31) {
    v = mant ? NAN : INFINITY;
  } else {
    v = ldexp((double)(mant | 0x400), expo - 25); /* (1.mant) * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* bfloat16 -> double, exact: the top 16 bits of an IEEE binary32. */
static double bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static double load_float(const void* base, int dtype, size_t idx) {
  if (dtype == OR_F32) {
    float f;
    memcpy(&f, (const char*)base + idx * 4, 4);
    return (double)f;
  }
  uint16_t h;
  memcpy(&h, (const char*)base + idx * 2, 2);
  return dtype == OR_F16 ? half_to_double(h) : bf16_to_double(h);
}

/* The dequantised value of element d of slot `slot` of KV head g in physical
 * block `blk` (OpenVINO issue 38153, reproduction step 1: u8 KV cache).
 * dim_major: the u8 record keeps its codes dim-major (the V cache). */
static double cache_value(const void* cache, int kv_dtype, int Hkv, int ps, int D,
                          int blk, int g, int slot, int d, int dim_major) {
  if (kv_dtype != OR_U8) {
    size_t idx = (((size_t)blk * Hkv + g) * ps + slot) * (size_t)D + d;
    return load_float(cache, kv_dtype, idx);
  }
  size_t rec_bytes = (size_t)ps * (D + 4);
  const unsigned char* rec = (const unsigned char*)cache + ((size_t)blk * Hkv + g) * rec_bytes;
  double code = (double)rec[dim_major ? (size_t)d * ps + slot : (size_t)slot * D + d];
  uint16_t s16, z16;
  memcpy(&s16, rec + (size_t)ps * D + 2 * (size_t)slot, 2);
  memcpy(&z16, rec + (size_t)ps * D + 2 * (size_t)ps + 2 * (size_t)slot, 2);
  return (code - half_to_double(z16)) * half_to_double(s16);
}

/*
 * pa_oracle_forward: the definition above, one output row at a time.
 * Returns 0, or -1 on inconsistent inputs (a block id outside
 * [0, num_blocks), a key position beyond the block table, bad begins).
 * out is [total_tokens, Hq, D] doubles.  nthreads <= 0 uses the OpenMP default.
 */
int pa_oracle_forward_tree(const void* q, int q_dtype, const void* k_cache, const void* v_cache,
                           int kv_dtype, const int32_t* block_tables, const int32_t* past_lens,
                           const int32_t* subsequence_begins, int num_seqs, int num_q_heads,
                           int num_kv_heads, int head_dim, int page_size, int num_blocks,
                           int max_blocks_per_seq, double scale, int sliding_window,
                           const uint8_t* tree_mask, double* out, int nthreads) {
  const int Hq = num_q_heads, Hkv = num_kv_heads, D = head_dim, ps = page_size;
  if (Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || ps <= 0 || num_seqs < 0) return -1;
  const int G = Hq / Hkv;
  const int total_tokens = subsequence_begins[num_seqs];

  /* Flatten (token, head) so each output row is one independent work item. */
  int* row_seq = (int*)malloc(sizeof(int) * (size_t)(total_tokens > 0 ? total_tokens : 1));
  if (!row_seq) return -1;
  for (int b = 0; b < num_seqs; ++b) {
    if (subsequence_begins[b] > subsequence_begins[b + 1] || past_lens[b] < 0 ||
        (tree_mask && subsequence_begins[b + 1] - subsequence_begins[b] > 8)) {
      free(row_seq);
      return -1;
    }
    for (int t = subsequence_begins[b]; t < subsequence_begins[b + 1]; ++t) row_seq[t] = b;
  }

  int bad = 0;
  const long n_items = (long)total_tokens * Hq;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
#endif
  for (long item = 0; item < n_items; ++item) {
    const int t = (int)(item / Hq), h = (int)(item % Hq);
    const int b = row_seq[t];
    const int i = t - subsequence_begins[b];
    const int T = subsequence_begins[b + 1] - subsequence_begins[b];
    const int g = h / G;
    const long L = past_lens[b];
    const long p = L + i;
    const long lo = sliding_window > 0 ? (p - sliding_window + 1 > 0 ? p - sliding_window + 1 : 0) : 0;
    /* with a tree mask, the new tokens this one attends are the bits of its mask */
    const unsigned m = tree_mask ? (unsigned)tree_mask[t] : 0u;
    const long last = L + T - 1; /* the last key any row of the sequence may see */
    double* o = out + ((size_t)t * Hq + h) * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (last / ps >= max_blocks_per_seq) {
      bad = 1;
      continue;
    }
    const long n = last - lo + 1;
    double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    if (!s) {
      bad = 1;
      continue;
    }
    /* scores s_j = scale * q . K_j over the visible keys: j >= lo, and
       without a tree mask j <= p (the causal rule, for any number of new
       tokens); with one, either a past key (j < L) or a new token whose bit
       is set */
    const size_t qoff = ((size_t)t * Hq + h) * D;
    double smax = -INFINITY;
    int row_bad = 0, seen = 0;
    for (long j = lo; j <= last; ++j) {
      const int vis = tree_mask ? (j < L || ((m >> (j - L)) & 1u)) : (j <= p);
      if (!vis) {
        s[j - lo] = -INFINITY;
        continue;
      }
      const int blk = block_tables[(size_t)b * max_blocks_per_seq + j / ps];
      if (blk < 0 || blk >= num_blocks) {
        row_bad = 1;
        break;
      }
      double acc = 0.0;
      for (int d = 0; d < D; ++d)
        acc += load_float(q, q_dtype, qoff + d) *
               cache_value(k_cache, kv_dtype, Hkv, ps, D, blk, g, (int)(j % ps), d, 0);
      s[j - lo] = scale * acc;
      if (s[j - lo] > smax) smax = s[j - lo];
      seen = 1;
    }
    if (row_bad) {
      free(s);
      bad = 1;
      continue;
    }
    if (seen) {
      /* softmax weights and the weighted sum of V */
      double denom = 0.0;
      for (long j = lo; j <= last; ++j) {
        if (s[j - lo] == -INFINITY) continue;
        const double w = exp(s[j - lo] - smax);
        denom += w;
        const int blk = block_tables[(size_t)b * max_blocks_per_seq + j / ps];
        for (int d = 0; d < D; ++d)
          o[d] += w * cache_value(v_cache, kv_dtype, Hkv, ps, D, blk, g, (int)(j % ps), d, 1);
      }
      for (int d = 0; d < D; ++d) o[d] /= denom;
    }
    free(s);
  }
  free(row_seq);
  return bad ? -1 : 0;
}

int pa_oracle_forward(const void* q, int q_dtype, const void* k_cache, const void* v_cache,
                      int kv_dtype, const int32_t* block_tables, const int32_t* past_lens,
                      const int32_t* subsequence_begins, int num_seqs, int num_q_heads,
                      int num_kv_heads, int head_dim, int page_size, int num_blocks,
                      int max_blocks_per_seq, double scale, int sliding_window, double* out,
                      int nthreads) {
  return pa_oracle_forward_tree(q, q_dtype, k_cache, v_cache, kv_dtype, block_tables, past_lens,
                                subsequence_begins, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                page_size, num_blocks, max_blocks_per_seq, scale, sliding_window, NULL,
                                out, nthreads);
}

/*
 * pa_oracle_pages_touched: which logical pages of each sequence the definition
 * reads, and through which physical block.  For sequence b with T_b >= 1 the
 * rows' key ranges [lo_i, past_len + i] have the union
 * [lo_0, past_len + T_b - 1]; every logical page overlapping it is read.
 * expected[b * max_blocks_per_seq + lp] = block_tables[b][lp] + 1 for a read
 * page, 0 otherwise (0 marks "not read", so block id 0 stays distinguishable).
 * Returns 0, or -1 if a range runs past the block table.
 */
int pa_oracle_pages_touched(const int32_t* block_tables, const int32_t* past_lens,
                            const int32_t* subsequence_begins, int num_seqs, int page_size,
                            int max_blocks_per_seq, int sliding_window, int32_t* expected) {
  memset(expected, 0, sizeof(int32_t) * (size_t)num_seqs * max_blocks_per_seq);
  for (int b = 0; b < num_seqs; ++b) {
    const int T = subsequence_begins[b + 1] - subsequence_begins[b];
    if (T <= 0) continue;
    const long L = past_lens[b];
    const long hi = L + T - 1;
    const long lo = sliding_window > 0 ? (L - sliding_window + 1 > 0 ? L - sliding_window + 1 : 0) : 0;
    if (hi / page_size >= max_blocks_per_seq) return -1;
    for (long lp = lo / page_size; lp <= hi / page_size; ++lp)
      expected[(size_t)b * max_blocks_per_seq + lp] = block_tables[(size_t)b * max_blocks_per_seq + lp] + 1;
  }
  return 0;
}

/* ---------------------------------------------------------------------------
 * The cache update: the step just before the verify (the OpenVINO
 * paged-attention op writes the new tokens' K/V into the cache itself, issue
 * 38153 "Step-by-step reproduction" step 3; u8 KV cache precision, step 1).
 *
 * Token i of sequence b goes to position p = past_len_b + i: page
 * block_tables[b][p / ps], slot p % ps, for every KV head, K and V alike.
 *  - float caches: the value rounded to nearest-even in the cache dtype;
 *  - u8 caches, per token and KV head over its D values x (binary32, every
 *    operation rounded to nearest-even):
 *        mn = min x, mx = max x
 *        scale = fp16(  (mx - mn) / 255  )        1.0 if that is 0 or not finite
 *        zp    = fp16(  (0 - mn) / scale  )       (any fp16 value)
 *        code  = clamp(rint(  x / scale + zp  ), 0, 255)
 *    and the value is read back as (code - zp) * scale.
 * Only the written slots change.
 * ------------------------------------------------------------------------- */

/* binary32 -> binary16 bits, round to nearest-even (overflow to inf). */
static uint16_t float_to_half_rn(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  const uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
  const uint32_t expo = (u >> 23) & 0xffu;
  uint32_t mant = u & 0x7fffffu;
  if (expo == 0xffu) return (uint16_t)(sign | 0x7c00u | (mant ? 0x200u : 0u));
  /* the value is (1.mant) * 2^(expo-127); binary16 keeps 10 fraction bits */
  const int e = (int)expo - 127;
  if (e > 15) return (uint16_t)(sign | 0x7c00u);
  if (e >= -14) {
    /* normal: drop 13 bits with round-to-nearest-even */
    uint32_t m = mant >> 13, rest = mant & 0x1fffu;
    uint32_t h = ((uint32_t)(e + 15) << 10) | m;
    if (rest > 0x1000u || (rest == 0x1000u && (m & 1u))) ++h; /* may carry into the exponent: still correct */
    return (uint16_t)(sign | h);
  }
  /* subnormal (or zero): value = m * 2^-24 with m = (1.mant) * 2^(e+24) */
  if (e < -25) return sign;
  if (expo == 0) return sign; /* binary32 subnormals are far below 2^-25 */
  mant |= 0x800000u;                        /* 24-bit significand, value = mant * 2^(e-23) */
  const int shift = -e - 1;                 /* mant * 2^(e-23) / 2^-24 = mant >> (-1 - e) */
  uint32_t m = mant >> shift;
  uint32_t rest = mant & ((1u << shift) - 1u), half = 1u << (shift - 1);
  if (rest > half || (rest == half && (m & 1u))) ++m;
  return (uint16_t)(sign | m);
}

/* binary32 -> bfloat16 bits, round to nearest-even (NaN kept quiet). */
static uint16_t float_to_bf16_rn(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x7fffffu)) return (uint16_t)((u >> 16) | 0x40u);
  const uint32_t rest = u & 0xffffu, keep = u >> 16;
  uint32_t r = keep;
  if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) ++r;
  return (uint16_t)r;
}

static float load_src(const void* base, int dtype, size_t idx) {
  return (float)load_float(base, dtype, idx); /* f32 / f16 / bf16 values are binary32-exact */
}

static void store_float(void* base, int dtype, size_t idx, float v) {
  if (dtype == OR_F32) {
    memcpy((char*)base + idx * 4, &v, 4);
  } else {
    const uint16_t h = dtype == OR_F16 ? float_to_half_rn(v) : float_to_bf16_rn(v);
    memcpy((char*)base + idx * 2, &h, 2);
  }
}

/* One token's D values of one KV head into slot `slot` of record `rec`
 * (codes slot-major, or dim-major for the V cache). */
static void quantize_u8_slot(const float* x, int D, int ps, int slot, unsigned char* rec, int dim_major) {
  float mn = x[0], mx = x[0];
  for (int d = 1; d < D; ++d) {
    if (x[d] < mn) mn = x[d];
    if (x[d] > mx) mx = x[d];
  }
  const float range = mx - mn;
  const float s32 = range / 255.0f;
  uint16_t s16 = float_to_half_rn(s32);
  float sf = (float)half_to_double(s16);
  if (!(sf > 0.0f) || isinf(sf)) {
    s16 = 0x3c00u; /* 1.0 */
    sf = 1.0f;
  }
  const float zq = (0.0f - mn) / sf; /* 0 - mn: a -0 minimum gives +0, whatever order found it */
  const uint16_t z16 = float_to_half_rn(zq);
  const float zf = (float)half_to_double(z16);
  for (int d = 0; d < D; ++d) {
    const float t = x[d] / sf;
    const float u = t + zf;
    float c = rintf(u);
    if (!(c >= 0.0f)) c = 0.0f; /* also NaN */
    if (c > 255.0f) c = 255.0f;
    rec[dim_major ? (size_t)d * ps + slot : (size_t)slot * D + d] = (unsigned char)c;
  }
  memcpy(rec + (size_t)ps * D + 2 * (size_t)slot, &s16, 2);
  memcpy(rec + (size_t)ps * D + 2 * (size_t)ps + 2 * (size_t)slot, &z16, 2);
}

/*
 * pa_oracle_cache_update: the definition above.  k_new / v_new are
 * [total_tokens, Hkv, D] in src_dtype (0 f32, 1 f16, 2 bf16); the caches use
 * the layouts of pa_oracle_forward.  Returns 0, or -1 on inconsistent inputs
 * (bad begins, a position beyond the block table, a block id outside
 * [0, num_blocks)); nothing is written then.
 */
int pa_oracle_cache_update(const void* k_new, const void* v_new, int src_dtype, void* k_cache, void* v_cache,
                           int kv_dtype, const int32_t* block_tables, const int32_t* past_lens,
                           const int32_t* subsequence_begins, int num_seqs, int Hkv, int D, int ps,
                           int num_blocks, int max_blocks_per_seq) {
  /* validate everything first so that a rejected call writes nothing */
  for (int b = 0; b < num_seqs; ++b) {
    const int t0 = subsequence_begins[b], t1 = subsequence_begins[b + 1];
    if (t0 < 0 || t1 < t0 || past_lens[b] < 0) return -1;
    for (int i = 0; i < t1 - t0; ++i) {
      const long p = (long)past_lens[b] + i;
      if (p / ps >= max_blocks_per_seq) return -1;
      const int blk = block_tables[(size_t)b * max_blocks_per_seq + p / ps];
      if (blk < 0 || blk >= num_blocks) return -1;
    }
  }
  float* x = (float*)malloc(sizeof(float) * (size_t)D);
  if (!x) return -1;
  for (int b = 0; b < num_seqs; ++b) {
    const int t0 = subsequence_begins[b], t1 = subsequence_begins[b + 1];
    for (int i = 0; i < t1 - t0; ++i) {
      const long p = (long)past_lens[b] + i;
      const int blk = block_tables[(size_t)b * max_blocks_per_seq + p / ps];
      const int slot = (int)(p % ps);
      const size_t t = (size_t)(t0 + i);
      for (int g = 0; g < Hkv; ++g) {
        for (int which = 0; which < 2; ++which) {
          const void* src = which ? v_new : k_new;
          void* cache = which ? v_cache : k_cache;
          const size_t sbase = (t * Hkv + g) * (size_t)D;
          if (kv_dtype != OR_U8) {
            const size_t cbase = (((size_t)blk * Hkv + g) * ps + slot) * (size_t)D;
            for (int d = 0; d < D; ++d) store_float(cache, kv_dtype, cbase + d, load_src(src, src_dtype, sbase + d));
          } else {
            for (int d = 0; d < D; ++d) x[d] = load_src(src, src_dtype, sbase + d);
            unsigned char* rec = (unsigned char*)cache + ((size_t)blk * Hkv + g) * (size_t)ps * (D + 4);
            quantize_u8_slot(x, D, ps, slot, rec, which);
          }
        }
      }
    }
  }
  free(x);
  return 0;
}

int pa_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
