/*
 * oracle.c -- plain, slow, fp64 CPU reference for the operations of a paged
 * KV cache decode step (and the chunked prefill that fills the cache):
 *
 *   1. the KV-cache append ("reshape and cache"): every new token's key and
 *      value vectors are copied, bit for bit, into the physical slot that the
 *      slot mapping names;
 *   2. paged decode attention: for every running sequence, one query token per
 *      query head attends over all of that sequence's cached tokens, which are
 *      found through the sequence's block table in a fixed pool of physical
 *      KV blocks.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it, to check and to time the CUDA path against it.
 * It shares no code, header or constant with the CUDA library.
 *
 * Sources (page title, then section):
 *   - "mini-vLLM" README, "How it works / Paged KV-cache": a fixed pool of
 *     physical blocks, each with block_size token slots, and a per-sequence
 *     block table from logical positions to physical storage.  Logical token
 *     j of a sequence lives in physical block table[j / block_size] at slot
 *     j % block_size.
 *   - "mini-vLLM" README, "Results / Correctness" table: paged attention
 *     (grouped-query heads included, non-power-of-two block tables included)
 *     equals dense attention over the same tokens scattered into blocks.
 *   - "mini-vLLM" README, "Results / End-to-end throughput vs baselines",
 *     paragraph on what changed: each query head reads its own KV head
 *     (grouped-query style) instead of expanding the pool, and the K/V write
 *     is one indexed assignment per layer.
 *   - "wLLM" project page, "Features / Core engine" and "CPU inference":
 *     block-based KV cache; the CPU path computes "the same math" as the
 *     CUDA kernel.
 *
 * Readings where the pages are silent (each is also listed in the design
 * notes of the repository):
 *   - cache layout [num_blocks][num_kv_heads][block_size][head_dim], the same
 *     for K and V, every dimension dense;
 *   - query head h reads KV head h / (num_q_heads / num_kv_heads);
 *   - a negative slot in the slot mapping means "no write" (padding);
 *   - context_lens[b] counts every token that sequence b attends to, the one
 *     appended in this step included; a length of 0 gives an all-zero output;
 *   - no mask, no ALiBi, no soft-capping, no sliding window;
 *   - scale is a binary32 value; it is widened to binary64 before use.
 *
 * Arithmetic: everything in binary64.  The softmax is the plain two-pass
 * definition: s_j = scale * <q, k_j>, m = max_j s_j, w_j = exp(s_j - m),
 * out = (sum_j w_j v_j) / (sum_j w_j), summed in logical token order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* element type codes used by the Python wrapper */
enum { ORACLE_F32 = 0, ORACLE_F16 = 1, ORACLE_BF16 = 2, ORACLE_E4M3 = 3 };

/* status codes */
enum {
  ORACLE_OK = 0,
  ORACLE_BAD_SHAPE = -1,
  ORACLE_BAD_DTYPE = -2,
  ORACLE_SLOT_OUT_OF_RANGE = -3,
  ORACLE_LEN_OUT_OF_RANGE = -4,
  ORACLE_BLOCK_OUT_OF_RANGE = -5,
  ORACLE_NO_MEMORY = -6
};

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -24); /* subnormal: f * 2^(1-15-10) */
  } else if (e == 31) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexp((double)(f + 1024), e - 25); /* (1 + f/2^10) * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE 754 binary32. */
static double bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* OCP FP8 E4M3 ("e4m3fn"): 1 sign bit, 4 exponent bits (bias 7), 3 fraction
 * bits; no infinities; exponent and fraction all ones is NaN; largest finite
 * magnitude 448. */
static double e4m3_to_double(uint8_t c) {
  int sign = (c >> 7) & 1;
  int e = (c >> 3) & 0xf;
  int f = c & 7;
  double v;
  if (e == 15 && f == 7) {
    v = NAN;
  } else if (e == 0) {
    v = ldexp((double)f, -9); /* subnormal: f * 2^(1-7-3) */
  } else {
    v = ldexp((double)(f + 8), e - 10); /* (1 + f/8) * 2^(e-7) */
  }
  return sign ? -v : v;
}

/* Round y to E4M3: the nearest finite code, ties to the code with an even
 * fraction; magnitudes beyond the largest finite value give +-448
 * (saturation); NaN gives NaN.  Written as a search over the 127 finite
 * non-negative codes, which is slow and plainly the definition. */
static uint8_t double_to_e4m3(double y) {
  if (isnan(y)) return 0x7f;
  const uint8_t sign = (y < 0 || (y == 0 && signbit(y))) ? 0x80 : 0;
  const double a = fabs(y);
  if (a >= 448.0) return (uint8_t)(sign | 0x7e);
  uint8_t best = 0;
  double best_d = INFINITY;
  for (int c = 0; c <= 0x7e; ++c) {
    const double d = fabs(e4m3_to_double((uint8_t)c) - a);
    if (d < best_d || (d == best_d && (c & 1) == 0)) {
      best_d = d;
      best = (uint8_t)c;
    }
  }
  return (uint8_t)(sign | best);
}

static double load_elt(const void* base, int64_t i, int dtype) {
  if (dtype == ORACLE_E4M3) return e4m3_to_double(((const uint8_t*)base)[i]);
  if (dtype == ORACLE_F32) {
    float f;
    memcpy(&f, (const char*)base + 4 * i, 4);
    return (double)f;
  }
  uint16_t h;
  memcpy(&h, (const char*)base + 2 * i, 2);
  return dtype == ORACLE_F16 ? half_to_double(h) : bf16_to_double(h);
}

static int elt_bytes(int dtype) {
  switch (dtype) {
    case ORACLE_E4M3: return 1;
    case ORACLE_F32: return 4;
    case ORACLE_F16:
    case ORACLE_BF16: return 2;
    default: return 0;
  }
}

/* Widen n stored elements to binary64 (exported so the tests can pin the
 * decoding of every 16-bit pattern against independent library routines). */
int oracle_widen(const void* src, double* dst, int64_t n, int dtype) {
  if (elt_bytes(dtype) == 0) return ORACLE_BAD_DTYPE;
  for (int64_t i = 0; i < n; ++i) dst[i] = load_elt(src, i, dtype);
  return ORACLE_OK;
}

/* Encode n binary32 values to E4M3 codes (exported so the tests can pin the
 * rounding against an independent library conversion). */
int oracle_e4m3_encode(const float* src, uint8_t* dst, int64_t n) {
  for (int64_t i = 0; i < n; ++i) dst[i] = double_to_e4m3((double)src[i]);
  return ORACLE_OK;
}

/*
 * KV-cache append into an FP8 (E4M3) cache with per-tensor scales.
 * key, value: [T][Hkv][D] dense, dtype f32/f16/bf16.  k_cache, v_cache:
 * [num_blocks][Hkv][block_size][D] bytes.  Every element x of key[t][h] is
 * stored as E4M3(fp32(x) * k_inv_scale) -- the product taken in binary32 --
 * in slot slot_mapping[t], and likewise for value with v_inv_scale.  Negative
 * slots write nothing; an out-of-range slot writes nothing and returns
 * ORACLE_SLOT_OUT_OF_RANGE.
 */
int oracle_reshape_and_cache_e4m3(const void* key, const void* value, uint8_t* k_cache, uint8_t* v_cache,
                                  const int64_t* slot_mapping, int64_t num_tokens, int64_t num_kv_heads,
                                  int64_t head_dim, int64_t num_blocks, int64_t block_size, int dtype,
                                  float k_inv_scale, float v_inv_scale) {
  if (elt_bytes(dtype) == 0 || dtype == ORACLE_E4M3) return ORACLE_BAD_DTYPE;
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks < 0 || block_size <= 0)
    return ORACLE_BAD_SHAPE;
  for (int64_t t = 0; t < num_tokens; ++t)
    if (slot_mapping[t] >= num_blocks * block_size) return ORACLE_SLOT_OUT_OF_RANGE;
  for (int64_t t = 0; t < num_tokens; ++t) {
    const int64_t s = slot_mapping[t];
    if (s < 0) continue;
    const int64_t blk = s / block_size, off = s % block_size;
    for (int64_t h = 0; h < num_kv_heads; ++h) {
      const int64_t src = (t * num_kv_heads + h) * head_dim;
      const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * head_dim;
      for (int64_t d = 0; d < head_dim; ++d) {
        const float xk = (float)load_elt(key, src + d, dtype);
        const float xv = (float)load_elt(value, src + d, dtype);
        const float yk = xk * k_inv_scale;
        const float yv = xv * v_inv_scale;
        k_cache[dst + d] = double_to_e4m3((double)yk);
        v_cache[dst + d] = double_to_e4m3((double)yv);
      }
    }
  }
  return ORACLE_OK;
}

/*
 * KV-cache append.  key, value: [T][Hkv][D] dense.  k_cache, v_cache:
 * [num_blocks][Hkv][block_size][D] dense.  For every t with
 * s = slot_mapping[t] >= 0 and every kv head h, the D stored elements of
 * key[t][h] are copied unchanged into k_cache[s / block_size][h]
 * [s % block_size], and likewise for value.  Every slot is checked before
 * anything is written; an out-of-range slot writes nothing and returns
 * ORACLE_SLOT_OUT_OF_RANGE.
 */
int oracle_reshape_and_cache(const void* key, const void* value, void* k_cache,
                             void* v_cache, const int64_t* slot_mapping,
                             int64_t num_tokens, int64_t num_kv_heads,
                             int64_t head_dim, int64_t num_blocks,
                             int64_t block_size, int dtype) {
  const int eb = elt_bytes(dtype);
  if (eb == 0) return ORACLE_BAD_DTYPE;
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      num_blocks < 0 || block_size <= 0)
    return ORACLE_BAD_SHAPE;
  for (int64_t t = 0; t < num_tokens; ++t)
    if (slot_mapping[t] >= num_blocks * block_size)
      return ORACLE_SLOT_OUT_OF_RANGE;
  const int64_t row_bytes = head_dim * eb;
  for (int64_t t = 0; t < num_tokens; ++t) {
    const int64_t s = slot_mapping[t];
    if (s < 0) continue; /* padding token: nothing to write */
    const int64_t blk = s / block_size, off = s % block_size;
    for (int64_t h = 0; h < num_kv_heads; ++h) {
      const int64_t src = (t * num_kv_heads + h) * row_bytes;
      const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * row_bytes;
      memcpy((char*)k_cache + dst, (const char*)key + src, (size_t)row_bytes);
      memcpy((char*)v_cache + dst, (const char*)value + src, (size_t)row_bytes);
    }
  }
  return ORACLE_OK;
}

/*
 * Paged decode attention for a chosen list of output rows.
 *
 * q: [B][Hq][D]; k_cache, v_cache: [num_blocks][Hkv][block_size][D];
 * block_tables: int32 [B][max_blocks]; context_lens: int32 [B].
 * rows: n_rows indices r = b * Hq + h (NULL means every row, in order).
 * out: binary64 [n_rows][D].
 *
 * For row (b, h): G = Hq / Hkv, kv head c = h / G, L = context_lens[b];
 * token j < L is K[table[b][j / bs]][c][j % bs][:] (and the same for V);
 * s_j = (double)scale * sum_d q[b][h][d] * K_j[d];
 * m = max_j s_j; w_j = exp(s_j - m);
 * out[b][h][:] = (sum_j w_j V_j[:]) / (sum_j w_j).
 * L == 0 gives zeros.  Inputs are validated first; nothing is written on error.
 */
int oracle_paged_decode_rows_kv(double* out, const int64_t* rows, int64_t n_rows,
                                const void* q, const void* k_cache,
                                const void* v_cache, const int32_t* block_tables,
                                const int32_t* context_lens, int64_t num_seqs,
                                int64_t num_q_heads, int64_t num_kv_heads,
                                int64_t head_dim, int64_t num_blocks,
                                int64_t block_size, int64_t max_blocks,
                                float scale, int dtype, int kv_dtype, float k_scale,
                                float v_scale, int num_threads) {
  if (elt_bytes(dtype) == 0 || dtype == ORACLE_E4M3 || elt_bytes(kv_dtype) == 0) return ORACLE_BAD_DTYPE;
  const double ks = (double)k_scale, vs = (double)v_scale;
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      block_size <= 0 || max_blocks < 0 || num_q_heads % num_kv_heads != 0)
    return ORACLE_BAD_SHAPE;
  if (rows == NULL && n_rows != num_seqs * num_q_heads) return ORACLE_BAD_SHAPE;
  const int64_t G = num_q_heads / num_kv_heads;
  const double scale_d = (double)scale;

  /* validate every row's sequence before computing anything */
  for (int64_t i = 0; i < n_rows; ++i) {
    const int64_t r = rows ? rows[i] : i;
    if (r < 0 || r >= num_seqs * num_q_heads) return ORACLE_BAD_SHAPE;
    const int64_t b = r / num_q_heads;
    const int64_t L = context_lens[b];
    if (L < 0 || L > max_blocks * block_size) return ORACLE_LEN_OUT_OF_RANGE;
    for (int64_t jb = 0; jb * block_size < L; ++jb) {
      const int64_t pb = block_tables[b * max_blocks + jb];
      if (pb < 0 || pb >= num_blocks) return ORACLE_BLOCK_OUT_OF_RANGE;
    }
  }

  int status = ORACLE_OK;
#ifdef _OPENMP
  if (num_threads <= 0) num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads)
#endif
  for (int64_t i = 0; i < n_rows; ++i) {
    const int64_t r = rows ? rows[i] : i;
    const int64_t b = r / num_q_heads, h = r % num_q_heads;
    const int64_t c = h / G;
    const int64_t L = context_lens[b];
    double* o = out + i * head_dim;
    for (int64_t d = 0; d < head_dim; ++d) o[d] = 0.0;
    if (L == 0) continue;

    double* s = (double*)malloc((size_t)L * sizeof(double));
    if (s == NULL) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      status = ORACLE_NO_MEMORY;
      continue;
    }
    const int64_t q_off = (b * num_q_heads + h) * head_dim;

    /* scores, in logical token order */
    for (int64_t j = 0; j < L; ++j) {
      const int64_t pb = block_tables[b * max_blocks + j / block_size];
      const int64_t k_off = ((pb * num_kv_heads + c) * block_size + j % block_size) * head_dim;
      double dot = 0.0;
      for (int64_t d = 0; d < head_dim; ++d)
        dot += load_elt(q, q_off + d, dtype) * (load_elt(k_cache, k_off + d, kv_dtype) * ks);
      s[j] = scale_d * dot;
    }
    double m = s[0];
    for (int64_t j = 1; j < L; ++j)
      if (s[j] > m) m = s[j];

    /* weights and the weighted sum of values */
    double denom = 0.0;
    for (int64_t j = 0; j < L; ++j) {
      const double w = exp(s[j] - m);
      denom += w;
      const int64_t pb = block_tables[b * max_blocks + j / block_size];
      const int64_t v_off = ((pb * num_kv_heads + c) * block_size + j % block_size) * head_dim;
      for (int64_t d = 0; d < head_dim; ++d) o[d] += w * (load_elt(v_cache, v_off + d, kv_dtype) * vs);
    }
    for (int64_t d = 0; d < head_dim; ++d) o[d] /= denom;
    free(s);
  }
  return status;
}

/* The same with K/V stored like q (scales 1). */
int oracle_paged_decode_rows(double* out, const int64_t* rows, int64_t n_rows, const void* q,
                             const void* k_cache, const void* v_cache, const int32_t* block_tables,
                             const int32_t* context_lens, int64_t num_seqs, int64_t num_q_heads,
                             int64_t num_kv_heads, int64_t head_dim, int64_t num_blocks,
                             int64_t block_size, int64_t max_blocks, float scale, int dtype,
                             int num_threads) {
  return oracle_paged_decode_rows_kv(out, rows, n_rows, q, k_cache, v_cache, block_tables,
                                     context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                     num_blocks, block_size, max_blocks, scale, dtype, dtype, 1.0f,
                                     1.0f, num_threads);
}

/*
 * Chunked-prefill (multi-query) paged attention for a chosen list of output
 * rows.  Source: the "wLLM" project page, "Features / Core engine" (chunked
 * prefill: a long prompt enters the cache a chunk at a time, between decode
 * steps, through the same paged KV cache).  Reading: causal attention, each
 * chunk token seeing the cached tokens before it and itself.
 *
 * q: [T][Hq][D], the chunks of all sequences packed one after another:
 * sequence b owns q rows query_start_loc[b] .. query_start_loc[b+1]-1 (n_b of
 * them, n_b may be 0).  Its chunk is the last n_b of its L = context_lens[b]
 * tokens, whose K/V are already in the cache: chunk token i sits at position
 * P = L - n_b + i, and for query head h (kv head c = h / G)
 *   s_j = (double)scale * sum_d q[t][h][d] * K_j[d]   for j = 0 .. P,
 *   out[t][h][:] = sum_j exp(s_j - m) V_j[:] / sum_j exp(s_j - m),  m = max_j s_j.
 * rows: indices r = t * Hq + h (NULL: every row in order); out: binary64
 * [n_rows][D].  Decode is the case n_b = 1.  K/V are stored as kv_dtype
 * (q's type, or E4M3 codes whose values are code * k_scale, resp.
 * v_scale, the scales widened from binary32).  Inputs are validated first;
 * nothing is written on error.
 */
int oracle_paged_prefill_rows_kv(double* out, const int64_t* rows, int64_t n_rows, const void* q,
                                 const void* k_cache, const void* v_cache, const int32_t* block_tables,
                                 const int32_t* context_lens, const int32_t* query_start_loc,
                                 int64_t num_seqs, int64_t num_tokens, int64_t num_q_heads,
                                 int64_t num_kv_heads, int64_t head_dim, int64_t num_blocks,
                                 int64_t block_size, int64_t max_blocks, float scale, int dtype,
                                 int kv_dtype, float k_scale, float v_scale, int num_threads) {
  if (elt_bytes(dtype) == 0 || dtype == ORACLE_E4M3 || elt_bytes(kv_dtype) == 0) return ORACLE_BAD_DTYPE;
  const double ks = (double)k_scale, vs = (double)v_scale;
  if (num_seqs < 0 || num_tokens < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      block_size <= 0 || max_blocks < 0 || num_q_heads % num_kv_heads != 0)
    return ORACLE_BAD_SHAPE;
  if (rows == NULL && n_rows != num_tokens * num_q_heads) return ORACLE_BAD_SHAPE;
  if (query_start_loc[0] != 0 || query_start_loc[num_seqs] != num_tokens) return ORACLE_BAD_SHAPE;
  for (int64_t b = 0; b < num_seqs; ++b) {
    const int64_t n = (int64_t)query_start_loc[b + 1] - query_start_loc[b];
    const int64_t L = context_lens[b];
    if (n < 0) return ORACLE_BAD_SHAPE;
    if (L < n || L > max_blocks * block_size) return ORACLE_LEN_OUT_OF_RANGE;
    if (n == 0) continue;
    for (int64_t jb = 0; jb * block_size < L; ++jb) {
      const int64_t pb = block_tables[b * max_blocks + jb];
      if (pb < 0 || pb >= num_blocks) return ORACLE_BLOCK_OUT_OF_RANGE;
    }
  }
  for (int64_t i = 0; i < n_rows; ++i) {
    const int64_t r = rows ? rows[i] : i;
    if (r < 0 || r >= num_tokens * num_q_heads) return ORACLE_BAD_SHAPE;
  }
  const int64_t G = num_q_heads / num_kv_heads;
  const double scale_d = (double)scale;

  int status = ORACLE_OK;
#ifdef _OPENMP
  if (num_threads <= 0) num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads)
#endif
  for (int64_t i = 0; i < n_rows; ++i) {
    const int64_t r = rows ? rows[i] : i;
    const int64_t t = r / num_q_heads, h = r % num_q_heads;
    const int64_t c = h / G;
    /* the sequence owning packed token t: the last b with query_start_loc[b] <= t */
    int64_t lo = 0, hi = num_seqs - 1;
    while (lo < hi) {
      const int64_t mid = (lo + hi + 1) / 2;
      if (query_start_loc[mid] <= t) lo = mid;
      else hi = mid - 1;
    }
    const int64_t b = lo;
    const int64_t n = (int64_t)query_start_loc[b + 1] - query_start_loc[b];
    const int64_t L = context_lens[b];
    const int64_t P = L - n + (t - query_start_loc[b]); /* this token's position */
    double* o = out + i * head_dim;
    for (int64_t d = 0; d < head_dim; ++d) o[d] = 0.0;

    double* s = (double*)malloc((size_t)(P + 1) * sizeof(double));
    if (s == NULL) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      status = ORACLE_NO_MEMORY;
      continue;
    }
    const int64_t q_off = (t * num_q_heads + h) * head_dim;
    for (int64_t j = 0; j <= P; ++j) {
      const int64_t pb = block_tables[b * max_blocks + j / block_size];
      const int64_t k_off = ((pb * num_kv_heads + c) * block_size + j % block_size) * head_dim;
      double dot = 0.0;
      for (int64_t d = 0; d < head_dim; ++d)
        dot += load_elt(q, q_off + d, dtype) * (load_elt(k_cache, k_off + d, kv_dtype) * ks);
      s[j] = scale_d * dot;
    }
    double m = s[0];
    for (int64_t j = 1; j <= P; ++j)
      if (s[j] > m) m = s[j];
    double denom = 0.0;
    for (int64_t j = 0; j <= P; ++j) {
      const double w = exp(s[j] - m);
      denom += w;
      const int64_t pb = block_tables[b * max_blocks + j / block_size];
      const int64_t v_off = ((pb * num_kv_heads + c) * block_size + j % block_size) * head_dim;
      for (int64_t d = 0; d < head_dim; ++d) o[d] += w * (load_elt(v_cache, v_off + d, kv_dtype) * vs);
    }
    for (int64_t d = 0; d < head_dim; ++d) o[d] /= denom;
    free(s);
  }
  return status;
}

/* The same with K/V stored like q (scales 1). */
int oracle_paged_prefill_rows(double* out, const int64_t* rows, int64_t n_rows, const void* q,
                              const void* k_cache, const void* v_cache, const int32_t* block_tables,
                              const int32_t* context_lens, const int32_t* query_start_loc,
                              int64_t num_seqs, int64_t num_tokens, int64_t num_q_heads,
                              int64_t num_kv_heads, int64_t head_dim, int64_t num_blocks,
                              int64_t block_size, int64_t max_blocks, float scale, int dtype,
                              int num_threads) {
  return oracle_paged_prefill_rows_kv(out, rows, n_rows, q, k_cache, v_cache, block_tables, context_lens,
                                      query_start_loc, num_seqs, num_tokens, num_q_heads, num_kv_heads,
                                      head_dim, num_blocks, block_size, max_blocks, scale, dtype, dtype,
                                      1.0f, 1.0f, num_threads);
}

/* Number of threads an OpenMP region uses by default (1 without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
