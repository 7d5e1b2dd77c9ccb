/*
 * Plain fp64 CPU oracle for paged decode attention and its KV write path.
 * TEST INFRASTRUCTURE ONLY: see oracle.h for who may use it and which passages
 * of the pages each function follows. Deliberately slow and unblocked: one
 * (sequence, query head) at a time, positions in order, fp64 throughout.
 */
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- codecs */

/* IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double orc_f16_to_f64(uint16_t h) {
  int s = (h >> 15) & 1;
  int e = (h >> 10) & 0x1F;
  int m = h & 0x3FF;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -24); /* 2^-14 * m / 1024 */
  } else if (e == 31) {
    v = (m == 0) ? INFINITY : NAN;
  } else {
    v = ldexp(1.0 + (double)m / 1024.0, e - 15);
  }
  return s ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32: 1 sign, 8 exponent
 * (bias 127), 7 fraction bits. */
double orc_bf16_to_f64(uint16_t h) {
  int s = (h >> 15) & 1;
  int e = (h >> 7) & 0xFF;
  int m = h & 0x7F;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -133); /* 2^-126 * m / 128 */
  } else if (e == 255) {
    v = (m == 0) ? INFINITY : NAN;
  } else {
    v = ldexp(1.0 + (double)m / 128.0, e - 127);
  }
  return s ? -v : v;
}

/* OCP E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits. Exponent 0 is
 * subnormal (2^-6 * m / 8). There are no infinities; S.1111.111 is NaN, so the
 * largest finite magnitude is 1.75 * 2^8 = 448. */
double orc_e4m3_to_f64(uint8_t c) {
  int s = (c >> 7) & 1;
  int e = (c >> 3) & 0xF;
  int m = c & 0x7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) {
    v = ldexp((double)m, -9);
  } else {
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  }
  return s ? -v : v;
}

/* Round a non-negative double to an integer, ties to even. */
static double round_half_even(double q) {
  double r = floor(q);
  double f = q - r;
  if (f > 0.5) return r + 1.0;
  if (f < 0.5) return r;
  return (fmod(r, 2.0) == 0.0) ? r : r + 1.0;
}

uint8_t orc_e4m3_from_f32(float x) {
  if (isnan(x)) return 0x7F;
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs((double)x);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E); /* saturate, includes inf */
  if (a < ldexp(1.0, -6)) {
    /* subnormal grid: multiples of 2^-9; m == 8 is the smallest normal 0x08 */
    double m = round_half_even(a * 512.0);
    return (uint8_t)(sign | (uint8_t)m);
  }
  int ex;
  double f = frexp(a, &ex); /* a = f * 2^ex, f in [0.5, 1) */
  int e = ex - 1;           /* a = (2f) * 2^e, 2f in [1, 2) */
  double q = (2.0 * f - 1.0) * 8.0;
  double m = round_half_even(q);
  if (m == 8.0) {
    m = 0.0;
    e += 1;
  }
  /* a < 448 keeps e + 7 <= 15 and excludes the NaN pattern. */
  return (uint8_t)(sign | (uint8_t)((e + 7) << 3) | (uint8_t)m);
}

void orc_decode16_array(const uint16_t* src, int dtype, double* dst, int64_t n) {
  for (int64_t i = 0; i < n; ++i)
    dst[i] = (dtype == ORC_F16) ? orc_f16_to_f64(src[i]) : orc_bf16_to_f64(src[i]);
}

void orc_e4m3_decode_array(const uint8_t* src, double* dst, int64_t n) {
  for (int64_t i = 0; i < n; ++i) dst[i] = orc_e4m3_to_f64(src[i]);
}

void orc_e4m3_encode_array(const float* src, uint8_t* dst, int64_t n) {
  for (int64_t i = 0; i < n; ++i) dst[i] = orc_e4m3_from_f32(src[i]);
}

static double decode16(uint16_t x, int dtype) {
  return dtype == ORC_F16 ? orc_f16_to_f64(x) : orc_bf16_to_f64(x);
}

/* ------------------------------------------------------------ threading */

typedef void (*orc_range_fn)(void* ctx, int64_t lo, int64_t hi);

typedef struct {
  orc_range_fn fn;
  void* ctx;
  int64_t lo, hi;
} orc_job;

static void* orc_job_main(void* p) {
  orc_job* j = (orc_job*)p;
  j->fn(j->ctx, j->lo, j->hi);
  return NULL;
}

/* Runs fn over [0, n) split into contiguous chunks, one per thread. Every item
 * is computed by exactly one thread with the same arithmetic, so the result
 * does not depend on the thread count. */
static void orc_parallel(orc_range_fn fn, void* ctx, int64_t n, int threads) {
  if (threads < 1) threads = 1;
  if ((int64_t)threads > n) threads = (int)(n > 0 ? n : 1);
  if (threads == 1) {
    fn(ctx, 0, n);
    return;
  }
  pthread_t* tid = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)threads);
  orc_job* jobs = (orc_job*)malloc(sizeof(orc_job) * (size_t)threads);
  int started = 0;
  for (int i = 0; i < threads; ++i) {
    jobs[i].fn = fn;
    jobs[i].ctx = ctx;
    jobs[i].lo = n * i / threads;
    jobs[i].hi = n * (i + 1) / threads;
    if (pthread_create(&tid[i], NULL, orc_job_main, &jobs[i]) == 0) {
      started = i + 1;
    } else {
      /* could not start a thread: run the rest here */
      fn(ctx, jobs[i].lo, n);
      break;
    }
  }
  for (int i = 0; i < started; ++i) pthread_join(tid[i], NULL);
  free(jobs);
  free(tid);
}

/* ------------------------------------------------------------ write path */

typedef struct {
  const uint16_t *k, *v;
  int64_t H, D;
  int src_dtype;
  void *kc, *vc;
  int64_t nb, bs;
  int cache_dtype;
  const int64_t* slots;
  float k_scale, v_scale;
} orc_reshape_ctx;

static void orc_store(const uint16_t* src, void* cache, int64_t dst_row, int64_t D,
                      int src_dtype, int cache_dtype, float scale) {
  if (cache_dtype == ORC_E4M3) {
    uint8_t* dst = (uint8_t*)cache + dst_row * D;
    for (int64_t d = 0; d < D; ++d) {
      float xf = (float)decode16(src[d], src_dtype);
      float qv = xf / scale; /* fp32 IEEE division */
      dst[d] = orc_e4m3_from_f32(qv);
    }
  } else {
    uint16_t* dst = (uint16_t*)cache + dst_row * D;
    for (int64_t d = 0; d < D; ++d) dst[d] = src[d];
  }
}

static void orc_reshape_range(void* p, int64_t lo, int64_t hi) {
  orc_reshape_ctx* c = (orc_reshape_ctx*)p;
  for (int64_t t = lo; t < hi; ++t) {
    int64_t slot = c->slots[t];
    if (slot < 0) continue;
    int64_t blk = slot / c->bs, off = slot % c->bs;
    for (int64_t h = 0; h < c->H; ++h) {
      int64_t row = (blk * c->H + h) * c->bs + off;
      const int64_t src = (t * c->H + h) * c->D;
      orc_store(c->k + src, c->kc, row, c->D, c->src_dtype, c->cache_dtype, c->k_scale);
      orc_store(c->v + src, c->vc, row, c->D, c->src_dtype, c->cache_dtype, c->v_scale);
    }
  }
}

int orc_reshape_and_cache(const uint16_t* k, const uint16_t* v, int64_t num_tokens,
                          int64_t num_heads, int64_t head_dim, int src_dtype,
                          void* key_cache, void* value_cache, int64_t num_blocks,
                          int64_t block_size, int cache_dtype, const int64_t* slot_mapping,
                          float k_scale, float v_scale, int threads) {
  if (num_tokens < 0 || num_heads <= 0 || head_dim <= 0 || block_size <= 0) return ORC_EINVAL;
  if (src_dtype != ORC_F16 && src_dtype != ORC_BF16) return ORC_EINVAL;
  if (cache_dtype != src_dtype && cache_dtype != ORC_E4M3) return ORC_EINVAL;
  for (int64_t t = 0; t < num_tokens; ++t)
    if (slot_mapping[t] >= num_blocks * block_size) return ORC_ERANGE;
  orc_reshape_ctx c = {k, v, num_heads, head_dim, src_dtype, key_cache, value_cache,
                       num_blocks, block_size, cache_dtype, slot_mapping, k_scale, v_scale};
  orc_parallel(orc_reshape_range, &c, num_tokens, threads);
  return ORC_OK;
}

/* --------------------------------------------------------------- decode */

typedef struct {
  double* out;
  const uint16_t* q;
  int q_dtype;
  const void *kc, *vc;
  int cache_dtype;
  const int32_t *bt, *lens;
  int64_t B, Hq, Hkv, D, nb, bs, mb, window;
  double scale, k_scale, v_scale;
  const int32_t* pairs;
  volatile int err;
} orc_decode_ctx;

/* Value of element d of row `row` (= (block * Hkv + kv_head) * bs + offset). */
static double cache_elem(const orc_decode_ctx* c, const void* cache, int64_t row, int64_t d,
                         double scale) {
  if (c->cache_dtype == ORC_E4M3)
    return orc_e4m3_to_f64(((const uint8_t*)cache)[row * c->D + d]) * scale;
  return decode16(((const uint16_t*)cache)[row * c->D + d], c->cache_dtype);
}

static void orc_decode_one(orc_decode_ctx* c, int64_t b, int64_t h, double* s) {
  const int64_t D = c->D;
  double* o = c->out + (b * c->Hq + h) * D;
  const int64_t group = c->Hq / c->Hkv;
  const int64_t kvh = h / group;
  const int64_t L = c->lens[b];
  const int64_t start = (c->window > 0 && L > c->window) ? L - c->window : 0;
  for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
  if (L <= 0) return;
  if (L > c->mb * c->bs) {
    c->err = ORC_ERANGE;
    return;
  }
  const uint16_t* qh = c->q + (b * c->Hq + h) * D;

  /* scores s_j = scale * sum_d q_d K_jd over attended positions j */
  double m = -INFINITY;
  for (int64_t j = start; j < L; ++j) {
    int64_t blk = c->bt[b * c->mb + j / c->bs];
    if (blk < 0 || blk >= c->nb) {
      c->err = ORC_ERANGE;
      return;
    }
    int64_t row = (blk * c->Hkv + kvh) * c->bs + j % c->bs;
    double dot = 0.0;
    for (int64_t d = 0; d < D; ++d)
      dot += decode16(qh[d], c->q_dtype) * cache_elem(c, c->kc, row, d, c->k_scale);
    s[j - start] = c->scale * dot;
    if (s[j - start] > m) m = s[j - start];
  }
  /* softmax weights and the weighted sum of V rows */
  double den = 0.0;
  for (int64_t j = start; j < L; ++j) {
    double w = exp(s[j - start] - m);
    den += w;
    int64_t blk = c->bt[b * c->mb + j / c->bs];
    int64_t row = (blk * c->Hkv + kvh) * c->bs + j % c->bs;
    for (int64_t d = 0; d < D; ++d) o[d] += w * cache_elem(c, c->vc, row, d, c->v_scale);
  }
  for (int64_t d = 0; d < D; ++d) o[d] /= den;
}

static void orc_decode_range(void* p, int64_t lo, int64_t hi) {
  orc_decode_ctx* c = (orc_decode_ctx*)p;
  int64_t maxlen = c->mb * c->bs;
  double* s = (double*)malloc(sizeof(double) * (size_t)(maxlen > 0 ? maxlen : 1));
  if (!s) {
    c->err = ORC_ENOMEM;
    return;
  }
  for (int64_t i = lo; i < hi; ++i) {
    int64_t b, h;
    if (c->pairs) {
      b = c->pairs[2 * i];
      h = c->pairs[2 * i + 1];
    } else {
      b = i / c->Hq;
      h = i % c->Hq;
    }
    orc_decode_one(c, b, h, s);
  }
  free(s);
}

int orc_decode(double* out, const uint16_t* q, int q_dtype, const void* key_cache,
               const void* value_cache, int cache_dtype, const int32_t* block_tables,
               const int32_t* seq_lens, int64_t batch, int64_t num_q_heads,
               int64_t num_kv_heads, int64_t head_dim, int64_t num_blocks,
               int64_t block_size, int64_t max_blocks, double scale, int64_t window,
               double k_scale, double v_scale, const int32_t* pairs, int64_t n_pairs,
               int threads) {
  if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0) return ORC_EINVAL;
  if (num_q_heads % num_kv_heads != 0 || block_size <= 0 || max_blocks < 0) return ORC_EINVAL;
  if (q_dtype != ORC_F16 && q_dtype != ORC_BF16) return ORC_EINVAL;
  if (cache_dtype != ORC_F16 && cache_dtype != ORC_BF16 && cache_dtype != ORC_E4M3)
    return ORC_EINVAL;
  int64_t n = pairs ? n_pairs : batch * num_q_heads;
  if (pairs) {
    for (int64_t i = 0; i < n; ++i)
      if (pairs[2 * i] < 0 || pairs[2 * i] >= batch || pairs[2 * i + 1] < 0 ||
          pairs[2 * i + 1] >= num_q_heads)
        return ORC_EINVAL;
  }
  orc_decode_ctx c = {out, q, q_dtype, key_cache, value_cache, cache_dtype, block_tables,
                      seq_lens, batch, num_q_heads, num_kv_heads, head_dim, num_blocks,
                      block_size, max_blocks, window, scale, k_scale, v_scale, pairs, 0};
  orc_parallel(orc_decode_range, &c, n, threads);
  return c.err;
}

/* ------------------------------------------------- multi-token (causal) */

typedef struct {
  double* out;
  const uint16_t* q;
  int q_dtype;
  const void *kc, *vc;
  int cache_dtype;
  const int32_t *bt, *lens;
  int64_t B, T, Hq, Hkv, D, nb, bs, mb, window;
  double scale, k_scale, v_scale;
  const int32_t* triples;
  volatile int err;
} orc_multi_ctx;

/* Query t of sequence b, head h: softmax over [start_t, p_t] of the causal
 * prefix ending at its own position. */
static void orc_multi_one(orc_multi_ctx* c, int64_t b, int64_t t, int64_t h, double* s) {
  const int64_t D = c->D;
  double* o = c->out + ((b * c->T + t) * c->Hq + h) * D;
  for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
  const int64_t L = c->lens[b];
  if (L > c->mb * c->bs) {
    c->err = ORC_ERANGE;
    return;
  }
  const int64_t p = L - c->T + t; /* this query's position */
  if (p < 0) return;
  const int64_t start = (c->window > 0 && p + 1 > c->window) ? p + 1 - c->window : 0;
  const int64_t kvh = h / (c->Hq / c->Hkv);
  const uint16_t* qh = c->q + ((b * c->T + t) * c->Hq + h) * D;
  orc_decode_ctx view = {0};
  view.kc = c->kc;
  view.vc = c->vc;
  view.cache_dtype = c->cache_dtype;
  view.D = D;
  double m = -INFINITY;
  for (int64_t j = start; j <= p; ++j) {
    int64_t blk = c->bt[b * c->mb + j / c->bs];
    if (blk < 0 || blk >= c->nb) {
      c->err = ORC_ERANGE;
      return;
    }
    int64_t row = (blk * c->Hkv + kvh) * c->bs + j % c->bs;
    double dot = 0.0;
    for (int64_t d = 0; d < D; ++d)
      dot += decode16(qh[d], c->q_dtype) * cache_elem(&view, c->kc, row, d, c->k_scale);
    s[j - start] = c->scale * dot;
    if (s[j - start] > m) m = s[j - start];
  }
  double den = 0.0;
  for (int64_t j = start; j <= p; ++j) {
    double w = exp(s[j - start] - m);
    den += w;
    int64_t blk = c->bt[b * c->mb + j / c->bs];
    int64_t row = (blk * c->Hkv + kvh) * c->bs + j % c->bs;
    for (int64_t d = 0; d < D; ++d) o[d] += w * cache_elem(&view, c->vc, row, d, c->v_scale);
  }
  for (int64_t d = 0; d < D; ++d) o[d] /= den;
}

static void orc_multi_range(void* p, int64_t lo, int64_t hi) {
  orc_multi_ctx* c = (orc_multi_ctx*)p;
  int64_t maxlen = c->mb * c->bs;
  double* s = (double*)malloc(sizeof(double) * (size_t)(maxlen > 0 ? maxlen : 1));
  if (!s) {
    c->err = ORC_ENOMEM;
    return;
  }
  for (int64_t i = lo; i < hi; ++i) {
    int64_t b, t, h;
    if (c->triples) {
      b = c->triples[3 * i];
      t = c->triples[3 * i + 1];
      h = c->triples[3 * i + 2];
    } else {
      b = i / (c->T * c->Hq);
      t = (i / c->Hq) % c->T;
      h = i % c->Hq;
    }
    orc_multi_one(c, b, t, h, s);
  }
  free(s);
}

int orc_decode_multi(double* out, const uint16_t* q, int q_dtype, const void* key_cache,
                     const void* value_cache, int cache_dtype, const int32_t* block_tables,
                     const int32_t* seq_lens, int64_t batch, int64_t num_queries,
                     int64_t num_q_heads, int64_t num_kv_heads, int64_t head_dim,
                     int64_t num_blocks, int64_t block_size, int64_t max_blocks, double scale,
                     int64_t window, double k_scale, double v_scale, const int32_t* triples,
                     int64_t n_triples, int threads) {
  if (batch < 0 || num_queries <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return ORC_EINVAL;
  if (num_q_heads % num_kv_heads != 0 || block_size <= 0 || max_blocks < 0) return ORC_EINVAL;
  if (q_dtype != ORC_F16 && q_dtype != ORC_BF16) return ORC_EINVAL;
  if (cache_dtype != ORC_F16 && cache_dtype != ORC_BF16 && cache_dtype != ORC_E4M3)
    return ORC_EINVAL;
  int64_t n = triples ? n_triples : batch * num_queries * num_q_heads;
  if (triples) {
    for (int64_t i = 0; i < n; ++i)
      if (triples[3 * i] < 0 || triples[3 * i] >= batch || triples[3 * i + 1] < 0 ||
          triples[3 * i + 1] >= num_queries || triples[3 * i + 2] < 0 ||
          triples[3 * i + 2] >= num_q_heads)
        return ORC_EINVAL;
  }
  orc_multi_ctx c = {out, q, q_dtype, key_cache, value_cache, cache_dtype, block_tables,
                     seq_lens, batch, num_queries, num_q_heads, num_kv_heads, head_dim,
                     num_blocks, block_size, max_blocks, window, scale, k_scale, v_scale,
                     triples, 0};
  orc_parallel(orc_multi_range, &c, n, threads);
  return c.err;
}
