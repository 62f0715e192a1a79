/*
 * mla_oracle.c -- float64 CPU oracle for MLA attention over an FP8-e4m3 latent KV cache.
 *
 * TEST INFRASTRUCTURE ONLY: called by the tests, by the package smoke check and by the
 * benchmark's CPU-baseline leg; never by the library. It is deliberately plain: every
 * query row is computed on its own, straight from the definition, in double precision,
 * with no blocking, fusion or reordering. Parallelism is OpenMP over independent rows.
 *
 * Definition followed for one query row r = (sequence b, new position j, head h):
 *   k[n][d]  = e4m3(code[n][d]) * kv_scale            d < 576   (whole row is the key)
 *   v[n][d]  = k[n][d]                                 d < 512   (first 512 entries are the value)
 *   s_n      = sm_scale * sum_d q[d] * k[n][d]
 *   visible  = { n : n <= L_b - n_q + j }               (causal, new positions last)
 *   lse      = m + ln sum_visible exp(s_n - m),  m = max_visible s_n
 *   out[d]   = sum_visible exp(s_n - lse) * v[n][d]
 * Sources: "MI355X Kimi K2.5 vLLM AITER 7x speedup", section "PR #35850 修复了什么" (keys
 * and values projected into one shared latent, FP8 KV cache); "Scaling Kimi K3 on AMD
 * Instinct MI355X", section "缓存可复用，还要能一致地恢复" (576 FP8 bytes per position;
 * partial attention merged by normalisation statistics), section "并行度必须适配真正的形状"
 * (heads attend independently).
 */
#include "mla_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_D 576
#define ORACLE_DV 512

/* OCP 8-bit floating point, E4M3 ("fn": finite, NaN only at S.1111.111):
 *   exponent field e in 1..15: (1 + m/8) * 2^(e-7);  e = 0: (m/8) * 2^-6. */
double oracle_e4m3_value(uint8_t code) {
  int sign = (code >> 7) & 1;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double mag;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, -6);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -mag : mag;
}

/* bfloat16 is the top 16 bits of an IEEE binary32. */
double oracle_bf16_value(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Address of cached position n of sequence b, or NULL if the page table points outside the pool. */
static const uint8_t* key_row(const uint8_t* pool, int64_t num_pages, int page_size,
                              const int32_t* page_table, int64_t pt_stride, int b, int64_t n) {
  int64_t logical_page = n / page_size;
  int32_t phys = page_table[(int64_t)b * pt_stride + logical_page];
  if (phys < 0 || phys >= num_pages) return NULL;
  return pool + ((int64_t)phys * page_size + (n % page_size)) * ORACLE_D;
}

/* Attention of one query q[576] (already in double) over keys [lo, hi) of sequence b.
 * scores is caller scratch of at least hi - lo doubles. Returns 0 or -1 (bad page). */
static int attend(const uint8_t* pool, int64_t num_pages, int page_size,
                  const int32_t* page_table, int64_t pt_stride, int b, int64_t lo, int64_t hi,
                  const double* table, const double* q, double sm_scale, double* scores,
                  double* out, double* lse) {
  for (int d = 0; d < ORACLE_DV; ++d) out[d] = 0.0;
  if (hi <= lo) {
    *lse = -INFINITY;
    return 0;
  }
  double m = -INFINITY;
  for (int64_t n = lo; n < hi; ++n) {
    const uint8_t* row = key_row(pool, num_pages, page_size, page_table, pt_stride, b, n);
    if (!row) return -1;
    double acc = 0.0;
    for (int d = 0; d < ORACLE_D; ++d) acc += q[d] * table[row[d]];
    scores[n - lo] = sm_scale * acc;
    if (scores[n - lo] > m) m = scores[n - lo];
  }
  double sum = 0.0;
  for (int64_t n = lo; n < hi; ++n) sum += exp(scores[n - lo] - m);
  double l = m + log(sum);
  for (int64_t n = lo; n < hi; ++n) {
    const uint8_t* row = key_row(pool, num_pages, page_size, page_table, pt_stride, b, n);
    double w = exp(scores[n - lo] - l);
    for (int d = 0; d < ORACLE_DV; ++d) out[d] += w * table[row[d]];
  }
  *lse = l;
  return 0;
}

static void build_table(double kv_scale, double* table) {
  for (int c = 0; c < 256; ++c) table[c] = oracle_e4m3_value((uint8_t)c) * kv_scale;
}

int oracle_attention_rows(const uint8_t* pool, int64_t num_pages, int page_size,
                          const int32_t* page_table, int64_t pt_stride, const int32_t* seq_lens,
                          double kv_scale, const uint16_t* q_bf16, int B, int n_q, int H,
                          double sm_scale, const int32_t* rows_b, const int32_t* rows_j,
                          const int32_t* rows_h, int64_t n_rows, double* out, double* lse,
                          int n_threads) {
  if (page_size <= 0 || B < 0 || n_q <= 0 || H <= 0) return -1;
  int64_t max_len = 0;
  for (int b = 0; b < B; ++b) {
    if (seq_lens[b] < 0) return -1;
    if (seq_lens[b] > max_len) max_len = seq_lens[b];
  }
  double table[256];
  build_table(kv_scale, table);
  int failed = 0;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#else
  (void)n_threads;
#endif
#pragma omp parallel
  {
    double* scores = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
    double q[ORACLE_D];
#pragma omp for schedule(dynamic, 1)
    for (int64_t i = 0; i < n_rows; ++i) {
      int b = rows_b[i], j = rows_j[i], h = rows_h[i];
      const uint16_t* qr = q_bf16 + (((int64_t)b * n_q + j) * H + h) * ORACLE_D;
      for (int d = 0; d < ORACLE_D; ++d) q[d] = oracle_bf16_value(qr[d]);
      int64_t visible = (int64_t)seq_lens[b] - n_q + j + 1; /* keys 0 .. L - n_q + j */
      if (visible < 0) visible = 0;
      if (attend(pool, num_pages, page_size, page_table, pt_stride, b, 0, visible, table, q,
                 sm_scale, scores, out + i * ORACLE_DV, lse + i) != 0) {
#pragma omp atomic write
        failed = 1;
      }
    }
    free(scores);
  }
  return failed ? -1 : 0;
}

int oracle_attention(const uint8_t* pool, int64_t num_pages, int page_size,
                     const int32_t* page_table, int64_t pt_stride, const int32_t* seq_lens,
                     double kv_scale, const uint16_t* q_bf16, int B, int n_q, int H,
                     double sm_scale, double* out, double* lse, int n_threads) {
  int64_t n_rows = (int64_t)B * n_q * H;
  int32_t* rb = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n_rows > 0 ? n_rows : 1));
  int32_t* rj = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n_rows > 0 ? n_rows : 1));
  int32_t* rh = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n_rows > 0 ? n_rows : 1));
  int64_t i = 0;
  for (int b = 0; b < B; ++b)
    for (int j = 0; j < n_q; ++j)
      for (int h = 0; h < H; ++h, ++i) {
        rb[i] = b;
        rj[i] = j;
        rh[i] = h;
      }
  int rc = oracle_attention_rows(pool, num_pages, page_size, page_table, pt_stride, seq_lens,
                                 kv_scale, q_bf16, B, n_q, H, sm_scale, rb, rj, rh, n_rows, out,
                                 lse, n_threads);
  free(rb);
  free(rj);
  free(rh);
  return rc;
}

int oracle_attention_range(const uint8_t* pool, int64_t num_pages, int page_size,
                           const int32_t* page_table, int64_t pt_stride, int b,
                           int64_t key_lo, int64_t key_hi, double kv_scale,
                           const uint16_t* q_row_bf16, double sm_scale, double* out,
                           double* lse) {
  double table[256];
  double q[ORACLE_D];
  build_table(kv_scale, table);
  for (int d = 0; d < ORACLE_D; ++d) q[d] = oracle_bf16_value(q_row_bf16[d]);
  int64_t n = key_hi > key_lo ? key_hi - key_lo : 1;
  double* scores = (double*)malloc(sizeof(double) * (size_t)n);
  int rc = attend(pool, num_pages, page_size, page_table, pt_stride, b, key_lo, key_hi, table, q,
                  sm_scale, scores, out, lse);
  free(scores);
  return rc;
}

void oracle_merge_lse(const double* part_out, const double* part_lse, int S, int64_t R,
                      double* out, double* lse) {
  for (int64_t r = 0; r < R; ++r) {
    double m = -INFINITY;
    for (int s = 0; s < S; ++s)
      if (part_lse[(int64_t)s * R + r] > m) m = part_lse[(int64_t)s * R + r];
    for (int d = 0; d < ORACLE_DV; ++d) out[r * ORACLE_DV + d] = 0.0;
    if (m == -INFINITY) {
      lse[r] = -INFINITY;
      continue;
    }
    double sum = 0.0;
    for (int s = 0; s < S; ++s) sum += exp(part_lse[(int64_t)s * R + r] - m);
    double l = m + log(sum);
    for (int s = 0; s < S; ++s) {
      double w = exp(part_lse[(int64_t)s * R + r] - l);
      if (w == 0.0) continue;
      const double* o = part_out + ((int64_t)s * R + r) * ORACLE_DV;
      for (int d = 0; d < ORACLE_DV; ++d) out[r * ORACLE_DV + d] += w * o[d];
    }
    lse[r] = l;
  }
}

/* Nearest finite e4m3 value by exhaustive comparison with the 127 non-negative codes
 * 0x00..0x7E (0x7F is NaN); a tie goes to the even code, whose mantissa bit 0 is clear. */
uint8_t oracle_e4m3_encode(double v) {
  if (isnan(v)) return 0x7F;
  const uint8_t sign = signbit(v) ? 0x80 : 0x00;
  double a = fabs(v);
  if (a > 448.0) a = 448.0;
  int best = 0;
  double best_err = INFINITY;
  for (int c = 0; c <= 0x7E; ++c) {
    const double err = fabs(oracle_e4m3_value((uint8_t)c) - a);
    if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      best_err = err;
    }
  }
  return (uint8_t)(sign | best);
}

int oracle_cache_append(uint8_t* pool, int64_t pool_rows, const uint16_t* x_bf16,
                        const int64_t* slots, int64_t n, float kv_scale) {
  /* binary32 arithmetic as the definition states (C evaluates float * float in float on the
     targets this is built for: FLT_EVAL_METHOD 0) */
  const float inv = 1.0f / kv_scale;
  int rc = 0;
  for (int64_t i = 0; i < n; ++i) {
    const int64_t s = slots[i];
    if (s < 0) continue;
    if (s >= pool_rows) {
      rc = -1;
      continue;
    }
    for (int d = 0; d < ORACLE_D; ++d) {
      const float x = (float)oracle_bf16_value(x_bf16[i * ORACLE_D + d]);
      const float prod = x * inv;
      pool[s * ORACLE_D + d] = oracle_e4m3_encode((double)prod);
    }
  }
  return rc;
}
