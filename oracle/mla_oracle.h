/*
 * mla_oracle.h -- float64 CPU oracle for MLA attention over an FP8-e4m3 latent KV cache.
 *
 * TEST INFRASTRUCTURE ONLY. This oracle is the correctness reference the tests and the
 * benchmark's CPU-baseline leg compare against. It shares no code, header, table or
 * constant with the CUDA library, and the library never calls it.
 *
 * What it computes (the plainest reading of the pages on MLA serving):
 *  - every cached position is one row of 576 e4m3 codes; K is the whole row, V its first
 *    512 entries ("MI355X Kimi K2.5 vLLM AITER 7x speedup", section "PR #35850 修复了什么":
 *    keys and values share one latent space; "Scaling Kimi K3 on AMD Instinct MI355X",
 *    section "缓存可复用，还要能一致地恢复": 576 FP8 bytes per position);
 *  - query j of the n_q new positions of sequence b sees cached keys n <= L_b - n_q + j
 *    (the new positions are already in the cache, causal among themselves);
 *  - partial results over key ranges combine through their log-sum-exp
 *    ("Scaling Kimi K3 ...", same section: partial attention merged by normalisation
 *    statistics).
 */
#ifndef MLA_ORACLE_H
#define MLA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Value of one OCP e4m3fn code (bias 7, 3 mantissa bits, no infinities, NaN = S.1111.111). */
double oracle_e4m3_value(uint8_t code);

/* Value of one bfloat16 bit pattern (the upper half of an IEEE binary32). */
double oracle_bf16_value(uint16_t bits);

/*
 * Full attention for every (sequence b, new position j, head h).
 *   pool        [num_pages][page_size][576] e4m3 codes
 *   page_table  [B][pt_stride] physical page of logical page p of sequence b
 *   seq_lens    [B] cached positions (including the n_q new ones)
 *   q_bf16      [B][n_q][H][576] bfloat16 bit patterns
 *   out         [B][n_q][H][512] float64
 *   lse         [B][n_q][H] float64, natural log of sum_n exp(score_n); -inf if no key visible
 * Returns 0, or -1 on a bad argument (a page index out of range, a negative length).
 */
int oracle_attention(const uint8_t* pool, int64_t num_pages, int page_size,
                     const int32_t* page_table, int64_t pt_stride, const int32_t* seq_lens,
                     double kv_scale, const uint16_t* q_bf16, int B, int n_q, int H,
                     double sm_scale, double* out, double* lse, int n_threads);

/*
 * The same attention for a list of rows only: row i is (rows_b[i], rows_j[i], rows_h[i]).
 * out [n_rows][512], lse [n_rows].
 */
int oracle_attention_rows(const uint8_t* pool, int64_t num_pages, int page_size,
                          const int32_t* page_table, int64_t pt_stride, const int32_t* seq_lens,
                          double kv_scale, const uint16_t* q_bf16, int B, int n_q, int H,
                          double sm_scale, const int32_t* rows_b, const int32_t* rows_j,
                          const int32_t* rows_h, int64_t n_rows, double* out, double* lse,
                          int n_threads);

/*
 * Attention of one query row over keys [key_lo, key_hi) of sequence b only (no causal
 * limit beyond the range itself): the partial result one split of the key axis holds.
 * out [512] (normalised over the range), *lse. An empty range gives out = 0, lse = -inf.
 */
int oracle_attention_range(const uint8_t* pool, int64_t num_pages, int page_size,
                           const int32_t* page_table, int64_t pt_stride, int b,
                           int64_t key_lo, int64_t key_hi, double kv_scale,
                           const uint16_t* q_row_bf16, double sm_scale, double* out, double* lse);

/*
 * Log-sum-exp merge of S partial results per row:
 *   lse = ln sum_s exp(lse_s),  out = sum_s exp(lse_s - lse) * out_s.
 * part_out [S][R][512], part_lse [S][R], out [R][512], lse [R]. Partials with
 * lse_s = -inf carry weight 0; a row whose partials are all -inf gets out = 0, lse = -inf.
 */
void oracle_merge_lse(const double* part_out, const double* part_lse, int S, int64_t R,
                      double* out, double* lse);

/*
 * e4m3fn code of the finite value nearest to v, ties to the code with the even mantissa
 * bit; |v| > 448 (and +-inf) saturate to +-448; the sign bit is v's (so -0 gives 0x80);
 * NaN gives 0x7F. Found by comparing v with the value of every finite code (the encoding
 * is the inverse of oracle_e4m3_value on the representable values).
 */
uint8_t oracle_e4m3_encode(double v);

/*
 * Append new latent rows to a paged FP8 cache: for each i < n with slots[i] >= 0,
 *   pool row slots[i] (byte offset slots[i] * 576) <- e4m3_encode(x_i[d] * inv), d < 576,
 * where inv = 1 / kv_scale and the product are both rounded to binary32 (round to nearest
 * even), x_i being the bfloat16 row i. Rows with a negative slot are skipped.
 * Returns 0, or -1 if a slot is not below pool_rows (nothing is written for that row).
 */
int oracle_cache_append(uint8_t* pool, int64_t pool_rows, const uint16_t* x_bf16,
                        const int64_t* slots, int64_t n, float kv_scale);

#ifdef __cplusplus
}
#endif
#endif
