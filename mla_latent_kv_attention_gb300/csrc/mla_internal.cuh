// mla_internal.cuh -- declarations shared by the translation units of libmla.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mla.h"

namespace mla {

constexpr int kD = MLA_D;
constexpr int kDV = MLA_DV;
constexpr int kKeyBlock = 128;     // keys per work block: the unit of split planning
// Split planning charges every sequence this many blocks' worth of time on top of its own
// blocks: a unit's epilogue and the refill of the pipeline after it. A CTA that takes a
// unit boundary gets correspondingly fewer blocks.
constexpr int kUnitCost = 5;
constexpr int kMaxRows = MLA_MAX_HEADS * MLA_MAX_NQ;  // query rows per sequence (64)

// Workspace header at offset 0 (256 bytes).
struct WsHeader {
  int num_ctas;      // CTAs of the last attention launch: status slots [0, num_ctas) are its
  int pad[63];
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Query rows one attention launch handles per unit (padded): 16, 32 or 48. More than 48
// rows per sequence run as two launches over halves of the heads.
inline int padded_rows(int rows_per_seq) {
  const int r = rows_per_seq > 48 ? (rows_per_seq + 1) / 2 : rows_per_seq;
  return r <= 16 ? 16 : (r <= 32 ? 32 : 48);
}

// One CTA's staged query image in global memory: the query operand of a later unit (two
// e4m3 terms of each padded row, in shared-memory layout) followed by the rows' score
// scales, copied into shared memory in one bulk copy when the unit starts.
inline size_t qimg_bytes(int rp) { return align_up((size_t)2 * rp * MLA_D + sizeof(float) * 48, 256); }

// Offsets of the workspace regions for one call.
//   status:   one word per CTA, written by that CTA at exit (0 or its first error)
//   qimg:     one staged query image per CTA
//   part_*:   two partial slots per CTA (the first and the last unit of its block range
//             are the only ones that can hold part of a sequence), R rows each
struct WsLayout {
  size_t hdr, status, qimg, part_lse, part_out, total;
  size_t qimg_stride;
  int max_slots;
};

inline WsLayout ws_layout(int B, int rows_per_seq, int num_sms) {
  WsLayout w;
  w.max_slots = 2 * num_sms;
  w.qimg_stride = qimg_bytes(padded_rows(rows_per_seq));
  size_t off = 0;
  w.hdr = off;
  off += sizeof(WsHeader);
  w.status = off = align_up(off, 256);
  off += sizeof(unsigned) * (size_t)num_sms;
  w.qimg = off = align_up(off, 256);
  off += w.qimg_stride * (size_t)num_sms;
  w.part_lse = off = align_up(off, 256);
  off += sizeof(float) * (size_t)w.max_slots * rows_per_seq;
  w.part_out = off = align_up(off, 256);
  off += sizeof(float) * (size_t)w.max_slots * rows_per_seq * kDV;
  w.total = align_up(off, 256);
  return w;
}

// Prefill: the header, the per-CTA status words, the per-CTA query images (48 rows), and
// the partials of the units of the last round that are split in two along the keys: one
// slot per CTA, 48 rows each (float32 LSE, then float32 outputs).
inline size_t ws_prefill_status(int) { return align_up(sizeof(WsHeader), 256); }
inline size_t ws_prefill_qimg(int num_sms) {
  return align_up(ws_prefill_status(num_sms) + sizeof(unsigned) * (size_t)num_sms, 256);
}
inline size_t ws_prefill_part_lse(int num_sms) {
  return align_up(ws_prefill_qimg(num_sms) + qimg_bytes(48) * (size_t)num_sms, 256);
}
inline size_t ws_prefill_part_out(int num_sms) {
  return align_up(ws_prefill_part_lse(num_sms) + sizeof(float) * 48 * (size_t)num_sms, 256);
}
inline size_t ws_prefill_bytes(int num_sms) {
  return align_up(ws_prefill_part_out(num_sms) + sizeof(float) * 48 * kDV * (size_t)num_sms, 256);
}

// Everything an attention kernel needs for one call.
struct AttnParams {
  const uint8_t* pool;
  int64_t num_pages;
  int page_size;
  const int32_t* page_table;
  int64_t pt_stride;
  const int32_t* seq_lens;
  float kv_scale;
  float sm_scale;
  const uint16_t* q;  // [B][n_q][H][576]
  int B, n_q, H, R;   // R = n_q * H rows per sequence
  uint16_t* out;      // [B][n_q][H][512] bf16
  float* out_f32;     // when set, the output goes here as float32 instead of to `out`
  float* lse;         // [B][n_q][H] or null
  float* part_out;    // [slots][part_rows][512]
  float* part_lse;    // [slots][part_rows]
  int part_rows;      // rows of a partial slot: R (decode/verify), 48 (prefill)
  unsigned* status;   // [num_ctas]
  uint8_t* qimg;      // [num_ctas] staged query images, qimg_stride bytes apart
  int64_t qimg_stride;
  WsHeader* hdr;
  int num_ctas;
  int test_stall;     // test hook: the producer issues no loads, so every consumer's bounded
                      // wait runs out and the call reports MLA_ERR_TIMEOUT
  int mask_shift;     // key n visible to new position j iff n <= L - n_q + j + mask_shift
  unsigned long long* trace;  // profiling hook: kTraceWords globaltimer stamps per CTA, or null
  int trace_ctas;             // CTAs the trace buffer has room for
};

// Per-CTA stamps of the profiling hook (mla_set_trace_buffer), in nanoseconds of the GPU's
// global timer: entry, end of the wait on the previous kernel, end of the split plan (with
// the first tile loads issued), the first tile's scores read by the softmax, the last tile's
// probabilities written, the last values MMA done, end of the last epilogue, exit; the
// tiles and units the CTA processed; end of the first unit's epilogue and the second unit's
// first scores (CTAs with two units or more); decode/verify: end of the plan's scan, end of
// its L2 prefetches.
constexpr int kTraceWords = 16;
enum TraceSlot { kTrEntry = 0, kTrWaited, kTrPlanned, kTrFirstScores, kTrLastP, kTrLastPV,
                 kTrEpilogue, kTrExit, kTrCounts, kTrUnit1End, kTrUnit2Scores, kTrPlanScan,
                 kTrPlanPrefetch };

// The split plan's cost axis: all sequences laid end to end, each as kUnitCost units of
// fixed cost followed by its 128-key blocks (an empty sequence takes no room); CTA c owns
// the positions [c * total / n, (c + 1) * total / n). range_of(x): the CTA that holds
// position x, the largest c whose range starts at or before x.
__host__ __device__ __forceinline__ int64_t range_lo(int64_t c, int64_t total, int64_t n) {
  return c * total / n;
}
__host__ __device__ __forceinline__ int64_t range_of(int64_t x, int64_t total, int64_t n) {
  return ((x + 1) * n + total - 1) / total - 1;
}

// Up-projected 16-bit columns per head in kvup: bf16 form 128 key + 128 value columns;
// precise form 128 key (hi) + 128 key (lo) + 128 value columns.
inline __host__ __device__ int mha_up_width(bool precise) { return precise ? 384 : 256; }

// MHA-form prefill workspace: header, status words (one per attention CTA, then one for the
// dequantisation), the dequantised latent [L][512] bf16, the RoPE rows [L][64] bf16, the
// up-projected keys and values [L][H][384] 16-bit (room for the precise form's hi, lo and
// value columns; the bf16 form uses the first 256 columns' worth of each row), and the
// partials of units split along the key axis: one slot per pair of CTAs, each
// [2][128][128] float32 outputs and [2][128] float32 LSE.
struct MhaWsLayout {
  size_t status, latent, rope, kvup, part_out, part_lse, total;
};
inline MhaWsLayout mha_ws_layout(int64_t L, int H, int num_sms) {
  MhaWsLayout w;
  size_t off = align_up(sizeof(WsHeader), 256);
  w.status = off;
  off = align_up(off + sizeof(unsigned) * (size_t)(num_sms + 1), 256);
  w.latent = off;
  off = align_up(off + (size_t)L * kDV * 2, 256);
  w.rope = off;
  off = align_up(off + (size_t)L * 64 * 2, 256);
  w.kvup = off;
  off = align_up(off + (size_t)L * H * mha_up_width(true) * 2, 256);
  const size_t slots = (size_t)(num_sms / 2 + 1);
  w.part_out = off;
  off = align_up(off + slots * 2 * 128 * 128 * sizeof(float), 256);
  w.part_lse = off;
  off = align_up(off + slots * 2 * 128 * sizeof(float), 256);
  w.total = off;
  return w;
}

struct MhaArgs {
  const uint8_t* pool;
  int64_t num_pages;
  int page_size;
  const int32_t* page_table;
  float kv_scale;
  int L, T, H;
  float sm_scale;
  const void* q;      // [T][H][192] bf16
  const void* w_ukv;  // [512][H][256] bf16
  void* latent;
  void* rope;
  void* kvup;
  void* part_out;     // partials of split units (see MhaWsLayout)
  void* part_lse;
  uint16_t* out;      // [T][H][128] bf16
  float* lse;         // [T][H] or null
  unsigned* status;   // [num attention CTAs + 1]
  WsHeader* hdr;
  int device;
  int precise;        // 1: keys as bf16 hi + lo pairs, fp16 values and probabilities
  cudaEvent_t prof_start, prof_stop;  // recorded around the attention kernel when both set
};

// Launchers (each returns the CUDA error of its launch).
cudaError_t launch_merge(const AttnParams& p, cudaStream_t s);
cudaError_t launch_decode_tc(const AttnParams& p, int num_sms, cudaStream_t s, int* launches);
cudaError_t launch_prefill_tc(const AttnParams& p, int num_sms, cudaStream_t s, int* launches);
cudaError_t launch_merge_prefill(const AttnParams& p, int P, int split_units, cudaStream_t s);
cudaError_t launch_merge_standalone(const float* part_out, const float* part_lse, int S, int64_t R,
                                    uint16_t* out, float* lse, int num_sms, cudaStream_t s);
cudaError_t launch_cache_append(uint8_t* pool, int64_t pool_rows, const uint16_t* x,
                                const int64_t* slots, int64_t n, float inv, unsigned* status,
                                int num_sms, cudaStream_t s);
cudaError_t launch_mha_prefill(const MhaArgs& a, int num_sms, cudaStream_t s, int* launches);
cudaError_t launch_mha_projection(const void* latent, const void* w, void* kvup, int L, int H,
                                  float kv_scale, int precise, unsigned* status, cudaStream_t s);
cudaError_t launch_top_k_renorm(const float* probs, float* out, int B, int V, const int32_t* top_k,
                                int k_all, cudaStream_t s);

}  // namespace mla
