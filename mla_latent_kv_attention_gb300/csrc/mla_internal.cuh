// mla_internal.cuh -- declarations shared by the translation units of libmla.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/mla.h"

namespace mla {

constexpr int kD = MLA_D;
constexpr int kDV = MLA_DV;
constexpr int kKeyBlock = 128;     // keys per work block: the unit of split planning
constexpr int kMaxRows = MLA_MAX_HEADS * MLA_MAX_NQ;  // query rows per sequence (64)

// Workspace header at offset 0 (256 bytes).
struct WsHeader {
  unsigned int status;   // mla_status_t written by the device (first error wins)
  int num_units;         // units the planner produced
  int blocks_per_unit;   // key blocks (of kKeyBlock keys) per unit
  int pad[61];
};

// One unit of split-KV work: keys [key_lo, key_hi) of sequence b.
struct Unit {
  int b, key_lo, key_hi, slot;
};

// Per-sequence unit range.
struct SeqUnits {
  int first, count;
};

// Offsets of the workspace regions for one decode/verify call.
struct WsLayout {
  size_t hdr, units, seqs, cta_first, blk_prefix, part_lse, part_out, total;
  int max_units, max_ctas;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline WsLayout ws_layout(int B, int rows_per_seq, int num_sms) {
  WsLayout w;
  // one contiguous block range per CTA, split only where a sequence ends: at most
  // (CTAs + B - 1) pieces
  w.max_ctas = num_sms;
  w.max_units = num_sms + B;
  size_t off = 0;
  w.hdr = off;
  off += sizeof(WsHeader);
  w.units = off = align_up(off, 256);
  off += sizeof(Unit) * (size_t)w.max_units;
  w.seqs = off = align_up(off, 256);
  off += sizeof(SeqUnits) * (size_t)(B > 0 ? B : 1);
  w.cta_first = off = align_up(off, 256);
  off += sizeof(int) * (size_t)(num_sms + 1);
  w.blk_prefix = off = align_up(off, 256);
  off += sizeof(int) * (size_t)(B + 1);
  w.part_lse = off = align_up(off, 256);
  off += sizeof(float) * (size_t)w.max_units * rows_per_seq;
  w.part_out = off = align_up(off, 256);
  off += sizeof(float) * (size_t)w.max_units * rows_per_seq * kDV;
  w.total = align_up(off, 256);
  return w;
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
  uint16_t* out;      // [B][n_q][H][512]
  float* lse;         // [B][n_q][H] or null
  float* part_out;    // [max_units][R][512]
  float* part_lse;    // [max_units][R]
  Unit* units;
  SeqUnits* seqs;
  int* cta_first;   // [num_ctas + 1]: CTA c owns units [cta_first[c], cta_first[c + 1])
  int* blk_prefix;  // [B + 1]: first 128-key block of each sequence in the flat block order
  WsHeader* hdr;
  int max_units;
  int num_ctas;
};

__device__ __forceinline__ void report(WsHeader* hdr, mla_status_t code) {
  atomicCAS(&hdr->status, 0u, (unsigned)code);
}

// Launchers (each returns the CUDA error of its launch).
cudaError_t launch_plan(const AttnParams& p, cudaStream_t s);
cudaError_t launch_merge(const AttnParams& p, cudaStream_t s);
cudaError_t launch_decode_tc(const AttnParams& p, int num_sms, cudaStream_t s, int* launches);
cudaError_t launch_prefill_tc(const AttnParams& p, int num_sms, cudaStream_t s, int* launches);
cudaError_t launch_merge_standalone(const float* part_out, const float* part_lse, int S, int64_t R,
                                    uint16_t* out, float* lse, cudaStream_t s);
cudaError_t launch_reset_status(WsHeader* hdr, cudaStream_t s);

}  // namespace mla
