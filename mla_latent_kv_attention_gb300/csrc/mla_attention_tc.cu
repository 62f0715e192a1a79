// mla_attention_tc.cu -- MLA attention on tcgen05 tensor cores: split-KV decode, speculative
// verify and causal prefill over the paged FP8 latent cache.
//
// Work: one persistent CTA per SM walks the planner's units (keys [key_lo, key_hi) of one
// sequence, all of its query rows). Keys stream through shared memory 128 at a time
// (two 64-position pages, fetched by TMA straight from the paged pool) and every key is
// read from HBM exactly once per unit, whatever the head count or verify depth.
//
// Both contractions run on the FP8 cache bytes as they are, with no dequantisation pass:
//   scores  S^T[key][n] = sum_d code[key][d] * Qt[n][d]      tcgen05 kind::f8f6f4,
//           M = 128 keys, N = 2 x (padded rows), K = 576
//           The bf16 query row, scaled by the power of two that puts its largest
//           magnitude in (224, 448], is split into two e4m3 terms stacked along N: the
//           first is the entry rounded to e4m3, the second the residual times 16 rounded
//           to e4m3 (the residual is at most 16, so this never saturates), and the two
//           accumulators are summed as S1 + S2 / 16. The split is exact for every entry of
//           at least 2^-14.8 of the row's largest magnitude (bf16 has 8 significant bits,
//           e4m3 4, and the scaled residual is a multiple of e4m3's subnormal step there);
//           a smaller entry is carried to within 2^-21.8 of the row's largest magnitude.
//   values  O^T[dv][n]  += sum_key code[key][dv] * Pt[n][key] tcgen05 kind::f8f6f4,
//           M = 128 dv (x4 chunks), N = rows, K = keys; the same FP8 tile read MN-major
//           (A: e4m3 codes) against the probabilities as three e5m2 terms (B). A weight
//           p = 2^(x - m + 11) (at most 2^15) is rounded to fp16 and split by round to
//           nearest into e5m2 terms t0 + t1 + t2: each term takes the leading 3 bits of
//           what the previous ones left, so the sum carries p to about fp16's precision,
//           and e5m2's range (2^-16 .. 57344) keeps that precision for weights down to
//           about 2^-19 of the running maximum. Smaller weights lose bits gradually; the
//           smallest one kept is 2^-28 of the maximum. (An e4m3 split loses every weight
//           below about 2^-14 of the maximum: a long tail under a dominant key would then
//           vanish from the numerator but not from the row sum.)
// Keys sit on the MMA's M side ("swap A/B"): 8-16 heads x 1-4 positions are far below
// M = 128, so the few query rows take the narrow N side and nothing is padded in memory.
// Softmax is online over key tiles; one warpgroup owns one key per thread (its TMEM
// lane), so the running max per row needs a cross-warp reduction each tile.
//
// Roles: warp 0 issues TMA, warp 1 owns TMEM and issues the score MMAs, warp 3 issues the
// value MMAs, warp 2 stages query rows, and from warp 4 on two warpgroups (three with 48
// rows per unit: 384 or 512 threads) run the softmax and write the epilogue. Every wait is
// bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math.h>
#include <stddef.h>

#include "mla_internal.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kTileKeys = 128;
constexpr int kStages = 2;
constexpr int kChunkBytes = 16384;                     // 128 keys x 128 bytes, SW128
constexpr int kStageBytes = 4 * kChunkBytes + 2 * 4096;  // 73,728 bytes loaded per tile
// A stage is filled and freed in two halves: latent chunks 0-1, then chunks 2-3 with the
// RoPE tail. The values MMA frees the first half as soon as its own MMAs complete, so the
// next tile's first half loads while the second is still being read. (Every
// tcgen05.commit costs the issuing thread time: measured, five parts ran slower than one,
// two fastest.)
constexpr int kParts = 2;
__host__ __device__ constexpr int part_of_chunk(int c) { return c / 2; }
constexpr int kTailPart = 1;
__host__ __device__ constexpr int part_bytes(int part) {
  return part == 0 ? 2 * kChunkBytes : 2 * kChunkBytes + 2 * 4096;
}
static_assert(part_bytes(0) + part_bytes(1) == kStageBytes, "the halves make up the stage");
constexpr int kMaxThreads = 512;  // producer, 2 MMA issuers, query stager, 2-3 softmax warpgroups
constexpr int kSoftmaxWarp0 = 4;
constexpr uint64_t kWaitLimitNs = 1000000000ull;        // 1 s
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kPScale = 11.0f;     // P carried as 2^(x - m + 11): at most 2^15 while x <= m + 4
constexpr float kRescaleGap = 4.0f;  // the running max (log2 units) moves only past m + 4
constexpr float kQTerm2 = 16.0f;     // the second query term carries the residual times 16
constexpr float kNoMax = -1e30f;     // running max (less kPScale) of a row that has seen no key
constexpr int kPrefetchTiles = 1;    // tiles the producer pulls into L2 ahead of its TMA loads

template <int RP>
struct Cfg {
  // softmax warpgroups: three at 48 rows (16 rows per thread), else two
  static constexpr int kNWG = (RP == 48) ? 3 : 2;
  static constexpr int kThreads = 128 + 128 * kNWG;
  static constexpr int kRH = RP / kNWG;                // query rows per softmax thread
  static constexpr int kStageWarps = kThreads / 32 - 2;  // warps 2.. stage the first units
  static constexpr int NQK = 2 * RP;                    // two query terms per row
  // S^T buffers: two (the next tile's scores land while the softmax works on this one),
  // one at 48 rows, where TMEM is needed for stacked O chunks
  static constexpr int kSBuf = (RP == 48) ? 1 : 2;
  // O^T chunk c (128 dv lanes) holds the three P terms' products side by side ("stacked":
  // one N = 3 RP MMA per k-step, the V^T tile read once) or summed in one accumulator
  // (three N = RP MMAs per k-step, V^T read three times). Stacked everywhere up to 32
  // rows; at 48 rows TMEM holds two stacked chunks and two summed ones.
  static constexpr int kStackedChunks = (RP == 48) ? 2 : 4;
  static constexpr __host__ __device__ int oterms(int c) { return c < kStackedChunks ? 3 : 1; }
  static constexpr int kSCol = 0;                       // S^T buffers: [0, kSBuf NQK)
  static constexpr int kOCol = kSBuf * NQK;             // O^T chunks from here
  static constexpr __host__ __device__ int ocol(int c) {
    return kOCol + (c < kStackedChunks ? c * 3 * RP : kStackedChunks * 3 * RP + (c - kStackedChunks) * RP);
  }
  static constexpr int kTmemUsed = ocol(3) + oterms(3) * RP;
  static constexpr int kTmemCols = kTmemUsed <= 256 ? 256 : 512;
  static constexpr int kQBytes = NQK * kD;
  // query operand buffers: two (the next unit is staged during this one) when they fit
  static constexpr int kQB = (RP == 16) ? 2 : 1;
  // A stage holds one key tile: dims 0..511 as four SW128 chunks of 128 keys x 128 bytes,
  // then dims 512..575 (the tail, SW64, 128 keys x 64 bytes). At 48 rows each stage also
  // holds its tile's probabilities (P^T, three e5m2 terms of 6 KB), so the softmax can
  // write the next tile's P while the values MMA still reads this one: terms 1 and 2 in
  // 12 KB between the chunks and the tail, term 0 over the first 6 KB of the tail, which
  // the scores no longer need by then. Otherwise one P buffer serves every tile.
  static constexpr bool kPInStage = (RP == 48);
  // dv-chunk loops of the epilogue and the rescale: rolled up at 16 rows (measured: smaller
  // code, a faster decode), unrolled at 32 and 48 (rolled, they spill)
  static constexpr int kUnrollChunks = (RP == 16) ? 1 : 4;
  static constexpr int kPTerm = (RP / 16) * 2048;       // one term: RP/16 groups of 16 rows
  static constexpr int kTail = 4 * kChunkBytes + (kPInStage ? 2 * kPTerm : 0);
  static constexpr int kStageStride = kTail + 2 * 4096;
  static constexpr int kPBytes = kPInStage ? 0 : 3 * kPTerm;
  // offset of P term t from the P base (the stage's P area, or the shared buffer)
  static constexpr __host__ __device__ int pterm(int t) {
    return kPInStage ? ((t + 2) % 3) * kPTerm : t * kPTerm;
  }
  // shared memory layout (offsets from a 1024-aligned base)
  static constexpr int kOffStages = 0;
  static constexpr int kOffP = kStages * kStageStride;
  static constexpr int kOffQ = kOffP + ((kPBytes + 1023) / 1024) * 1024;
  static constexpr int kOffMisc = kOffQ + kQB * kQBytes;
  static_assert(kTmemUsed <= 512, "TMEM budget");
  static_assert(kOffMisc % 16 == 0 && kOffQ % 1024 == 0 && kOffP % 1024 == 0 &&
                    kQBytes % 1024 == 0, "alignment");
};

struct Misc {
  // float arrays first: they are read as float4 and must be 16-byte aligned
  alignas(16) float row_scale[2][48];  // by unit parity
  alignas(16) float red[2][48 * 4];  // per-tile warp maxima, [row][warp]
  alignas(16) float lred[4][48];
  alignas(16) float alpha[48];       // this tile's rescale factors (each warp of a
                                     // warpgroup writes the same values for its rows)
  alignas(16) int grow[2][12];       // per tile parity and warp: some row's max moves
  alignas(16) int row_j[48];         // new-position index j of each row (very negative for padding)
  alignas(16) int row_off[48];       // j * H + h: the row's index among its sequence's rows
  alignas(8) uint64_t kv_full[kStages][kParts];  // part landed (TMA transaction bytes)
  uint64_t kv_free[kStages][kParts];             // part no longer read by any MMA
  uint64_t s_full[2], s_empty[2];
  uint64_t p_full[2];   // P of tile g is written: p_full[g % 2] (the softmax may run a tile
                        // ahead of the value MMAs when P lives in the stage)
  uint64_t q_full[2];   // query operand buffer holds its unit's terms
  uint64_t q_empty[2];  // the unit that used the buffer has finished its scores
  uint64_t q0_done;     // the first unit's query rows are staged (by warps 2.. together)
  uint64_t q1_done;     // the second unit's rows are in this CTA's global query image
  uint64_t wg_bar[3];  // bounded barriers of the softmax warpgroups (128 arrivals)
  // decode/verify split plan of this CTA: positions [x0, x1) of the cost axis (all
  // sequences end to end, each as kUnitCost fixed units then its blocks); its first unit
  // is sequence b0 (length L0), whose first block sits at pre0
  long long plan_x0, plan_x1, plan_pre0;
  int plan_b0, plan_L0;
  int scan[kMaxThreads / 32];
  uint32_t tmem_base;
  int abort;
  unsigned status;  // this CTA's first error
};
static_assert(offsetof(Misc, row_scale) % 16 == 0 && offsetof(Misc, red) % 16 == 0 &&
                  offsetof(Misc, lred) % 16 == 0 && offsetof(Misc, alpha) % 16 == 0 &&
                  offsetof(Misc, grow) % 16 == 0,
              "vector-accessed arrays must be 16-byte aligned");
static_assert(offsetof(Misc, kv_full) % 8 == 0, "mbarriers must be 8-byte aligned");

template <int RP>
constexpr int smem_bytes() {
  return Cfg<RP>::kOffMisc + (int)sizeof(Misc) + 1024;
}
static_assert(smem_bytes<16>() <= 232448 && smem_bytes<32>() <= 232448 && smem_bytes<48>() <= 232448,
              "dynamic shared memory per CTA");

struct DecodeArgs {
  AttnParams p;
  int h0, Hs;  // heads [h0, h0 + Hs) handled by this launch
  int rows;    // rows per unit: n_q * Hs (decode/verify) or P * H (prefill), <= RP
  int prefill;    // 1: units are blocks of P new positions of one sequence (no split plan)
  int P;          // prefill: new positions per unit
  int num_units;  // prefill: ceil(n_q / P)
  int unit_end;   // prefill: this launch's units are [blockIdx.x, unit_end) in steps of the grid
  int split_base;  // prefill: units [split_base, num_units) run as two halves each
  int status_overwrite;  // 1: each CTA writes its status word even when clean (first launch)
};

// One unit of work as every role of the kernel sees it.
struct UnitInfo {
  int b, key_lo, key_hi;
  int L;          // cached positions of sequence b
  int qrow0;      // global row (of q, out, lse) of the unit's row 0
  int j0;         // new-position index of the unit's first position
  int rows;       // valid rows of the unit
  int final_out;  // 1: bf16 out + lse directly; 0: normalised partial for the merge
  int slot;       // partial slot (when final_out == 0)
};

// Position in this CTA's list of units. Decode/verify: the sequences whose blocks overlap
// the CTA's range, in order (b, the cost-axis position pre of its first block, its length
// L). Prefill: unit index u.
struct Cursor {
  int u;
  int b;
  long long pre;
  int L;
};

__device__ __forceinline__ int seq_len_of(const AttnParams& p, int b) {
  int L = p.seq_lens[b];
  const int64_t cap = p.pt_stride * (int64_t)p.page_size;
  if (L < 0) return 0;
  if ((int64_t)L > cap) return (int)cap;
  return L;
}

__device__ __forceinline__ int blocks_of(int L) { return (L + kKeyBlock - 1) / kKeyBlock; }

// A final output element: bf16, or float32 when the caller asked for it.
__device__ __forceinline__ void store_out(const AttnParams& p, int64_t idx, float v) {
  if (p.out_f32)
    p.out_f32[idx] = v;
  else
    p.out[idx] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// PF: 0 decode/verify (the split plan's units); 1 prefill (units are blocks of new
// positions, one a round per CTA); 2 prefill, the two halves along the keys of each unit of
// an incomplete last round (one half a CTA, a partial for the merge). A compile-time
// parameter: each kernel carries only its own paths.
template <int PF>
__device__ __forceinline__ Cursor first_unit(const DecodeArgs& a, const Misc* ms) {
  Cursor c;
  c.u = blockIdx.x;
  c.b = ms->plan_b0;
  c.pre = ms->plan_pre0;
  c.L = ms->plan_L0;
  return c;
}

template <int PF>
__device__ __forceinline__ bool has_unit(const DecodeArgs& a, const Misc* ms, const Cursor& c) {
  return PF ? c.u < a.unit_end : (c.b < a.p.B && c.pre < ms->plan_x1);
}

// The next unit: the next sequence with at least one key (decode/verify), or the next
// unit index this CTA owns (prefill).
template <int PF>
__device__ __forceinline__ Cursor next_unit(const DecodeArgs& a, Cursor c) {
  if (PF) {
    c.u += gridDim.x;
    return c;
  }
  c.pre += blocks_of(c.L);
  do {
    ++c.b;
    c.L = (c.b < a.p.B) ? seq_len_of(a.p, c.b) : 0;
  } while (c.b < a.p.B && c.L == 0);
  c.pre += kUnitCost;  // the next sequence's fixed cost precedes its blocks
  return c;
}

template <int PF>
__device__ __forceinline__ UnitInfo unit_info(const DecodeArgs& a, const Misc* ms, const Cursor& c) {
  const AttnParams& p = a.p;
  UnitInfo x;
  if (!PF) {
    const long long nb = blocks_of(c.L);
    const long long blo = max(ms->plan_x0, c.pre), bhi = min(ms->plan_x1, c.pre + nb);
    x.b = c.b;
    x.L = c.L;
    x.key_lo = (int)(blo - c.pre) * kKeyBlock;
    x.key_hi = (bhi > blo) ? min(c.L, (int)(bhi - c.pre) * kKeyBlock) : x.key_lo;
    x.qrow0 = c.b * p.R;
    x.j0 = 0;
    x.rows = a.rows;
    x.final_out = (blo == c.pre && bhi == c.pre + nb);
    // the CTA's first unit (nothing of an earlier sequence in its range) takes slot 2c
    x.slot = 2 * (int)blockIdx.x + (c.pre - kUnitCost <= ms->plan_x0 ? 0 : 1);
  } else {
    // the last positions see the most keys: hand those out first
    int v = c.u;
    if constexpr (PF == 2) v = a.split_base + c.u / 2;  // unit v, half c.u & 1
    const int pos0 = (a.num_units - 1 - v) * a.P;
    const int npos = min(a.P, p.n_q - pos0);
    const int L = seq_len_of(p, 0);
    x.b = 0;
    x.L = L;
    x.key_lo = 0;
    x.key_hi = max(0, min(L, L - p.n_q + pos0 + npos));  // last key the unit's last position sees, + 1
    x.qrow0 = pos0 * p.H;
    x.j0 = pos0;
    x.rows = npos * p.H;
    x.final_out = 1;
    x.slot = 0;
    if constexpr (PF == 2) {  // keys [0, mid) or [mid, key_hi), partial slot c.u
      const int mid = min(x.key_hi, ((x.key_hi + 2 * kTileKeys - 1) / (2 * kTileKeys)) * kTileKeys);
      if (c.u & 1)
        x.key_lo = mid;
      else
        x.key_hi = mid;
      x.final_out = 0;
      x.slot = c.u;
    }
  }
  return x;
}

__device__ __forceinline__ int tiles_in(const UnitInfo& x) {
  return (x.key_hi - x.key_lo + kTileKeys - 1) / kTileKeys;
}

// First error of this CTA wins; the CTA writes it to its status word at exit.
__device__ __forceinline__ void report(Misc* m, mla_status_t code) {
  atomicCAS(&m->status, 0u, (unsigned)code);
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Misc* m,
                                              const AttnParams& p) {
  if (mbar_wait(bar, parity, kWaitLimitNs)) return true;
  m->abort = 1;
  report(m, MLA_ERR_TIMEOUT);
  return false;
}

__device__ __forceinline__ bool aborted(const Misc* m) {
  return *reinterpret_cast<const volatile int*>(&m->abort) != 0;
}

// fp8 e4m3 helpers (round to nearest even, saturating; and exact back-conversion)
__device__ __forceinline__ uint16_t to_e4m3x2(float lo, float hi) {
  return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}
__device__ __forceinline__ float2 from_e4m3x2(uint16_t v) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)v, __NV_E4M3);
  return __half22float2(*reinterpret_cast<__half2*>(&h));
}

__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// (lo, hi) -> f16x2 with lo in the low half
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi) {
  uint32_t h;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(hi), "f"(lo));
  return h;
}
__device__ __forceinline__ uint32_t f16x2_to_e5m2x2(uint32_t h) {
  uint16_t c;
  asm("cvt.rn.satfinite.e5m2x2.f16x2 %0, %1;" : "=h"(c) : "r"(h));
  return c;
}
__device__ __forceinline__ uint32_t e5m2x2_to_f16x2(uint32_t c) {
  uint32_t h;
  asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(h) : "h"((uint16_t)c));
  return h;
}
__device__ __forceinline__ uint32_t hsub2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Byte offset of the 16-byte group `w16` (16 codes, dims 16*w16 .. +15) of term-row n
// inside the query operand (K-major: four SW128 chunks of 128 dims, then one SW64 chunk).
template <int NQK>
__device__ __forceinline__ int q_offset(int n, int w16) {
  if (w16 < 32) {
    const int c = w16 >> 3, w = w16 & 7;
    return c * (NQK * 128) + (n >> 3) * 1024 + (n & 7) * 128 + ((w ^ (n & 7)) << 4);
  }
  const int w = w16 - 32;
  return 4 * (NQK * 128) + (n >> 3) * 512 + (n & 7) * 64 + (((w ^ ((n & 7) >> 1)) & 3) << 4);
}

// Stage rows w, w + nw, ... (< RP) of one unit's queries into a query operand buffer as two
// e4m3 terms after a per-row power-of-two scale (the entry rounded, then 16 x the residual
// rounded: exact for entries down to 2^-14.8 of the row's largest magnitude, within
// 2^-21.8 of it below), and the rows' score scales into row_scale[]. Rows at or past R are
// written as zeros.
template <int RP, int NW>
__device__ __forceinline__ void stage_rows(const AttnParams& p, int R, const int* row_off,
                                       const uint16_t* qseq, uint8_t* qdst, float* row_scale,
                                       int w0, int lane) {
  using C = Cfg<RP>;
  const float kv_scale = p.kv_scale;
  constexpr int nw = NW;  // warps staging together
  // rows of one pass of a warp (at most four; no more than NW warps leave for it)
  constexpr int K2 = (RP + NW - 1) / NW < 4 ? (RP + NW - 1) / NW : 4;
  // rows r0, r0 + nw, ... of this warp: all loads first, then the arithmetic
  for (int r0 = w0; r0 < RP; r0 += K2 * nw) {
    uint4 ld[K2][2], tl[K2][2];
#pragma unroll
    for (int k2 = 0; k2 < K2; ++k2) {
      const int r = r0 + nw * k2;
      ld[k2][0] = ld[k2][1] = tl[k2][0] = tl[k2][1] = make_uint4(0, 0, 0, 0);
      if (r < R) {
        const uint4* s4 = reinterpret_cast<const uint4*>(qseq + (int64_t)row_off[r] * kD);
        ld[k2][0] = s4[2 * lane];
        ld[k2][1] = s4[2 * lane + 1];
        if (lane < 4) {  // dims 512 + 16*lane .. +15 (1024 bytes in: 64 uint4)
          tl[k2][0] = s4[64 + 2 * lane];
          tl[k2][1] = s4[64 + 2 * lane + 1];
        }
      }
    }
#pragma unroll
    for (int k2 = 0; k2 < K2; ++k2) {
      const int r = r0 + nw * k2;
      if (r >= RP) break;
      const bool real = r < R;
      float v[16], tail[16];
      {
        const uint32_t w[8] = {ld[k2][0].x, ld[k2][0].y, ld[k2][0].z, ld[k2][0].w,
                               ld[k2][1].x, ld[k2][1].y, ld[k2][1].z, ld[k2][1].w};
        const uint32_t wt[8] = {tl[k2][0].x, tl[k2][0].y, tl[k2][0].z, tl[k2][0].w,
                                tl[k2][1].x, tl[k2][1].y, tl[k2][1].z, tl[k2][1].w};
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          v[e] = __uint_as_float((w[e >> 1] >> ((e & 1) * 16)) << 16);
          tail[e] = __uint_as_float((wt[e >> 1] >> ((e & 1) * 16)) << 16);
        }
      }
      float amax = 0.f;
#pragma unroll
      for (int e = 0; e < 16; ++e) amax = fmaxf(amax, fmaxf(fabsf(v[e]), fabsf(tail[e])));
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      // scale 2^ex so that amax * 2^ex lies in (224, 448]; from the exponent field of
      // amax (normal floats: biased exponent E means amax in [2^(E-127), 2^(E-126)))
      int ex = 0;
      if (amax >= 1.17549435e-38f && amax <= 3.4e38f) {
        const int E = (__float_as_int(amax) >> 23) & 0xFF;
        ex = 135 - E;  // amax * 2^ex in [256, 512)
        if (amax * __int_as_float((127 + ex) << 23) > 448.f) ex -= 1;
        ex = max(-126, min(126, ex));  // both 2^ex and 2^-ex stay normal floats
      }
      const float up = __int_as_float((127 + ex) << 23);    // 2^ex, exact
      const float down = __int_as_float((127 - ex) << 23);  // 2^-ex, exact
      if (lane == 0) row_scale[r] = real ? p.sm_scale * kv_scale * down * kLog2e : 0.f;
      // two terms per value, packed 16 codes per 16-byte group
      auto emit = [&](const float* x, int w16) {
        uint32_t t1w[4], t2w[4];
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          const float a0 = x[e] * up, a1 = x[e + 1] * up;
          const uint16_t c1 = to_e4m3x2(a0, a1);
          const float2 b1 = from_e4m3x2(c1);
          const uint16_t c2 = to_e4m3x2((a0 - b1.x) * kQTerm2, (a1 - b1.y) * kQTerm2);
          const int wi = e >> 2, sh = (e & 2) * 8;
          if ((e & 2) == 0) {
            t1w[wi] = c1;
            t2w[wi] = c2;
          } else {
            t1w[wi] |= (uint32_t)c1 << sh;
            t2w[wi] |= (uint32_t)c2 << sh;
          }
        }
        *reinterpret_cast<uint4*>(qdst + q_offset<C::NQK>(r, w16)) = make_uint4(t1w[0], t1w[1], t1w[2], t1w[3]);
        *reinterpret_cast<uint4*>(qdst + q_offset<C::NQK>(RP + r, w16)) = make_uint4(t2w[0], t2w[1], t2w[2], t2w[3]);
      };
      emit(v, lane);
      if (lane < 4) emit(tail, 32 + lane);
    }
  }
}

template <int RP, int PF, bool TR>
__global__ void __launch_bounds__(Cfg<RP>::kThreads, 1)
    attn_tc_kernel(const __grid_constant__ DecodeArgs args,
                     const __grid_constant__ CUtensorMap map_main,
                     const __grid_constant__ CUtensorMap map_tail) {
  using C = Cfg<RP>;
  const AttnParams& p = args.p;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Misc* ms = reinterpret_cast<Misc*>(smem + C::kOffMisc);
  uint8_t* pbuf = smem + C::kOffP;
  uint8_t* qbuf = smem + C::kOffQ;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // profiling hook: this CTA's stamps, or null
  // (TR: a separate instantiation for traced calls, so the usual one carries no stamp code)
  unsigned long long* const trace = (TR && p.trace && (int)blockIdx.x < p.trace_ctas)
                                        ? p.trace + (size_t)blockIdx.x * kTraceWords
                                        : nullptr;
  if (trace && threadIdx.x == 0) trace[kTrEntry] = globaltimer_ns();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s)
      for (int c = 0; c < kParts; ++c) {
        mbar_init(&ms->kv_full[s][c], 1);
        mbar_init(&ms->kv_free[s][c], 1);
      }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ms->s_full[s], 1);
      mbar_init(&ms->s_empty[s], 4 * C::kNWG);  // one arrival per softmax warp
    }
    for (int w = 0; w < C::kNWG; ++w) mbar_init(&ms->wg_bar[w], 4);
    mbar_init(&ms->p_full[0], 4 * C::kNWG);
    mbar_init(&ms->p_full[1], 4 * C::kNWG);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ms->q_full[s], 1);
      mbar_init(&ms->q_empty[s], 1);
    }
    mbar_init(&ms->q0_done, 32 * C::kStageWarps);
    mbar_init(&ms->q1_done, 32 * C::kStageWarps);
    ms->abort = 0;
    ms->status = 0;
    ms->plan_b0 = args.p.B;  // no unit unless the plan finds one
    ms->plan_x0 = ms->plan_x1 = ms->plan_pre0 = 0;
    ms->plan_L0 = 0;
    fence_mbar_init();
    prefetch_tensormap(&map_main);
    prefetch_tensormap(&map_tail);
  }
  // the unit's row tables, one entry a thread (a single thread spent about 3 us on them,
  // integer divisions included, ahead of everything else)
  if (threadIdx.x < 48) {
    const int r = threadIdx.x;
    ms->row_j[r] = (r < args.rows) ? r / args.Hs : -(1 << 30);
    ms->row_off[r] = (r < args.rows) ? (r / args.Hs) * p.H + args.h0 + r % args.Hs : 0;
  }
  if (warp == 1) tmem_alloc(&ms->tmem_base, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms->tmem_base;
  // Everything above may overlap the previous kernel in the stream (programmatic dependent
  // launch); inputs are read only after it has completed. The merge kernel, a programmatic
  // dependent of this one, may be scheduled from here on and waits for this grid itself.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  if (trace && threadIdx.x == 0) trace[kTrWaited] = globaltimer_ns();

  if (!PF) {
    // ---- split plan (decode/verify), computed by every CTA for itself. All sequences,
    // laid end to end on a cost axis (each as kUnitCost fixed units, then its 128-key
    // blocks), are cut into gridDim.x nearly equal contiguous ranges; this CTA owns
    // [x0, x1), one unit per sequence whose blocks the range overlaps. A long history thus
    // spreads over every SM ("Scaling Kimi K3 on AMD Instinct MI355X", section
    // "并行度必须适配真正的形状": hand the long history to more work groups), a batch of
    // short sequences stays one unit per sequence, a sequence is split only where a range
    // boundary falls inside it, and a CTA that crosses into another sequence takes fewer
    // blocks.
    const int B = p.B, tid = threadIdx.x;
    const int per = (B + C::kThreads - 1) / C::kThreads;  // sequences per thread, contiguous
    const int b_lo = min(B, tid * per), b_hi = min(B, b_lo + per);
    long long mine = 0;
    for (int b = b_lo; b < b_hi; ++b) {
      const int L = p.seq_lens[b];
      const int64_t cap = p.pt_stride * (int64_t)p.page_size;
      if (L < 0 || (int64_t)L > cap) report(ms, MLA_ERR_BOUNDS);
      const int nb = blocks_of(seq_len_of(p, b));
      mine += nb > 0 ? nb + kUnitCost : 0;
    }
    // exclusive prefix of the per-thread block counts over the CTA
    long long incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) ms->scan[warp] = (int)incl;
    __syncthreads();
    long long before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < C::kThreads / 32; ++w) {
      if (w < warp) before += ms->scan[w];
      total += ms->scan[w];
    }
    long long pre = before + incl - mine;
    const long long n = gridDim.x, c = blockIdx.x;
    const long long x0 = total > 0 ? range_lo(c, total, n) : 0;
    const long long x1 = total > 0 ? range_lo(c + 1, total, n) : 0;
    for (int b = b_lo; b < b_hi; ++b) {
      const int nb = blocks_of(seq_len_of(p, b));
      const long long first = pre + kUnitCost;  // the sequence's first block
      // the range's first unit: the sequence whose span holds x0, if the range reaches
      // one of its blocks
      if (nb > 0 && pre <= x0 && x0 < first + nb && first < x1 && x0 < x1) {
        ms->plan_b0 = b;
        ms->plan_pre0 = first;
        ms->plan_L0 = seq_len_of(p, b);
      }
      if (nb > 0) pre = first + nb;
    }
    if (tid == 0) {
      ms->plan_x0 = x0;
      ms->plan_x1 = x1;
    }
    __syncthreads();
    if (trace && threadIdx.x == 0) trace[kTrPlanScan] = globaltimer_ns();
    // Ask L2 for the first unit's query rows and page-table entries before the first TMA
    // loads go out: behind the initial burst of key traffic they would arrive late, and
    // both are on the path to the first scores.
    if (warp >= 2 && ms->plan_b0 < B) {
      const int b0 = ms->plan_b0;
      const int t = threadIdx.x - 64;
      const int qlines = args.rows * 9;  // 1,152 bytes per row
      if (t < qlines)
        prefetch_l2(reinterpret_cast<const uint8_t*>(
                        p.q + ((int64_t)b0 * p.R + ms->row_off[t / 9]) * kD) + (t % 9) * 128);
      // and the second unit's rows (its sequence follows b0) for the prologue's second pass
      const Cursor c1 = next_unit<PF>(args, first_unit<PF>(args, ms));
      if (t < qlines && has_unit<PF>(args, ms, c1))
        prefetch_l2(reinterpret_cast<const uint8_t*>(
                        p.q + ((int64_t)c1.b * p.R + ms->row_off[t / 9]) * kD) + (t % 9) * 128);
      // four lines of 32 page-table entries, by the CTA's last four threads (past the
      // query lines: at most 48 rows x 9)
      const int64_t pg0 = max(0ll, ms->plan_x0 - ms->plan_pre0) * kKeyBlock / p.page_size;
      const int tp = (int)threadIdx.x - (C::kThreads - 4);
      const int64_t pg = pg0 + (int64_t)tp * 32;
      if (tp >= 0 && pg < p.pt_stride) prefetch_l2(p.page_table + (int64_t)b0 * p.pt_stride + pg);
    }
    __syncthreads();
    if (trace && threadIdx.x == 0) trace[kTrPlanPrefetch] = globaltimer_ns();
  }
  // Loads of one key tile into its stage (producer thread): the two 64-key halves' pool rows
  // from the page table, then the stage's two halves, each once the MMAs of the tile that
  // held it have released it.
  const int64_t rows64 = p.num_pages * (int64_t)p.page_size;
  const int total_rows = rows64 > 0x7fffff00 ? 0x7fffff00 : (int)rows64;
  auto issue_tile = [&](const UnitInfo& un, int k0, uint32_t fill, uint64_t policy) -> bool {
    const int s = fill % kStages;
    const uint32_t n = fill / kStages;
    uint8_t* st = smem + C::kOffStages + s * C::kStageStride;
    int y[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int kk = k0 + 64 * h;
      y[h] = total_rows;  // fully out of range: TMA fills zeros
      if (kk < un.key_hi) {
        const int lp = kk / p.page_size;
        const int phys = p.page_table[(int64_t)un.b * p.pt_stride + lp];
        if (phys >= 0 && phys < p.num_pages)
          y[h] = phys * p.page_size + (kk % p.page_size);
        else
          report(ms, MLA_ERR_BOUNDS);
      }
    }
#pragma unroll
    for (int c = 0; c < 5; ++c) {  // chunks 0..3, then the tail
      const int part = c < 4 ? part_of_chunk(c) : kTailPart;
      uint64_t* full = &ms->kv_full[s][part];
      if (c == 0 || c == 2) {  // a half begins
        if (!wait_or_abort(&ms->kv_free[s][part], (n & 1) ^ 1, ms, p)) return false;
        mbar_arrive_expect_tx(full, part_bytes(part));
      }
      if (c < 4) {
#pragma unroll
        for (int h = 0; h < 2; ++h)
          tma_load_2d_hint(st + c * kChunkBytes + h * 8192, &map_main, c * 128, y[h], full, policy);
      } else {
#pragma unroll
        for (int h = 0; h < 2; ++h)
          tma_load_2d_hint(st + C::kTail + h * 4096, &map_tail, 0, y[h], full, policy);
      }
    }
    return true;
  };
  // Decode reads each cached row once per call: its lines should not push out of L2 what is
  // reused (code, query rows, page tables, the partials the merge reads next). Prefill
  // re-reads the same rows for every unit and keeps the default policy.
  const uint64_t read_once = PF ? l2_policy_evict_normal() : l2_policy_evict_first();
  // The first unit's first tiles go out from here, straight after the plan: on the way to
  // the producer's loop a cold kernel spends microseconds fetching instructions.
  uint32_t early = 0;
  if (threadIdx.x == 0 && !p.test_stall) {
    const Cursor c0 = first_unit<PF>(args, ms);
    if (has_unit<PF>(args, ms, c0)) {
      const UnitInfo u0 = unit_info<PF>(args, ms, c0);
      for (int k0 = u0.key_lo; k0 < u0.key_hi && early < (uint32_t)kStages; k0 += kTileKeys) {
        if (!issue_tile(u0, k0, early, read_once)) break;
        ++early;
      }
    }
  }
  if (trace && threadIdx.x == 0) trace[kTrPlanned] = globaltimer_ns();

  // The first unit's queries are on every CTA's critical path: warps 2.. stage them into
  // shared memory together (about two rows each). Later units' rows go to this CTA's query
  // image in global memory and reach shared memory in one bulk copy when their unit starts
  // (staging takes one warp far longer than a unit boundary may last): warps 2.. stage the
  // second unit there before the first key tile lands, the stager warp each later one while
  // the unit before it runs.
  if (warp >= 2) {
    Cursor c0 = first_unit<PF>(args, ms);
    while (has_unit<PF>(args, ms, c0) && tiles_in(unit_info<PF>(args, ms, c0)) == 0) c0 = next_unit<PF>(args, c0);
    if (has_unit<PF>(args, ms, c0)) {
      const UnitInfo ui = unit_info<PF>(args, ms, c0);
      stage_rows<RP, C::kStageWarps>(p, ui.rows, ms->row_off, p.q + (int64_t)ui.qrow0 * kD, qbuf,
                                     ms->row_scale[0], warp - 2, lane);
      fence_proxy_async_smem();
      mbar_arrive(&ms->q0_done);
      Cursor c1 = next_unit<PF>(args, c0);
      while (has_unit<PF>(args, ms, c1) && tiles_in(unit_info<PF>(args, ms, c1)) == 0) c1 = next_unit<PF>(args, c1);
      if (has_unit<PF>(args, ms, c1)) {
        const UnitInfo u1 = unit_info<PF>(args, ms, c1);
        uint8_t* img = p.qimg + (int64_t)blockIdx.x * p.qimg_stride;
        stage_rows<RP, C::kStageWarps>(p, u1.rows, ms->row_off, p.q + (int64_t)u1.qrow0 * kD, img,
                                       reinterpret_cast<float*>(img + C::kQBytes), warp - 2, lane);
        fence_proxy_async_global();
        mbar_arrive(&ms->q1_done);
      }
    }
  }

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t fill = 0;  // tiles issued so far (the first `early` ones in the prologue)
      // L2 prefetch cursor: runs kPrefetchTiles tiles ahead of the TMA loads so that they
      // find their pages in L2 (deeper than the two shared-memory stages allow). The first
      // kStages tiles are the TMA loads' own: the cursor starts past them (no page-table
      // reads there: each is a round trip the second tile's load would wait behind).
      Cursor pf_c = first_unit<PF>(args, ms);
      UnitInfo pu = has_unit<PF>(args, ms, pf_c) ? unit_info<PF>(args, ms, pf_c) : UnitInfo{};
      int pf_k = pu.key_lo;
      uint32_t pf_tiles = 0;
      auto prefetch_upto = [&](uint32_t target, bool issue) {
        while (pf_tiles < target && has_unit<PF>(args, ms, pf_c)) {
          if (pf_k >= pu.key_hi) {  // unit done (or empty)
            pf_c = next_unit<PF>(args, pf_c);
            if (has_unit<PF>(args, ms, pf_c)) pu = unit_info<PF>(args, ms, pf_c);
            pf_k = pu.key_lo;
            continue;
          }
          for (int h = 0; h < 2 && issue; ++h) {
            const int kk = pf_k + 64 * h;
            if (kk < pu.key_hi) {
              const int phys = p.page_table[(int64_t)pu.b * p.pt_stride + kk / p.page_size];
              if (phys >= 0 && phys < p.num_pages) {
                const int rows = min(64, pu.key_hi - kk);
                bulk_prefetch_l2(p.pool + ((int64_t)phys * p.page_size + kk % p.page_size) * kD,
                                 (uint32_t)rows * kD);
              }
            }
          }
          ++pf_tiles;
          pf_k += kTileKeys;
        }
      };
      prefetch_upto(kStages, false);
      for (Cursor cu = first_unit<PF>(args, ms); has_unit<PF>(args, ms, cu) && !aborted(ms) && !p.test_stall;
           cu = next_unit<PF>(args, cu)) {
        const UnitInfo un = unit_info<PF>(args, ms, cu);
        for (int k0 = un.key_lo; k0 < un.key_hi; k0 += kTileKeys) {
          const bool ok = fill < early || issue_tile(un, k0, fill, read_once);
          if (!ok) break;
          ++fill;
          prefetch_upto(fill + kPrefetchTiles, true);
        }
      }
      // Drain: wait (bounded) until the consumers released every part still holding a load.
      for (uint32_t f = (fill > kStages ? fill - kStages : 0); f < fill; ++f)
        for (int c = 0; c < kParts; ++c)
          mbar_wait(&ms->kv_free[f % kStages][c], (f / kStages) & 1, kWaitLimitNs);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ scores issuer
    // QK of every tile, chunk by chunk as its KV stage fills, once its S^T buffer has been
    // read and its unit's query terms are staged. Values (PV) have their own issuing warp: a
    // single thread spends tens of cycles per tcgen05.mma, so one issuer would serialise the
    // two.
    if (lane == 0) {
      constexpr uint32_t idesc_qk = instr_desc(0, 0, 0, 0, 128, C::NQK);
      const uint64_t a_main0 = smem_desc(smem_addr(smem + C::kOffStages), 16, 1024, Swizzle::k128B);
      const uint64_t a_tail0 = smem_desc(smem_addr(smem + C::kOffStages + C::kTail), 16, 512, Swizzle::k64B);
      const uint64_t b_main0 = smem_desc(smem_addr(qbuf), 16, 1024, Swizzle::k128B);
      const uint64_t b_tail0 = smem_desc(smem_addr(qbuf + 4 * (C::NQK * 128)), 16, 512, Swizzle::k64B);
      uint32_t g = 0, units_done = 0;
      bool ok = true;
      for (Cursor cu = first_unit<PF>(args, ms); has_unit<PF>(args, ms, cu) && ok; cu = next_unit<PF>(args, cu)) {
        const int n = tiles_in(unit_info<PF>(args, ms, cu));
        if (n == 0) continue;
        const int qslot = units_done % C::kQB;
        if (!(ok = wait_or_abort(&ms->q_full[qslot], (units_done / C::kQB) & 1, ms, p))) break;
        const uint32_t qoff = (uint32_t)(qslot * C::kQBytes) >> 4;
        for (int t = 0; t < n; ++t, ++g) {
          const int s = g % kStages, sb = g % C::kSBuf;
          const uint32_t ph = (g / kStages) & 1;
          if (!(ok = wait_or_abort(&ms->s_empty[sb], ((g / C::kSBuf) & 1) ^ 1, ms, p))) break;
          const uint32_t soff = (uint32_t)(s * C::kStageStride) >> 4;
          const uint32_t d = tmem + C::kSCol + sb * C::NQK;
          // each latent chunk as soon as it has landed, then the RoPE tail
#pragma unroll
          for (int c = 0; c < 4 && ok; ++c) {
            if (c == 0 || c == 2) {  // a half has landed
              if (!(ok = wait_or_abort(&ms->kv_full[s][part_of_chunk(c)], ph, ms, p))) break;
              tc_fence_after();
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_f8f6f4(d, a_main0 + soff + ((c * kChunkBytes + kk * 32) >> 4),
                         b_main0 + qoff + ((c * (C::NQK * 128) + kk * 32) >> 4), idesc_qk,
                         (c | kk) != 0);
          }
          if (!ok) break;  // the tail belongs to the second half, landed by now
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
            mma_f8f6f4(d, a_tail0 + soff + ((kk * 32) >> 4), b_tail0 + qoff + ((kk * 32) >> 4),
                       idesc_qk, 1);
          mma_commit(&ms->s_full[sb]);
        }
        if (!ok) break;
        mma_commit(&ms->q_empty[qslot]);  // that query buffer is free once these complete
        ++units_done;
      }
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------------ values issuer
    // PV of every tile the moment its probabilities are in shared memory; completion hands
    // the KV stage back to the producer, part by part, and lets the softmax reuse P and
    // rescale O.
    if (lane == 0) {
      // A = V^T as e4m3 codes, B = P^T as e5m2 terms (kind::f8f6f4 takes each operand's
      // format from its own descriptor field), both MN-major
      constexpr uint32_t idesc_stacked = instr_desc(kFmtE4M3, kFmtE5M2, 1, 1, 128, 3 * RP);
      constexpr uint32_t idesc_term = instr_desc(kFmtE4M3, kFmtE5M2, 1, 1, 128, RP);
      const uint64_t a0 = smem_desc(smem_addr(smem + C::kOffStages), kChunkBytes, 1024, Swizzle::k128B);
      // P^T of stage 0's tile (at 48 rows; each stage has its own) or the shared buffer
      const uint64_t b0 = smem_desc(smem_addr(C::kPInStage ? smem + C::kOffStages + 4 * kChunkBytes : pbuf),
                                    128, 2048, Swizzle::kNone);
      uint32_t g = 0;
      bool ok = true;
      for (Cursor cu = first_unit<PF>(args, ms); has_unit<PF>(args, ms, cu) && ok; cu = next_unit<PF>(args, cu)) {
        const int n = tiles_in(unit_info<PF>(args, ms, cu));
        for (int t = 0; t < n; ++t, ++g) {
          if (!(ok = wait_or_abort(&ms->p_full[g & 1], (g >> 1) & 1, ms, p))) break;
          tc_fence_after();
          const int s = g % kStages;
          const uint32_t soff = (uint32_t)(s * C::kStageStride) >> 4;
          const uint32_t poff = C::kPInStage ? soff : 0u;
          // chunk by chunk, each freed for the next tile's load once its own MMAs complete
          // (back-to-back MMAs into one accumulator cost no more than alternating ones)
          // chunk by chunk (back-to-back MMAs into one accumulator cost no more than
          // alternating ones); each half of the stage is handed back once its MMAs complete.
          // The second half's release also stands for the whole tile's values being done
          // (P, which lives in the tail at 48 rows, and O for the softmax's rescale).
#pragma unroll
          for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              const uint64_t a = a0 + soff + ((c * kChunkBytes + ks * 4096) >> 4);
              if (C::oterms(c) == 3) {  // stacked: one MMA over all three terms' rows
                mma_f8f6f4(tmem + C::ocol(c), a, b0 + poff + ((ks * 512) >> 4), idesc_stacked,
                           t > 0 || ks > 0);
              } else {  // summed: one MMA per term into the same accumulator
#pragma unroll
                for (int term = 0; term < 3; ++term)
                  mma_f8f6f4(tmem + C::ocol(c), a, b0 + poff + ((C::pterm(term) + ks * 512) >> 4),
                             idesc_term, t > 0 || ks > 0 || term > 0);
              }
            }
            if (c == 1 || c == 3) mma_commit(&ms->kv_free[s][part_of_chunk(c)]);
          }
        }
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------------ query stager
    // Each unit's query rows go into the query operand as two e4m3 terms with a per-row
    // power-of-two scale, as soon as the previous unit's scores stopped reading it; the
    // softmax warps meanwhile finish the previous unit.
    uint32_t k = 0;  // units with work, in order
    uint8_t* img = p.qimg + (int64_t)blockIdx.x * p.qimg_stride;
    constexpr uint32_t kImgBytes = C::kQBytes + 48 * sizeof(float);
    for (Cursor cu = first_unit<PF>(args, ms); has_unit<PF>(args, ms, cu); cu = next_unit<PF>(args, cu)) {
      const UnitInfo ui = unit_info<PF>(args, ms, cu);
      if (tiles_in(ui) == 0) continue;
      const int slot = k % C::kQB;
      if (k == 0) {  // staged into shared memory by warps 2.. in the prologue
        if (!wait_or_abort(&ms->q0_done, 0, ms, p)) break;
        if (lane == 0) mbar_arrive(&ms->q_full[0]);
        ++k;
        continue;
      }
      if (k == 1) {  // staged into the image by warps 2.. in the prologue
        if (!wait_or_abort(&ms->q1_done, 0, ms, p)) break;
      } else {
        // the image is free once the previous unit's copy out of it has landed
        const uint32_t pk = k - 1;
        if (!wait_or_abort(&ms->q_full[pk % C::kQB], (pk / C::kQB) & 1, ms, p)) break;
        stage_rows<RP, 1>(p, ui.rows, ms->row_off, p.q + (int64_t)ui.qrow0 * kD, img,
                          reinterpret_cast<float*>(img + C::kQBytes), 0, lane);
        fence_proxy_async_global();
        __syncwarp();
      }
      if (k >= (uint32_t)C::kQB && !wait_or_abort(&ms->q_empty[slot], ((k / C::kQB) - 1) & 1, ms, p)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&ms->q_full[slot], kImgBytes);
        bulk_g2s(qbuf + slot * C::kQBytes, img, C::kQBytes, &ms->q_full[slot]);
        bulk_g2s(ms->row_scale[k & 1], img + C::kQBytes, 48 * sizeof(float), &ms->q_full[slot]);
      }
      __syncwarp();
      ++k;
    }
  } else if (warp >= kSoftmaxWarp0) {
    // ------------------------------------------------------------------ softmax warpgroups
    // Two or three warpgroups, each owning an equal share of the query rows; thread i of a
    // warpgroup owns key i of the tile (its TMEM lane).
    constexpr int RH = C::kRH;
    const int wg = (warp - kSoftmaxWarp0) >> 2;
    const int rb = wg * RH;  // rows [rb, rb + RH)
    const int wq = warp & 3;  // TMEM lane quadrant
    const int i = wq * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(wq * 32) << 16;
    const float kv_scale = p.kv_scale;
    uint32_t tile = 0, wg_phase = 0, k = 0;  // k: units with work, in order
    // PV completions are confirmed in tile order, each before the PV two tiles later can
    // complete (that one needs this warpgroup's next P), so a phase parity names one tile
    // A wait that gives up does not make its lane leave on its own: `ok` collects the
    // outcome and the warp votes at fixed points (once a tile, before the epilogue), so a
    // timeout never splits a warp ahead of a warp-wide instruction (tcgen05.ld, __syncwarp).
    // After a failed wait the lanes run on to the vote on whatever they read; the call
    // reports MLA_ERR_TIMEOUT and its outputs are not to be used.
    // Arrivals are one per warp: the lanes meet at __syncwarp first (which also orders
    // their earlier memory accesses before lane 0's release).
    auto warp_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
      return wait_or_abort(bar, parity, ms, p);
    };
    auto warp_arrive = [&](uint64_t* bar) {
      __syncwarp();
      if (lane == 0) mbar_arrive(bar);
    };
    int pv_seen = -1;
    auto wait_pv_upto = [&](int target) -> bool {
      for (int g = pv_seen + 1; g <= target; ++g) {
        if (!warp_wait(&ms->kv_free[g % kStages][kParts - 1], (g / kStages) & 1)) return false;
        pv_seen = g;
      }
      return true;
    };
    uint64_t* wg_bar = &ms->wg_bar[wg];
    // Bounded warpgroup barrier: every warp arrives, then waits for the phase.
    auto wg_sync = [&]() -> bool {
      warp_arrive(wg_bar);
      const bool good = warp_wait(wg_bar, wg_phase & 1);
      ++wg_phase;
      return good;
    };
    bool ok = true;
    for (Cursor cu = first_unit<PF>(args, ms); has_unit<PF>(args, ms, cu) && ok; cu = next_unit<PF>(args, cu)) {
      const UnitInfo un = unit_info<PF>(args, ms, cu);
      const int R = un.rows;
      const int ntiles = tiles_in(un);
      const bool final_out = un.final_out != 0;
      if (ntiles == 0) {  // no visible key at all: out = 0, lse = -inf (or an empty partial)
        for (int r = rb; r < rb + RH && r < R; ++r) {
          if (final_out) {
            const int64_t row = (int64_t)un.qrow0 + ms->row_off[r];
            for (int dv = i; dv < kDV; dv += 128) store_out(p, row * kDV + dv, 0.f);
            if (i == 0 && p.lse) p.lse[row] = -INFINITY;
          } else if (i == 0) {
            p.part_lse[(int64_t)un.slot * p.part_rows + ms->row_off[r]] = -INFINITY;
          }
        }
        continue;
      }
      const int L = un.L;
      // last visible key of new position j is L - n_q + j + mask_shift (and the unit ends at
      // key_hi); mask_shift is 0 except for a shard that holds none of the new positions
      const int lim_cap = un.key_hi - 1;
      const int lim0 = min(lim_cap, L - p.n_q + un.j0 + p.mask_shift);
      // this unit's row scales (staged with its query terms)
      ok &= warp_wait(&ms->q_full[k % C::kQB], (k / C::kQB) & 1);
      // mo: the row's running max less kPScale (p = 2^(x - mo)); kNoMax before its first key
      float rs[RH], mo[RH], l[RH];
#pragma unroll
      for (int r = 0; r < RH; ++r) {
        rs[r] = ms->row_scale[k & 1][rb + r];
        mo[r] = kNoMax;
        l[r] = 0.f;
      }
      for (int t = 0; t < ntiles; ++t, ++tile) {
        const int sb = tile % C::kSBuf;
        const int s = tile % kStages;
        const int k0 = un.key_lo + t * kTileKeys;
        const int kabs = k0 + i;
        ok &= warp_wait(&ms->s_full[sb], (tile / C::kSBuf) & 1);
        tc_fence_after();
        float x[RH];
        {
          const uint32_t base = tmem + lane_addr + C::kSCol + sb * C::NQK + rb;
          // every load of the tile first, one wait
          float a[RH], b2[RH];
#pragma unroll
          for (int c = 0; c < RH; c += 8) {
            tmem_ld8(base + c, *reinterpret_cast<float(*)[8]>(&a[c]));
            tmem_ld8(base + RP + c, *reinterpret_cast<float(*)[8]>(&b2[c]));
          }
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < RH; ++e) x[e] = fmaf(b2[e], 1.0f / kQTerm2, a[e]) * rs[e];
        }
        tc_fence_before();
        warp_arrive(&ms->s_empty[sb]);
        if (trace && threadIdx.x == 32 * kSoftmaxWarp0 && t == 0) {
          if (tile == 0) trace[kTrFirstScores] = globaltimer_ns();
          if (k == 1) trace[kTrUnit2Scores] = globaltimer_ns();
        }
        // masking only on tiles that reach past the first new position's last visible key
        if (k0 + kTileKeys - 1 > lim0) {
#pragma unroll
          for (int r = 0; r < RH; ++r) {
            const int lim = min(lim_cap, lim0 + ms->row_j[rb + r]);
            if (kabs > lim) x[r] = -INFINITY;
          }
        }
        // The running max of a row moves only when some score exceeds it by more than the
        // 2^8 headroom (kRescaleGap in log2 units); only then is the exact tile max needed.
        // The warps of the warpgroup first agree whether that happens anywhere, and the
        // common case skips the exchange of per-row maxima.
        bool over = false;
#pragma unroll
        for (int r = 0; r < RH; ++r) over |= (x[r] > mo[r] + (kPScale + kRescaleGap));
        over = __any_sync(0xffffffffu, over);
        if (__any_sync(0xffffffffu, !ok)) {  // the warp's once-a-tile vote on its waits
          ok = false;
          break;
        }
        if (lane == 0) ms->grow[tile & 1][wg * 4 + wq] = over ? 1 : 0;
        ok &= wg_sync();
        const int4 gf = *reinterpret_cast<const int4*>(&ms->grow[tile & 1][wg * 4]);
        bool need_rescale = false;
        if ((gf.x | gf.y | gf.z | gf.w) != 0) {
          // tile max per row: warp max in hardware, then the four warps through shared memory
          float* red = &ms->red[tile & 1][0];
#pragma unroll
          for (int r = 0; r < RH; ++r) {
            const float v = warp_max(x[r]);
            if (lane == 0) red[(rb + r) * 4 + wq] = v;
          }
          ok &= wg_sync();
#pragma unroll
          for (int r = 0; r < RH; ++r) {
            const float4 t4 = *reinterpret_cast<const float4*>(&red[(rb + r) * 4]);
            const float tm = fmaxf(fmaxf(t4.x, t4.y), fmaxf(t4.z, t4.w));
            float al = 1.f;
            if (tm > mo[r] + (kPScale + kRescaleGap)) {  // lazy: the headroom absorbs small increases
              al = ex2(mo[r] + kPScale - tm);  // 0 before the first key (nothing accumulated yet)
              need_rescale |= (mo[r] != kNoMax);
              l[r] *= al;
              mo[r] = tm - kPScale;
            }
            if (lane == 0) ms->alpha[rb + r] = al;
          }
        }
        // p = 2^(x - m + 11) <= 2^15 rounded to fp16, then three e5m2 terms, each the
        // nearest e5m2 value to what the terms before it left (the differences are exact
        // in fp16); the row sum takes the float32 p
        uint32_t w1[RH / 4], w2[RH / 4], w3[RH / 4];
#pragma unroll
        for (int r = 0; r < RH; r += 2) {
          const float p0 = ex2(x[r] - mo[r]);  // masked (x = -inf) and keyless rows give 0
          const float p1 = ex2(x[r + 1] - mo[r + 1]);
          l[r] += p0;
          l[r + 1] += p1;
          const uint32_t h = f32x2_to_f16x2(p0, p1);
          const uint32_t c1 = f16x2_to_e5m2x2(h);
          const uint32_t r1 = hsub2(h, e5m2x2_to_f16x2(c1));
          const uint32_t c2 = f16x2_to_e5m2x2(r1);
          const uint32_t r2 = hsub2(r1, e5m2x2_to_f16x2(c2));
          const uint32_t c3 = f16x2_to_e5m2x2(r2);
          const int wi = r >> 2;
          if ((r & 2) == 0) {
            w1[wi] = c1;
            w2[wi] = c2;
            w3[wi] = c3;
          } else {
            w1[wi] |= c1 << 16;
            w2[wi] |= c2 << 16;
            w3[wi] |= c3 << 16;
          }
        }
        // The previous tile's PV must be done before O is rescaled, and before P is written
        // when one P buffer serves every tile. With P in the stage, PV(tile - 2) is known
        // done (this tile's keys replaced its stage) and is only confirmed here.
        {
          const int upto = (int)tile - ((C::kPInStage && !need_rescale) ? 2 : 1);
          ok &= wait_pv_upto(upto);
          tc_fence_after();
        }
        if (t > 0) {
          if (need_rescale) {
            __syncwarp();
            const float* al = &ms->alpha[rb];
            // (rare: rolled up at 16 rows, so that the code of the tile loop stays small; at
            // more rows the rolled loop needs more registers than there are)
#pragma unroll(C::kUnrollChunks)
            for (int c = 0; c < 4; ++c) {
#pragma unroll
              for (int term = 0; term < C::oterms(c); ++term) {
#pragma unroll
                for (int cc = 0; cc < RH; cc += 8) {
                  const uint32_t a = tmem + lane_addr + C::ocol(c) + term * RP + rb + cc;
                  float v[8];
                  tmem_ld8(a, v);
                  tmem_wait_ld();
#pragma unroll
                  for (int e = 0; e < 8; ++e) v[e] *= al[cc + e];
                  tmem_st8(a, v);
                }
              }
            }
            tmem_wait_st();
          }
        }
        // keys past this unit's range: zero their V bytes so 0 * garbage cannot be NaN
        if (wg == 0 && kabs >= un.key_hi) {
          uint8_t* st = smem + C::kOffStages + s * C::kStageStride + (i >> 6) * 8192 + (i & 63) * 128;
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 8; ++e)
              reinterpret_cast<uint4*>(st + c * kChunkBytes)[e] = make_uint4(0, 0, 0, 0);
        }
        // P^T: MN-major, 16 rows x 8 keys core matrices; term t, row group g at
        // pterm(t) + g * 2048, key i at (i / 8) * 128 + (i % 8) * 16, row r at byte r % 16.
        // A warpgroup with 16 rows (a whole row group) writes each key's 16 bytes at once: a
        // warp then stores 512 contiguous bytes, free of bank conflicts (8-byte halves at a
        // 16-byte stride took four shared-memory wavefronts a store where two suffice). With
        // 8 rows it writes its 8-byte half.
        uint8_t* pb = C::kPInStage ? smem + C::kOffStages + s * C::kStageStride + 4 * kChunkBytes : pbuf;
        const int off = (i >> 3) * 128 + (i & 7) * 16;
        if constexpr (RH % 16 == 0) {
#pragma unroll
          for (int blk = 0; blk < RH / 16; ++blk) {
            const int o = ((rb >> 4) + blk) * 2048 + off;
            *reinterpret_cast<uint4*>(pb + C::pterm(0) + o) =
                make_uint4(w1[4 * blk], w1[4 * blk + 1], w1[4 * blk + 2], w1[4 * blk + 3]);
            *reinterpret_cast<uint4*>(pb + C::pterm(1) + o) =
                make_uint4(w2[4 * blk], w2[4 * blk + 1], w2[4 * blk + 2], w2[4 * blk + 3]);
            *reinterpret_cast<uint4*>(pb + C::pterm(2) + o) =
                make_uint4(w3[4 * blk], w3[4 * blk + 1], w3[4 * blk + 2], w3[4 * blk + 3]);
          }
        } else {
#pragma unroll
          for (int blk = 0; blk < RH / 8; ++blk) {
            const int row0 = rb + 8 * blk;
            const int o = (row0 >> 4) * 2048 + off + ((row0 & 15) >> 3) * 8;
            *reinterpret_cast<uint2*>(pb + C::pterm(0) + o) = make_uint2(w1[2 * blk], w1[2 * blk + 1]);
            *reinterpret_cast<uint2*>(pb + C::pterm(1) + o) = make_uint2(w2[2 * blk], w2[2 * blk + 1]);
            *reinterpret_cast<uint2*>(pb + C::pterm(2) + o) = make_uint2(w3[2 * blk], w3[2 * blk + 1]);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        warp_arrive(&ms->p_full[tile & 1]);
      }
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      if (trace && threadIdx.x == 32 * kSoftmaxWarp0) trace[kTrLastP] = globaltimer_ns();
      // ---- epilogue: row sums, then O / l
#pragma unroll
      for (int r = 0; r < RH; ++r) {
        float v = l[r];
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) ms->lred[wq][rb + r] = v;
      }
      ok &= wg_sync();
      float inv[RH];
#pragma unroll
      for (int r = 0; r < RH; ++r) {
        const int rr = rb + r;
        const float lt = ms->lred[0][rr] + ms->lred[1][rr] + ms->lred[2][rr] + ms->lred[3][rr];
        l[r] = lt;
        inv[r] = lt > 0.f ? kv_scale / lt : 0.f;
      }
      ok &= wait_pv_upto((int)tile - 1);
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (trace && threadIdx.x == 32 * kSoftmaxWarp0) trace[kTrLastPV] = globaltimer_ns();
      // (once a unit: rolled up over the dv chunks at 16 rows, fewer instructions to fetch)
#pragma unroll(C::kUnrollChunks)
      for (int c = 0; c < 4; ++c) {
        const int NT = C::oterms(c);
#pragma unroll
        for (int cc = 0; cc < RH; cc += 8) {
          if (rb + cc >= R) break;
          // The rows' output offsets go to registers before any of these stores: as far as
          // the compiler knows a store may alias the table, so a lookup between two stores
          // would wait for the first one to drain (about 60 ns a store when every SM writes).
          int roffs[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) roffs[e] = ms->row_off[rb + cc + e];
          float o[3][8];
#pragma unroll
          for (int term = 0; term < 3; ++term)
            if (term < NT) tmem_ld8(tmem + lane_addr + C::ocol(c) + term * RP + rb + cc, o[term]);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int r = cc + e;
            if (rb + r >= R) break;
            float acc = o[0][e];
#pragma unroll
            for (int term = 1; term < 3; ++term)
              if (term < NT) acc += o[term][e];
            const int dv = c * 128 + i;
            if (final_out) {
              store_out(p, ((int64_t)un.qrow0 + roffs[e]) * kDV + dv, acc * inv[r]);
            } else {
              p.part_out[((int64_t)un.slot * p.part_rows + roffs[e]) * kDV + dv] = acc * inv[r];
            }
          }
        }
      }
      tc_fence_before();
      if (i < RH && rb + i < R) {
        float lt = 0.f, mm = kNoMax;
#pragma unroll
        for (int r = 0; r < RH; ++r)
          if (r == i) {
            lt = l[r];
            mm = mo[r];
          }
        const float lse = (lt > 0.f) ? 0.6931471805599453f * (mm + log2f(lt)) : -INFINITY;
        const int roff = ms->row_off[rb + i];
        if (final_out) {
          if (p.lse) p.lse[(int64_t)un.qrow0 + roff] = lse;
        } else {
          p.part_lse[(int64_t)un.slot * p.part_rows + roff] = lse;
        }
      }
      ++k;
      if (trace && threadIdx.x == 32 * kSoftmaxWarp0) {
        trace[kTrEpilogue] = globaltimer_ns();
        trace[kTrCounts] = ((unsigned long long)tile << 32) | k;
        if (k == 1) trace[kTrUnit1End] = globaltimer_ns();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (trace && threadIdx.x == 0) trace[kTrExit] = globaltimer_ns();
  if (threadIdx.x == 0) {
    // this CTA's status word (a later launch of the same call only adds errors)
    if (args.status_overwrite || ms->status != 0) p.status[blockIdx.x] = ms->status;
    if (blockIdx.x == 0 && args.status_overwrite) p.hdr->num_ctas = gridDim.x;
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled, looked up through the runtime so the library needs no link-time
// dependency on the driver library.
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
    else
      cudaGetLastError();
  }
  return fn;
}

bool encode_pool_maps(const AttnParams& p, CUtensorMap* main_map, CUtensorMap* tail_map) {
  const EncodeTiledFn encode = encode_fn();
  if (!encode) return false;
  const uint64_t rows = (uint64_t)p.num_pages * (uint64_t)p.page_size;
  if (rows == 0 || rows > 0x7fffff00ull) return false;
  cuuint64_t dims_main[2] = {512, rows};
  cuuint64_t dims_tail[2] = {64, rows};
  cuuint64_t strides[1] = {(cuuint64_t)kD};
  cuuint32_t box_main[2] = {128, 64};
  cuuint32_t box_tail[2] = {64, 64};
  cuuint32_t estr[2] = {1, 1};
  CUresult r1 = encode(main_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                                       const_cast<uint8_t*>(p.pool), dims_main, strides, box_main,
                                       estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                       CU_TENSOR_MAP_SWIZZLE_128B,
                                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  CUresult r2 = encode(tail_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                                       const_cast<uint8_t*>(p.pool + 512), dims_tail, strides,
                                       box_tail, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                       CU_TENSOR_MAP_SWIZZLE_64B,
                                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r1 == CUDA_SUCCESS && r2 == CUDA_SUCCESS;
}

template <int RP, int PF, bool TR>
cudaError_t launch_rp_tr(const DecodeArgs& a, const CUtensorMap& mm, const CUtensorMap& mt,
                         int grid, cudaStream_t s) {
  constexpr int smem = smem_bytes<RP>();
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<RP, PF, TR>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(Cfg<RP>::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_tc_kernel<RP, PF, TR>, a, mm, mt);
}

template <int RP, int PF>
cudaError_t launch_rp(const DecodeArgs& a, const CUtensorMap& mm, const CUtensorMap& mt,
                      int grid, cudaStream_t s) {
  if constexpr (PF == 2) {  // (never traced)
    return launch_rp_tr<RP, PF, false>(a, mm, mt, grid, s);
  } else {
    return a.p.trace ? launch_rp_tr<RP, PF, true>(a, mm, mt, grid, s)
                     : launch_rp_tr<RP, PF, false>(a, mm, mt, grid, s);
  }
}

}  // namespace

// Decode / verify attention for every unit of the plan. Rows per launch are limited to 48
// (three query terms of 48 rows fit TMEM); 16 heads x 4 positions run as two head halves.
cudaError_t launch_decode_tc(const AttnParams& p, int num_sms, cudaStream_t s, int* launches) {
  CUtensorMap mm, mt;
  if (!encode_pool_maps(p, &mm, &mt)) return cudaErrorInvalidValue;
  const int grid = p.num_ctas;  // the split plan cuts the blocks into this many ranges
  (void)num_sms;
  const int groups = (p.R > 48) ? 2 : 1;
  for (int gi = 0; gi < groups; ++gi) {
    DecodeArgs a;
    a.p = p;
    a.Hs = p.H / groups;
    a.h0 = gi * a.Hs;
    if (gi == groups - 1) a.Hs = p.H - a.h0;
    a.rows = p.n_q * a.Hs;
    a.prefill = 0;
    a.P = 0;
    a.num_units = 0;
    a.unit_end = 0;
    a.split_base = 0;
    a.status_overwrite = (gi == 0);
    cudaError_t e;
    if (a.rows <= 16)
      e = launch_rp<16, 0>(a, mm, mt, grid, s);
    else if (a.rows <= 32)
      e = launch_rp<32, 0>(a, mm, mt, grid, s);
    else
      e = launch_rp<48, 0>(a, mm, mt, grid, s);
    if (e != cudaSuccess) return e;
    ++*launches;
  }
  return cudaSuccess;
}

// Causal prefill of one sequence: units are blocks of P = 48 / H new positions (all their
// heads, at most 48 rows) over every key they see, handed out longest first, one a round
// per CTA. A last round that would leave CTAs idle runs instead as a second launch over
// the halves of its units (keys split in two), and a merge kernel joins the halves.
cudaError_t launch_prefill_tc(const AttnParams& p, int num_sms, cudaStream_t s, int* launches) {
  CUtensorMap mm, mt;
  if (!encode_pool_maps(p, &mm, &mt)) return cudaErrorInvalidValue;
  DecodeArgs a;
  a.p = p;
  a.h0 = 0;
  a.Hs = p.H;
  a.P = 48 / p.H;
  a.rows = a.P * p.H;
  a.prefill = 1;
  a.status_overwrite = 1;
  a.num_units = (p.n_q + a.P - 1) / a.P;
  const int grid = min(num_sms, a.num_units);
  const int left = a.num_units % grid;  // units of an incomplete last round
  const bool split = left > 0 && 2 * left <= grid;
  a.split_base = a.num_units - left;
  a.unit_end = split ? a.split_base : a.num_units;
  cudaError_t e = launch_rp<48, 1>(a, mm, mt, grid, s);
  if (e != cudaSuccess) return e;
  ++*launches;
  if (!split) return cudaSuccess;
  DecodeArgs b = a;
  b.unit_end = 2 * left;  // halves: one a CTA
  b.status_overwrite = 0;
  b.p.trace = nullptr;    // the profiling hook traces the main launch
  if ((e = launch_rp<48, 2>(b, mm, mt, 2 * left, s)) != cudaSuccess) return e;
  ++*launches;
  if ((e = launch_merge_prefill(p, a.P, left, s)) != cudaSuccess) return e;
  ++*launches;
  return cudaSuccess;
}

}  // namespace mla
