// mla_merge.cu -- the log-sum-exp merge of split-KV partial results.
//
// Per query row, lse = ln sum_s exp(lse_s) and out = sum_s exp(lse_s - lse) out_s, the
// "merge by normalisation statistics" of position-sharded attention ("Scaling Kimi K3 on
// AMD Instinct MI355X", section "缓存可复用，还要能一致地恢复").
//
// Where the partials come from: the attention kernel lays all sequences end to end on a
// cost axis (a fixed cost per sequence, then its 128-key blocks) and cuts it into one
// contiguous range per CTA; a sequence is split only where a range boundary falls inside
// its blocks, so its pieces sit on consecutive CTAs, and only the first and the last unit
// of a CTA's range can hold part of a sequence. Partial slot 2c is the piece that is CTA
// c's first unit, slot 2c + 1 the piece that ends its range after an earlier sequence.
#include <cuda_bf16.h>
#include <math.h>

#include "mla_internal.cuh"

namespace mla {

namespace {

constexpr int kMergeWarps = 8;
constexpr int kMergeThreads = 32 * kMergeWarps;


// Merge one dv chunk (32 * VEC values; lane l owns VEC consecutive ones) of one row from
// `count` partials; slot_of(i) gives the partial index of piece i, whose row sits at
// po[(slot * R + r) * 512] and pl[slot * R + r]. Latency sets the cost (the partials were
// written by the kernel just before), so everything is loaded in one round: each lane the
// lse values it reduces (every warp reduces them all, no barrier) and warp w's pieces
// w, w + 8, ..., with their own lse values for the weights; only pieces past the first
// batch, or lse values past 256, take further rounds. The warps' sums meet in shared memory.
__device__ __forceinline__ void store_val(uint16_t* p, float v) {
  *p = __bfloat16_as_ushort(__float2bfloat16_rn(v));
}
__device__ __forceinline__ void store_val(float* p, float v) { *p = v; }

// WPR: warps on one row (kMergeWarps / WPR rows a CTA, each its own group of warps with its
// own named barrier, so one group may leave early without the other).
template <int VEC, int WPR, typename OutT, typename SlotOf>
__device__ void merge_row_chunk(const float* __restrict__ po, const float* __restrict__ pl,
                                int count, SlotOf slot_of, int64_t r, int64_t R, int chunk,
                                OutT* __restrict__ out_row, float* lse_out) {
  constexpr int W = 32 * VEC;                             // dv per CTA
  constexpr int NB = VEC >= 16 ? 2 : (VEC >= 4 ? 8 : 24);  // pieces per batch and warp
  constexpr int kLse = 8;                                 // lse values per lane (256 pieces)
  constexpr int kGroupThreads = 32 * WPR;
  __shared__ __align__(16) float s_acc[kMergeWarps][W];
  const int lane = threadIdx.x & 31, gw = threadIdx.x >> 5;
  const int g = gw / WPR, warp = gw % WPR;  // row group, warp within it
  const int gt = threadIdx.x - g * kGroupThreads;
  if (count <= 0) {  // nothing to merge: out = 0, lse = -inf
    for (int x = gt; x < W; x += kGroupThreads) store_val(out_row + chunk * W + x, 0.f);
    if (gt == 0 && chunk == 0 && lse_out) *lse_out = -INFINITY;
    return;
  }
  // load the pieces i0 + k * 8 (k < NB) of this warp: weights' lse values and data;
  // indices past the end are clamped to the last piece (a valid address) and dropped later
  float v[NB][VEC];
  float w[NB];
  auto load_batch = [&](int i0) {
    int64_t at[NB];
#pragma unroll
    for (int k = 0; k < NB; ++k) at[k] = slot_of(min(i0 + k * WPR, count - 1)) * R + r;
#pragma unroll
    for (int k = 0; k < NB; ++k) {
      w[k] = __ldg(pl + at[k]);
      const float* src = po + at[k] * kDV + chunk * W + lane * VEC;
      if constexpr (VEC % 4 == 0) {
#pragma unroll
        for (int e = 0; e < VEC; e += 4) {
          const float4 t = __ldg(reinterpret_cast<const float4*>(src + e));
          v[k][e] = t.x;
          v[k][e + 1] = t.y;
          v[k][e + 2] = t.z;
          v[k][e + 3] = t.w;
        }
      } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) v[k][e] = __ldg(src + e);
      }
    }
#pragma unroll
    for (int k = 0; k < NB; ++k)
      if (i0 + k * WPR >= count) w[k] = -INFINITY;
  };
  // round one: this lane's share of the lse values, and the warp's first batch
  float lv[kLse];
  {
    int64_t at[kLse];
#pragma unroll
    for (int j = 0; j < kLse; ++j) at[j] = slot_of(min(lane + 32 * j, count - 1)) * R + r;
#pragma unroll
    for (int j = 0; j < kLse; ++j) lv[j] = __ldg(pl + at[j]);
  }
  load_batch(warp);
  // lse = max + ln sum exp(lse_i - max)
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < kLse; ++j) {
    if (lane + 32 * j >= count) lv[j] = -INFINITY;
    m = fmaxf(m, lv[j]);
  }
  float sum = 0.f;
  for (int i = lane + 32 * kLse; i < count; i += 32) {  // online, past 256 pieces
    const float x = __ldg(pl + slot_of(i) * R + r);
    if (x == -INFINITY) continue;  // an empty partial adds nothing (and -inf - -inf is NaN)
    if (x > m) {
      sum = sum * expf(m - x);
      m = x;
    }
    sum += expf(x - m);
  }
  float mw = m;
  for (int o = 16; o > 0; o >>= 1) mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, o));
  sum = (m == -INFINITY) ? 0.f : sum * expf(m - mw);
#pragma unroll
  for (int j = 0; j < kLse; ++j)
    if (lv[j] != -INFINITY) sum += expf(lv[j] - mw);
  m = mw;
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float lse = (m == -INFINITY) ? -INFINITY : m + logf(sum);
  float acc[VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
  if (m != -INFINITY) {
    for (int i0 = warp;;) {
#pragma unroll
      for (int k = 0; k < NB; ++k) {
        // an empty partial (lse = -inf) has weight 0; whatever its data holds is skipped
        if (w[k] == -INFINITY) continue;
        const float wk = expf(w[k] - lse);
#pragma unroll
        for (int e = 0; e < VEC; ++e) acc[e] += wk * v[k][e];
      }
      i0 += NB * WPR;
      if (i0 >= count) break;
      load_batch(i0);
    }
  }
#pragma unroll
  for (int e = 0; e < VEC; ++e) s_acc[gw][lane * VEC + e] = acc[e];
  // the row group's warps meet (barrier 1 + g, its threads only)
  asm volatile("bar.sync %0, %1;" ::"r"(1 + g), "r"(kGroupThreads) : "memory");
  // every thread finishes W / kGroupThreads (or one) of the chunk's outputs
  for (int x = gt; x < W; x += kGroupThreads) {
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < WPR; ++k) t += s_acc[g * WPR + k][x];
    store_val(out_row + chunk * W + x, t);
  }
  if (gt == 0 && chunk == 0 && lse_out) *lse_out = lse;
}

// Blocks of sequence b on the split plan's cost axis: its length clamped to what its
// page-table row can address, as the attention kernel plans it (which also reports a
// length out of range).
__device__ __forceinline__ int plan_blocks(const AttnParams& p, int b) {
  int L = __ldg(p.seq_lens + b);
  const int64_t cap = p.pt_stride * (int64_t)p.page_size;
  if (L < 0) L = 0;
  if ((int64_t)L > cap) L = (int)cap;
  return (L + kKeyBlock - 1) / kKeyBlock;
}

// Rows of the decode/verify path whose sequence was split over several CTAs, and rows of
// sequences with no key at all (out = 0, lse = -inf). Launched as a programmatic dependent
// of the attention kernel. Before waiting for that grid it works out, from the lengths
// alone, where each of its rows' pieces sit: the lengths are inputs of the call, complete
// before the attention kernel passed its own wait on the kernels before it, and only then
// could this grid start. So after the wait the partials are loaded at once, and rows with
// nothing to merge never wait. A following attention call launched the same way may be
// scheduled from the wait on (its prologue overlaps this kernel, its inputs are read only
// after this grid has completed).
// Minimum resident CTAs an SM (register budget) of each instantiation, measured: two rows
// a CTA want their registers (fewer, with spills, ran slower), one row with eight warps
// wants three CTAs an SM (384 CTAs for 384 rows), the narrow chunks of a few long rows run
// best with the compiler's own choice (0).
template <int VEC, int WPR>
constexpr int kMergeMinBlocks = (VEC == 16 && WPR == 4) ? 2 : ((VEC == 1) ? 0 : 3);

template <int VEC, int WPR, typename OutT>
__global__ void __launch_bounds__(kMergeThreads, kMergeMinBlocks<VEC, WPR>)
    merge_split_kernel(AttnParams p) {
  constexpr int kRowsPerCta = kMergeWarps / WPR;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = warp / WPR, gt = threadIdx.x - g * 32 * WPR;
  const int64_t rows = (int64_t)p.B * p.R;
  const int64_t row0 = (int64_t)blockIdx.x * kRowsPerCta;
  // the cost axis: every sequence as kUnitCost units, then its blocks (none if empty);
  // its length, and the units before each row group's sequence
  int bg[kRowsPerCta];
  long long tot = 0, before[kRowsPerCta];
#pragma unroll
  for (int k = 0; k < kRowsPerCta; ++k) {
    bg[k] = (int)(min(row0 + k, rows - 1) / p.R);
    before[k] = 0;
  }
  for (int x = threadIdx.x; x < p.B; x += kMergeThreads) {
    const int nb = plan_blocks(p, x);
    const long long cost = nb > 0 ? nb + kUnitCost : 0;
    tot += cost;
#pragma unroll
    for (int k = 0; k < kRowsPerCta; ++k)
      if (x < bg[k]) before[k] += cost;
  }
  __shared__ long long s_red[kMergeWarps][1 + kRowsPerCta];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    tot += __shfl_xor_sync(0xffffffffu, tot, o);
#pragma unroll
    for (int k = 0; k < kRowsPerCta; ++k) before[k] += __shfl_xor_sync(0xffffffffu, before[k], o);
  }
  if (lane == 0) {
    s_red[warp][0] = tot;
#pragma unroll
    for (int k = 0; k < kRowsPerCta; ++k) s_red[warp][1 + k] = before[k];
  }
  __syncthreads();
  long long total = 0, pre = 0;
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) {
    total += s_red[w][0];
    pre += s_red[w][1 + g];
  }
  const int64_t row = row0 + g;  // b * R + r
  if (row >= rows) return;
  const int chunk = blockIdx.y;
  static_assert(kRowsPerCta <= 2, "row groups a CTA");
  const int b = (g == 0) ? bg[0] : bg[kRowsPerCta - 1];  // (no indexing of a local array)
  const int64_t r = row % p.R;
  const int num_blocks = plan_blocks(p, b);
  OutT* out_row;
  if constexpr (sizeof(OutT) == 4)
    out_row = p.out_f32 + row * kDV;
  else
    out_row = p.out + row * kDV;
  float* lse_out = p.lse ? p.lse + row : nullptr;
  if (num_blocks == 0) {  // no unit of the attention kernel touches these rows
    for (int x = gt; x < 32 * VEC; x += 32 * WPR) store_val(out_row + chunk * 32 * VEC + x, 0.f);
    if (gt == 0 && chunk == 0 && lse_out) *lse_out = -INFINITY;
    return;
  }
  const int64_t n = p.num_ctas;
  const int64_t first = pre + kUnitCost;  // the sequence's first block
  // pieces: one per CTA range the sequence's blocks overlap (with fewer blocks than CTAs
  // every range holds at most one block)
  const int64_t c0 = range_of(first, total, n);
  const int count = (total >= n) ? (int)(range_of(first + num_blocks - 1, total, n) - c0 + 1)
                                 : num_blocks;
  if (count == 1) return;  // the attention kernel writes this row itself
  // piece 0 takes the second slot of its CTA when that CTA's range began before this
  // sequence's span (in an earlier sequence); every later piece begins its CTA's range
  const int64_t first_odd = (range_lo(c0, total, n) < first - kUnitCost) ? 1 : 0;
  auto slot_of = [&](int i) -> int64_t {
    if (i == 0) return 2 * c0 + first_odd;
    return 2 * ((total >= n) ? c0 + i : range_of(first + i, total, n));
  };
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  merge_row_chunk<VEC, WPR, OutT>(p.part_out, p.part_lse, count, slot_of, r, p.R, chunk, out_row,
                                  lse_out);
}

// Prefill units of an incomplete last round, each run as two halves along the keys: split
// unit v (v = 0 .. split_units - 1, the units handed out last, i.e. the first positions)
// covers positions [pos0, pos0 + npos) with rows j * H + h, and its halves sit in partial
// slots 2v and 2v + 1 of 48 rows. Two rows a CTA (four warps a row), 24 CTAs a unit.
template <typename OutT>
__global__ void __launch_bounds__(kMergeThreads, 2)
    merge_prefill_kernel(AttnParams p, int P, int split_units) {
  constexpr int WPR = 4;
  const int g = (threadIdx.x >> 5) / WPR;
  const int v = blockIdx.x / 24;
  const int r = (blockIdx.x % 24) * 2 + g;  // row of the unit
  const int pos0 = (split_units - 1 - v) * P;
  const int npos = min(P, p.n_q - pos0);
  if (r >= npos * p.H) return;
  const int64_t row = (int64_t)pos0 * p.H + r;
  OutT* out_row;
  if constexpr (sizeof(OutT) == 4)
    out_row = p.out_f32 + row * kDV;
  else
    out_row = p.out + row * kDV;
  float* lse_out = p.lse ? p.lse + row : nullptr;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  merge_row_chunk<16, WPR, OutT>(p.part_out, p.part_lse, 2,
                                 [v](int i) -> int64_t { return 2 * v + i; }, r, p.part_rows, 0,
                                 out_row, lse_out);
}

template <int VEC>
__global__ void __launch_bounds__(kMergeThreads)
    merge_standalone_kernel(const float* po, const float* pl, int S, int64_t R, uint16_t* out,
                            float* lse) {
  const int64_t row = blockIdx.x;
  merge_row_chunk<VEC, kMergeWarps, uint16_t>(po, pl, S, [](int i) -> int64_t { return i; }, row, R,
                                              blockIdx.y, out + row * kDV, lse ? lse + row : nullptr);
}

// Chunk width: whole 512-wide rows when there are rows enough to fill the GPU, narrower
// chunks (more CTAs per row) for the few rows of a long history split over every SM.
int merge_vec(int64_t rows, int num_sms) {
  if (rows >= num_sms) return 16;
  if (rows * 4 >= num_sms) return 4;
  return 1;
}

}  // namespace

cudaError_t launch_merge(const AttnParams& p, cudaStream_t s) {
  const int64_t rows = (int64_t)p.B * p.R;
  const int vec = merge_vec(rows, p.num_ctas);
  // Whole 512-wide rows split over few CTAs each (a batch of short sequences): two rows a
  // CTA, four warps a row (half the CTAs to launch: measured faster). Rows with many pieces
  // (a sequence over more than 8 CTAs) keep eight warps, which load twice the pieces a round.
  const bool two_rows = vec == 16 && p.num_ctas <= 8 * p.B;
  const int64_t per = two_rows ? 2 : 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((rows + per - 1) / per), kDV / (32 * vec));
  cfg.blockDim = dim3(kMergeThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (p.out_f32) {
    if (two_rows) return cudaLaunchKernelEx(&cfg, merge_split_kernel<16, 4, float>, p);
    if (vec == 16) return cudaLaunchKernelEx(&cfg, merge_split_kernel<16, kMergeWarps, float>, p);
    if (vec == 4) return cudaLaunchKernelEx(&cfg, merge_split_kernel<4, kMergeWarps, float>, p);
    return cudaLaunchKernelEx(&cfg, merge_split_kernel<1, kMergeWarps, float>, p);
  }
  if (two_rows) return cudaLaunchKernelEx(&cfg, merge_split_kernel<16, 4, uint16_t>, p);
  if (vec == 16) return cudaLaunchKernelEx(&cfg, merge_split_kernel<16, kMergeWarps, uint16_t>, p);
  if (vec == 4) return cudaLaunchKernelEx(&cfg, merge_split_kernel<4, kMergeWarps, uint16_t>, p);
  return cudaLaunchKernelEx(&cfg, merge_split_kernel<1, kMergeWarps, uint16_t>, p);
}

cudaError_t launch_merge_prefill(const AttnParams& p, int P, int split_units, cudaStream_t s) {
  if (split_units <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)split_units * 24);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  if (p.out_f32) return cudaLaunchKernelEx(&cfg, merge_prefill_kernel<float>, p, P, split_units);
  return cudaLaunchKernelEx(&cfg, merge_prefill_kernel<uint16_t>, p, P, split_units);
}

cudaError_t launch_merge_standalone(const float* part_out, const float* part_lse, int S, int64_t R,
                                    uint16_t* out, float* lse, int num_sms, cudaStream_t s) {
  const int vec = merge_vec(R, num_sms);
  const dim3 grid((unsigned)R, kDV / (32 * vec));
  if (vec == 16)
    merge_standalone_kernel<16><<<grid, kMergeThreads, 0, s>>>(part_out, part_lse, S, R, out, lse);
  else if (vec == 4)
    merge_standalone_kernel<4><<<grid, kMergeThreads, 0, s>>>(part_out, part_lse, S, R, out, lse);
  else
    merge_standalone_kernel<1><<<grid, kMergeThreads, 0, s>>>(part_out, part_lse, S, R, out, lse);
  return cudaGetLastError();
}

}  // namespace mla
