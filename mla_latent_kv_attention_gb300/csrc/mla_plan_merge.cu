// mla_plan_merge.cu -- split-KV planning and the log-sum-exp merge.
//
// Planning: the key axis of every sequence is cut into units of whole 128-key blocks; the
// blocks of all sequences are shared out evenly, one contiguous range per CTA.
// A long history therefore spreads over all SMs, which is what made the pages' decode
// faster ("Scaling Kimi K3 on AMD Instinct MI355X", section "并行度必须适配真正的形状":
// the long history handed to more work groups), while short batches stay one unit per
// sequence and skip the merge.
//
// Merge: per query row, lse = ln sum_s exp(lse_s) and out = sum_s exp(lse_s - lse) out_s,
// the "merge by normalisation statistics" of position-sharded attention (same page,
// section "缓存可复用，还要能一致地恢复").
#include <cuda_bf16.h>
#include <math.h>

#include "mla_internal.cuh"

namespace mla {

namespace {

constexpr int kPlanThreads = 1024;

// Cached length clamped to what the page table can hold (no status report).
__device__ int clamp_len_quiet(const AttnParams& p, int b) {
  const int L = p.seq_lens[b];
  const int64_t cap = p.pt_stride * (int64_t)p.page_size;
  return L < 0 ? 0 : ((int64_t)L > cap ? (int)cap : L);
}

__device__ int clamp_len(const AttnParams& p, int b) {
  int L = p.seq_lens[b];
  int64_t cap = p.pt_stride * (int64_t)p.page_size;
  if (L < 0) {
    report(p.hdr, MLA_ERR_BOUNDS);
    return 0;
  }
  if ((int64_t)L > cap) {
    report(p.hdr, MLA_ERR_BOUNDS);
    return (int)cap;
  }
  return L;
}

template <typename T, typename Op>
__device__ T block_reduce(T v, Op op, T* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  const int nw = blockDim.x >> 5;
  T r = scratch[0];
  for (int w = 1; w < nw; ++w) r = op(r, scratch[w]);
  return r;
}

// Inclusive scan over the block (blockDim.x threads); *total gets the block sum.
__device__ int block_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  const int nw = blockDim.x >> 5;
  int prefix = 0, all = 0;
  for (int w = 0; w < nw; ++w) {
    if (w < warp) prefix += scratch[w];
    all += scratch[w];
  }
  *total = all;
  return x + prefix;
}

// First block of CTA c's range when `total` blocks are cut into n nearly equal ranges.
__device__ __forceinline__ int64_t range_lo(int64_t c, int64_t total, int64_t n) {
  return c * total / n;
}
// The CTA whose range holds block x: the largest c with range_lo(c) <= x.
__device__ __forceinline__ int64_t range_of(int64_t x, int64_t total, int64_t n) {
  return ((x + 1) * n + total - 1) / total - 1;
}

// Split planning: the 128-key blocks of all sequences, laid end to end, are cut into one
// contiguous range per CTA of nearly equal size; a CTA's range becomes one unit per
// sequence it touches. Every CTA gets the same amount of key traffic, a sequence is split
// only where a range boundary falls inside it, and units are numbered in block order, so
// each sequence's units and each CTA's units are contiguous.
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(AttnParams p) {
  __shared__ int s_i[32];
  // the attention kernel may start its prologue now; it waits for this grid before
  // reading the plan
  asm volatile("griddepcontrol.launch_dependents;");
  const int tid = threadIdx.x;
  // Warm L2 with every query row while the memory system is still quiet: the attention
  // kernel stages them right when its KV stream starts, and then they would queue behind it.
  {
    const char* q = reinterpret_cast<const char*>(p.q);
    const int64_t lines = (int64_t)p.B * p.R * (kD * 2 / 128);
    for (int64_t x = tid; x < lines; x += blockDim.x)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(q + x * 128));
  }
  if (tid == 0) p.hdr->status = 0;  // this call's status word starts clean
  __syncthreads();
  // 1. blocks per sequence -> exclusive prefix in flat block order
  int carry = 0;
  for (int base = 0; base < p.B; base += blockDim.x) {
    const int b = base + tid;
    const int nb = (b < p.B) ? (clamp_len(p, b) + kKeyBlock - 1) / kKeyBlock : 0;
    int chunk_total;
    const int incl = block_scan(nb, s_i, &chunk_total);
    if (b < p.B) p.blk_prefix[b] = carry + incl - nb;
    carry += chunk_total;
    __syncthreads();
  }
  const int64_t total = carry;
  const int64_t n = p.num_ctas;
  if (tid == 0) p.blk_prefix[p.B] = carry;
  __syncthreads();
  // 2. pieces per sequence (one per CTA range it overlaps): counts and first unit index
  int ucarry = 0;
  for (int base = 0; base < p.B; base += blockDim.x) {
    const int b = base + tid;
    int cnt = 0;
    if (b < p.B) {
      const int start = p.blk_prefix[b], nb = p.blk_prefix[b + 1] - start;
      // with at least one block per CTA every range is non-empty; with fewer blocks than
      // CTAs each block is a range of its own
      if (nb > 0)
        cnt = (total >= n) ? (int)(range_of(start + nb - 1, total, n) - range_of(start, total, n) + 1)
                           : nb;
    }
    int chunk_total;
    const int incl = block_scan(cnt, s_i, &chunk_total);
    if (b < p.B) p.seqs[b] = SeqUnits{ucarry + incl - cnt, cnt};
    ucarry += chunk_total;
    __syncthreads();
  }
  const int num_units = ucarry;
  // 3. per CTA range (one thread each): its first unit, and the units it owns: one per
  //    sequence the range touches, numbered in block order
  for (int c = tid; c <= p.num_ctas; c += blockDim.x) {
    const int64_t x0 = range_lo(c, total, n);
    const int64_t x1 = (c < p.num_ctas) ? range_lo(c + 1, total, n) : x0;
    int first = num_units;
    if (x0 < total) {
      int lo = 0, hi = p.B - 1;  // last sequence b with blk_prefix[b] <= x0
      while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (p.blk_prefix[mid] <= x0) lo = mid; else hi = mid - 1;
      }
      // the unit holding block x0 (sequence lo holds it); an empty range owns nothing and
      // points at the next range's first unit
      const int start_lo = p.blk_prefix[lo];
      first = p.seqs[lo].first + ((total >= n)
                                      ? (int)(range_of(x0, total, n) - range_of(start_lo, total, n))
                                      : (int)(x0 - start_lo));
      for (int b = lo; b < p.B && p.blk_prefix[b] < x1; ++b) {
        const int start = p.blk_prefix[b], end = p.blk_prefix[b + 1];
        if (end <= x0 || end == start) continue;
        const int64_t plo = max((int64_t)start, x0), phi = min((int64_t)end, x1);
        const int k = (total >= n) ? (int)(range_of(plo, total, n) - range_of(start, total, n))
                                   : (int)(plo - start);
        const int idx = p.seqs[b].first + k;
        if (phi <= plo) continue;  // an empty range owns nothing
        const int L = clamp_len_quiet(p, b);
        p.units[idx] = Unit{b, (int)(plo - start) * kKeyBlock,
                            min(L, (int)(phi - start) * kKeyBlock), idx};
      }
    }
    p.cta_first[c] = first;
  }
  if (tid == 0) {
    p.hdr->num_units = num_units;
    p.hdr->blocks_per_unit = (int)((total + n - 1) / n);
  }
}

constexpr int kMergeWarps = 8;
constexpr int kMergeThreads = 32 * kMergeWarps;
constexpr int kMergeMaxCached = 1024;  // partial weights kept in shared memory per row

// Merge one dv chunk (W = 4 * 32 or 1 * 32 values) of one row. Partial u of the row sits
// at po + (base + u * stride) * 512 and pl[base + u * stride]. The block reduces the lse
// values together (max, then sum of exponentials) and keeps the weights in shared memory;
// warp w then sums partials w, w + 8, ... with lane l owning VEC consecutive outputs.
template <int VEC>
__device__ void merge_chunk(const float* __restrict__ po, const float* __restrict__ pl,
                            int64_t base, int64_t stride, int count, int chunk,
                            uint16_t* __restrict__ out_row, float* lse_out) {
  constexpr int W = 32 * VEC;  // dv per CTA
  __shared__ float s_red[32];
  __shared__ float s_w[kMergeMaxCached];
  __shared__ float s_acc[kMergeWarps][W];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float m = -INFINITY;
  for (int u = threadIdx.x; u < count; u += blockDim.x) m = fmaxf(m, pl[base + (int64_t)u * stride]);
  m = block_reduce(m, [](float a, float c) { return fmaxf(a, c); }, s_red);
  float sum = 0.f;
  if (m != -INFINITY)
    for (int u = threadIdx.x; u < count; u += blockDim.x) sum += expf(pl[base + (int64_t)u * stride] - m);
  sum = block_reduce(sum, [](float a, float c) { return a + c; }, s_red);
  const float lse = (m == -INFINITY) ? -INFINITY : m + logf(sum);
  const int cached = min(count, kMergeMaxCached);
  for (int u = threadIdx.x; u < cached; u += blockDim.x)
    s_w[u] = (m == -INFINITY) ? 0.f : expf(pl[base + (int64_t)u * stride] - lse);
  __syncthreads();
  float acc[VEC];
#pragma unroll
  for (int e = 0; e < VEC; ++e) acc[e] = 0.f;
#pragma unroll 4
  for (int u = warp; u < count; u += kMergeWarps) {
    const int64_t r = base + (int64_t)u * stride;
    const float w = (u < kMergeMaxCached) ? s_w[u]
                                          : ((m == -INFINITY) ? 0.f : expf(pl[r] - lse));
    if (w == 0.f) continue;  // an empty partial (lse = -inf) holds no data worth reading
    const float* src = po + r * kDV + chunk * W + lane * VEC;
    if (VEC == 4) {
      const float4 v = *reinterpret_cast<const float4*>(src);
      acc[0] += w * v.x;
      acc[VEC > 1 ? 1 : 0] += w * v.y;
      acc[VEC > 2 ? 2 : 0] += w * v.z;
      acc[VEC > 3 ? 3 : 0] += w * v.w;
    } else {
      acc[0] += w * src[0];
    }
  }
#pragma unroll
  for (int e = 0; e < VEC; ++e) s_acc[warp][lane * VEC + e] = acc[e];
  __syncthreads();
  if (warp == 0) {
    float t[VEC];
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      t[e] = 0.f;
#pragma unroll
      for (int g = 0; g < kMergeWarps; ++g) t[e] += s_acc[g][lane * VEC + e];
    }
    uint16_t* dst = out_row + chunk * W + lane * VEC;
#pragma unroll
    for (int e = 0; e < VEC; ++e) dst[e] = __bfloat16_as_ushort(__float2bfloat16_rn(t[e]));
  }
  if (threadIdx.x == 0 && chunk == 0 && lse_out) *lse_out = lse;
}

// Rows of the decode/verify path whose sequence has more (or fewer) than one unit.
// Launched as a programmatic dependent of the attention kernel: it waits for that grid.
template <int VEC>
__global__ void __launch_bounds__(kMergeThreads) merge_split_kernel(AttnParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t row = blockIdx.x;  // b * R + r
  const int chunk = blockIdx.y;
  const int b = (int)(row / p.R), r = (int)(row % p.R);
  const SeqUnits su = p.seqs[b];
  if (su.count == 1) return;  // the attention kernel wrote this row directly
  merge_chunk<VEC>(p.part_out, p.part_lse, (int64_t)su.first * p.R + r, p.R, su.count, chunk,
                   p.out + row * kDV, p.lse ? p.lse + row : nullptr);
}

template <int VEC>
__global__ void __launch_bounds__(kMergeThreads)
    merge_standalone_kernel(const float* po, const float* pl, int S, int64_t R, uint16_t* out,
                            float* lse) {
  const int64_t row = blockIdx.x;
  merge_chunk<VEC>(po, pl, row, R, S, blockIdx.y, out + row * kDV, lse ? lse + row : nullptr);
}

__global__ void reset_status_kernel(WsHeader* hdr) { hdr->status = 0; }

}  // namespace

cudaError_t launch_plan(const AttnParams& p, cudaStream_t s) {
  plan_kernel<<<1, kPlanThreads, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_merge(const AttnParams& p, cudaStream_t s) {
  // few rows (one long sequence): narrow dv chunks so that more CTAs share the partials
  const int rows = p.B * p.R;
  const bool narrow = rows < 128;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)rows, narrow ? kDV / 32 : kDV / 128);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return narrow ? cudaLaunchKernelEx(&cfg, merge_split_kernel<1>, p)
                : cudaLaunchKernelEx(&cfg, merge_split_kernel<4>, p);
}

cudaError_t launch_merge_standalone(const float* part_out, const float* part_lse, int S, int64_t R,
                                    uint16_t* out, float* lse, cudaStream_t s) {
  if (R < 128) {
    merge_standalone_kernel<1><<<dim3((unsigned)R, kDV / 32), kMergeThreads, 0, s>>>(part_out, part_lse, S, R, out, lse);
  } else {
    merge_standalone_kernel<4><<<dim3((unsigned)R, kDV / 128), kMergeThreads, 0, s>>>(part_out, part_lse, S, R, out, lse);
  }
  return cudaGetLastError();
}

cudaError_t launch_reset_status(WsHeader* hdr, cudaStream_t s) {
  reset_status_kernel<<<1, 1, 0, s>>>(hdr);
  return cudaGetLastError();
}

}  // namespace mla
