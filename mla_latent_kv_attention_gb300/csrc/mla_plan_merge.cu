// mla_plan_merge.cu -- split-KV planning and the log-sum-exp merge.
//
// Planning: the key axis of every sequence is cut into units of whole 128-key blocks so
// that the number of units is about kUnitsPerSm x SMs and units are balanced in keys.
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

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(AttnParams p, int target_units) {
  __shared__ long long s_ll[32];
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
  long long blocks = 0;
  for (int b = tid; b < p.B; b += blockDim.x) {
    int L = clamp_len(p, b);
    blocks += (L + kKeyBlock - 1) / kKeyBlock;
  }
  long long total = block_reduce(blocks, [](long long a, long long c) { return a + c; }, s_ll);
  int bpu = (int)((total + target_units - 1) / target_units);
  if (bpu < 1) bpu = 1;
  int carry = 0;
  for (int base = 0; base < p.B; base += blockDim.x) {
    const int b = base + tid;
    int L = 0, n = 0;
    if (b < p.B) {
      L = clamp_len(p, b);
      int nb = (L + kKeyBlock - 1) / kKeyBlock;
      n = (nb + bpu - 1) / bpu;
    }
    int chunk_total;
    int incl = block_scan(n, s_i, &chunk_total);
    int first = carry + incl - n;
    if (b < p.B) {
      p.seqs[b] = SeqUnits{first, n};
      for (int k = 0; k < n; ++k) {
        int lo = k * bpu * kKeyBlock;
        int hi = min(L, (k + 1) * bpu * kKeyBlock);
        p.units[first + k] = Unit{b, lo, hi, first + k};
      }
    }
    carry += chunk_total;
    __syncthreads();
  }
  if (tid == 0) {
    p.hdr->num_units = carry;
    p.hdr->blocks_per_unit = bpu;
  }
}

constexpr int kMergeWarps = 4;
constexpr int kMergeThreads = 32 * kMergeWarps;
constexpr int kMergeChunks = kDV / 128;  // one CTA per (row, 128-wide dv chunk)

// Merge one 128-wide dv chunk of one row. Partial u of the row sits at
// po + (base + u * stride) * 512 and pl[base + u * stride]. Every thread scans all the
// lse values itself (they are few and cached); warp w sums partials w, w + 4, ...;
// lane l owns four consecutive outputs.
__device__ void merge_chunk(const float* __restrict__ po, const float* __restrict__ pl,
                            int64_t base, int64_t stride, int count, int chunk,
                            uint16_t* __restrict__ out_row, float* lse_out) {
  __shared__ float4 s_acc[kMergeWarps][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float m = -INFINITY;
#pragma unroll 8
  for (int u = 0; u < count; ++u) m = fmaxf(m, pl[base + (int64_t)u * stride]);
  float sum = 0.f;
  if (m != -INFINITY) {
#pragma unroll 8
    for (int u = 0; u < count; ++u) sum += expf(pl[base + (int64_t)u * stride] - m);
  }
  const float lse = (m == -INFINITY) ? -INFINITY : m + logf(sum);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (m != -INFINITY) {
#pragma unroll 4
    for (int u = warp; u < count; u += kMergeWarps) {
      const int64_t r = base + (int64_t)u * stride;
      const float w = expf(pl[r] - lse);
      if (w == 0.f) continue;  // an empty partial (lse = -inf) holds no data worth reading
      const float4 v = reinterpret_cast<const float4*>(po + r * kDV + chunk * 128)[lane];
      acc.x += w * v.x;
      acc.y += w * v.y;
      acc.z += w * v.z;
      acc.w += w * v.w;
    }
  }
  s_acc[warp][lane] = acc;
  __syncthreads();
  if (warp == 0) {
    float4 t = s_acc[0][lane];
#pragma unroll
    for (int g = 1; g < kMergeWarps; ++g) {
      t.x += s_acc[g][lane].x;
      t.y += s_acc[g][lane].y;
      t.z += s_acc[g][lane].z;
      t.w += s_acc[g][lane].w;
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(t.x, t.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(t.z, t.w);
    uint2 packed;
    packed.x = *reinterpret_cast<unsigned int*>(&lo);
    packed.y = *reinterpret_cast<unsigned int*>(&hi);
    reinterpret_cast<uint2*>(out_row + chunk * 128)[lane] = packed;
  }
  if (threadIdx.x == 0 && chunk == 0 && lse_out) *lse_out = lse;
}

// Rows of the decode/verify path whose sequence has more (or fewer) than one unit.
// Launched as a programmatic dependent of the attention kernel: it waits for that grid.
__global__ void __launch_bounds__(kMergeThreads) merge_split_kernel(AttnParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t row = blockIdx.x;  // b * R + r
  const int chunk = blockIdx.y;
  const int b = (int)(row / p.R), r = (int)(row % p.R);
  const SeqUnits su = p.seqs[b];
  if (su.count == 1) return;  // the attention kernel wrote this row directly
  merge_chunk(p.part_out, p.part_lse, (int64_t)su.first * p.R + r, p.R, su.count, chunk,
              p.out + row * kDV, p.lse ? p.lse + row : nullptr);
}

__global__ void __launch_bounds__(kMergeThreads)
    merge_standalone_kernel(const float* po, const float* pl, int S, int64_t R, uint16_t* out,
                            float* lse) {
  const int64_t row = blockIdx.x;
  merge_chunk(po, pl, row, R, S, blockIdx.y, out + row * kDV, lse ? lse + row : nullptr);
}

__global__ void reset_status_kernel(WsHeader* hdr) { hdr->status = 0; }

}  // namespace

cudaError_t launch_plan(const AttnParams& p, int target_units, cudaStream_t s) {
  plan_kernel<<<1, kPlanThreads, 0, s>>>(p, target_units);
  return cudaGetLastError();
}

cudaError_t launch_merge(const AttnParams& p, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.B * p.R), kMergeChunks);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, merge_split_kernel, p);
}

cudaError_t launch_merge_standalone(const float* part_out, const float* part_lse, int S, int64_t R,
                                    uint16_t* out, float* lse, cudaStream_t s) {
  dim3 grid((unsigned)R, kMergeChunks);
  merge_standalone_kernel<<<grid, kMergeThreads, 0, s>>>(part_out, part_lse, S, R, out, lse);
  return cudaGetLastError();
}

cudaError_t launch_reset_status(WsHeader* hdr, cudaStream_t s) {
  reset_status_kernel<<<1, 1, 0, s>>>(hdr);
  return cudaGetLastError();
}

}  // namespace mla
