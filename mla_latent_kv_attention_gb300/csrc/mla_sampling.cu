// mla_sampling.cu -- top-k renormalisation of probability rows for speculative verify.
//
// Acceptance sampling after a verify pass draws from the target model's probabilities cut
// down to the k most likely tokens: keep the k largest entries of each row, zero the rest
// and rescale the kept ones to sum to one ("AMD MI355X推理Kimi K3：吞吐量超NVIDIA，首字优化显著",
// section "ROCm适配迎来突破，软件壁垒不再高不可攀"; "在 MI355X 上运行 Kimi K3 的性价比比 B300 更好",
// the part on how the throughput was reached, which builds it from a sort, a masked fill and
// a divide). As with a sort and a mask, the cut is by value: pivot = the k-th largest entry,
// every p_i >= pivot is kept (ties at the pivot are all kept), out_i = p_i / sum of the kept.
// k <= 0 or k >= V keeps the whole row (out = p / sum p). Entries must be >= 0.
//
// A cluster of up to eight CTAs takes one row; each CTA holds its slice of the row in
// registers (32 entries a thread, loaded and stored as 16-byte vectors), so the row is read
// from memory once and written once. The pivot comes from radix selection on the bit
// patterns (for non-negative floats the bit pattern orders like the value): up to three
// passes of 11, 11 and 9 bits below the sign bit, each a count histogram of the next digit
// of the entries still in play, counted by every CTA into its own shared memory. Selection
// stops early when the bin that holds the k-th largest entry is kept whole.
//
// First pass: the 2,048 bins are cut into eight slices of 256. Before the cluster barrier
// each CTA counts its entries per slice; after it every CTA reads the n CTAs' eight slice
// counts, finds the slice that holds the k-th largest entry and adds up that slice's bins
// over the cluster (distributed shared memory) to select the bin in it: about 8 KB of
// remote reads a CTA and one barrier, where every CTA gathering every histogram took 64 KB.
//
// The selected bin usually holds a few dozen entries of the row. When it holds at most
// kCandCap, the cluster skips the remaining passes: every CTA sends the bin's entries (their
// bit patterns) to rank 0, with the sum of its own entries above the bin; rank 0 finds the
// k-th largest among them by two local 10-bit radix passes, adds the kept entries of the bin
// (they share one exponent, so their significands add exactly as integers, in any order) to
// the sums from above the bin, and hands the pivot and the reciprocal of the kept sum to
// every CTA. Otherwise (and when nothing needs selecting) the later passes gather the full
// histograms and the kept sum is one more cluster-wide reduction.
#include <cuda_runtime.h>

#include "mla_internal.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

constexpr int kTkThreads = 512;
constexpr int kTkVec = 8;                                 // 16-byte vectors a thread holds
constexpr int kTkPerThread = 4 * kTkVec;                  // register-resident entries a thread
constexpr int kTkChunk = kTkThreads * kTkPerThread;       // positions a CTA holds (16,384)
constexpr int kTkMaxCluster = 8;
constexpr int kBins = 2048;
constexpr int kSlices = 8;                                // first-pass bins in slices of 256
constexpr int kSliceBins = kBins / kSlices;
constexpr int kWarps = kTkThreads / 32;
constexpr int kPasses = 3;
constexpr int kCandCap = 2 * kBins;  // candidates rank 0 can hold (in the histograms of passes 2, 3)
constexpr int kRankCount = 128;      // up to this many candidates, each is ranked directly
// digit width of a pass, below the sign bit (always 0 in a key): bits 30..20, 19..9, 8..0
__device__ constexpr int digit_width(int pass) { return pass == kPasses - 1 ? 9 : 11; }

struct __align__(16) TkSmem {
  unsigned hist[kPasses][kBins];  // this CTA's counts, one buffer a pass (read remotely)
  unsigned tot[kBins];            // the cluster's counts of every bin of a later pass (rank 0:
                                  // its local passes over the candidates)
  unsigned sel[kSliceBins];       // first pass: the cluster's counts of the selected slice
  unsigned slice_tot[kSlices];    // this CTA's first-pass count in each slice (read remotely)
  unsigned slice_all[kSlices];    // the cluster's count of each slice
  unsigned wsum[kWarps];
  float wsum_f[kWarps];
  float part;                     // this CTA's kept sum (read by the other CTAs)
  int bin;
  unsigned above, in_bin;
  // candidate path: rank 0's slot counter and the CTAs' sums above the bin (written by
  // every CTA into rank 0), the pivot and reciprocal rank 0 hands out, a slot base
  unsigned cta_cnt[kTkMaxCluster];  // first-pass counts of the selected bin, CTAs before this one
  unsigned piv_local;
  float above_w[kTkMaxCluster][kWarps];  // per CTA and warp: the sum above the bin
  unsigned b_pivot;
  float b_inv;
  unsigned long long sig_w[kWarps];
};

// Largest bin b with count(bins >= b) >= k, from the totals: writes b, the count of the
// bins above it and its own count. Thread t owns the four bins nbins-4-4t .. nbins-1-4t.
__device__ void select_bin(TkSmem& s, const unsigned* bins, unsigned k, int nbins) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int lo = nbins - 4 - 4 * t;
  uint4 c4 = make_uint4(0u, 0u, 0u, 0u);
  if (lo >= 0) c4 = *reinterpret_cast<const uint4*>(&bins[lo]);
  const unsigned c = c4.x + c4.y + c4.z + c4.w;
  unsigned incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s.wsum[warp] = incl;
  __syncthreads();
  incl += __reduce_add_sync(0xffffffffu, lane < warp ? s.wsum[lane] : 0u);
  unsigned a = incl - c;  // count of the bins above this thread's
  if (a < k && incl >= k) {
    const unsigned v[4] = {c4.w, c4.z, c4.y, c4.x};  // from the top
    int j = 0;
    while (a + v[j] < k) a += v[j++];
    s.bin = lo + 3 - j;
    s.above = a;
    s.in_bin = v[j];
  }
  __syncthreads();
}

// Sum over the block of one float a thread; the result is valid in every thread.
__device__ __forceinline__ float block_sum(TkSmem& s, float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) s.wsum_f[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) t += s.wsum_f[w];
  return t;
}

// The candidate path (see the top of the file). bin: the 12 high bits (sign bit, always 0,
// then bits 30..20) every candidate shares; k: the rank sought among the bin's entries
// (1-based, from the largest). Returns the pivot; *inv_out = 1 / (sum of the kept entries).
template <typename TailKey>
__device__ unsigned candidate_select(TkSmem& s, const unsigned (&key)[kTkPerThread], int64_t tail0,
                                     int64_t tail_step, int lane, int64_t span, TailKey tail_key,
                                     unsigned rank, int n, unsigned bin, unsigned k, float* inv_out) {
  const int t = threadIdx.x;
  // this CTA's candidates and its sum above the bin
  unsigned cnt = 0;
  float above = 0.f;
#pragma unroll
  for (int j = 0; j < kTkPerThread; ++j) {
    const unsigned hi = key[j] >> 20;
    cnt += hi == bin;
    if (hi > bin) above += __uint_as_float(key[j]);
  }
  for (int64_t i = tail0 + lane; i < span; i += tail_step) {
    const unsigned kv = tail_key(i);
    cnt += (kv >> 20) == bin;
    if ((kv >> 20) > bin) above += __uint_as_float(kv);
  }
  // Slots in rank 0, in CTA then thread order: the CTAs before this one hold their
  // first-pass counts of the bin (read from their histograms), the warps before this one
  // and the lanes before this one follow. The warp's sum above the bin goes to rank 0 too,
  // which adds the sums in a fixed order.
  const int warp = t >> 5;
  unsigned incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s.wsum[warp] = incl;
  if (t < (int)rank) s.cta_cnt[t] = sm100::ld_dsmem_u32(&s.hist[0][bin], (uint32_t)t);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) above += __shfl_xor_sync(0xffffffffu, above, o);
  if (lane == 0) sm100::st_dsmem_u32(&s.above_w[rank][warp], 0, __float_as_uint(above));
  __syncthreads();
  unsigned pos = incl - cnt;
  for (int w = 0; w < warp; ++w) pos += s.wsum[w];
  for (unsigned r = 0; r < rank; ++r) pos += s.cta_cnt[r];
  unsigned* cand = &s.hist[1][0];  // in rank 0: kCandCap slots
#pragma unroll
  for (int j = 0; j < kTkPerThread; ++j)
    if ((key[j] >> 20) == bin) sm100::st_dsmem_u32(cand + pos++, 0, key[j]);
  for (int64_t i = tail0 + lane; i < span; i += tail_step) {
    const unsigned kv = tail_key(i);
    if ((kv >> 20) == bin) sm100::st_dsmem_u32(cand + pos++, 0, kv);
  }
  sm100::cluster_sync();  // rank 0 holds every candidate and every sum above the bin
  if (rank == 0) {
    const unsigned nc = s.in_bin;  // the cluster's count of the bin: every entry was sent
    unsigned piv = bin << 20;
    unsigned pre = 0;  // selected bits 19..10
    if (nc <= (unsigned)kRankCount) {
      // few candidates: each of the first nc threads counts the candidates above its own;
      // the k-th largest value v is the one with #(> v) < k <= #(>= v) (threads holding an
      // equal value write the same pivot)
      if (t < (int)nc) {
        const unsigned mine = cand[t];
        unsigned gt = 0, ge = 0;
        for (unsigned c = 0; c < nc; ++c) {
          const unsigned x = cand[c];
          gt += x > mine;
          ge += x >= mine;
        }
        if (gt < k && ge >= k) s.piv_local = mine;
      }
      __syncthreads();
      piv = s.piv_local;
    }
    // otherwise two local passes of 10 bits: bits 19..10, then 9..0 of the entries in play
#pragma unroll
    for (int pass = 0; pass < 2 && nc > (unsigned)kRankCount; ++pass) {
      const int shift = pass == 0 ? 10 : 0;
      for (int b = t; b < 1024; b += kTkThreads) s.tot[b] = 0u;
      __syncthreads();
      for (unsigned c = t; c < nc; c += kTkThreads) {
        const unsigned kv = cand[c];
        if (pass == 0 || ((kv >> 10) & 1023u) == pre) atomicAdd(&s.tot[(kv >> shift) & 1023u], 1u);
      }
      __syncthreads();
      select_bin(s, s.tot, k, 1024);
      const unsigned b = (unsigned)s.bin, a = s.above, in = s.in_bin;
      __syncthreads();  // s.bin / s.above / s.in_bin read before anything rewrites them
      k -= a;
      if (pass == 0) {
        pre = b;
        piv |= b << 10;
        if (k == in) break;  // bin kept whole: its lowest pattern is the pivot
      } else {
        piv |= b;
      }
    }
    // kept entries of the bin: one exponent, so the significands add exactly
    const unsigned ex = bin >> 3;  // exponent field, bits 30..23
    unsigned long long sig = 0;
    for (unsigned c = t; c < nc; c += kTkThreads) {
      const unsigned kv = cand[c];
      if (kv >= piv) sig += (kv & 0x7FFFFFu) | (ex != 0 ? 0x800000u : 0u);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sig += __shfl_xor_sync(0xffffffffu, sig, o);
    if (lane == 0) s.sig_w[t >> 5] = sig;
    __syncthreads();
    if (t < 32) {
      // float arithmetic only (float64 is slow on this part): the warps' sums above the bin
      // in a fixed order (four a lane, then a butterfly), then the bin's kept entries
      float a = 0.f;
#pragma unroll
      for (int q = 0; q < (kTkMaxCluster * kWarps) / 32; ++q) {
        const int idx = q * 32 + t;
        if (idx / kWarps < n) a += s.above_w[idx / kWarps][idx % kWarps];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
      if (t == 0) {
        unsigned long long sig_all = 0;
        for (int w = 0; w < kWarps; ++w) sig_all += s.sig_w[w];
        // significand sum times 2^(exponent - 150): one rounding, then an exact scaling
        const float bin_sum = ldexpf(__ull2float_rn(sig_all), (int)(ex != 0 ? ex : 1u) - 150);
        const float inv = 1.f / (a + bin_sum);
        for (int r = 0; r < n; ++r) {
          sm100::st_dsmem_u32(&s.b_pivot, (uint32_t)r, piv);
          sm100::st_dsmem_u32(&s.b_inv, (uint32_t)r, __float_as_uint(inv));
        }
      }
    }
  }
  sm100::cluster_sync();  // every CTA has the pivot and the reciprocal
  *inv_out = s.b_inv;
  return s.b_pivot;
}

__global__ void __launch_bounds__(kTkThreads, 2)
    top_k_renorm_kernel(const float* __restrict__ probs, float* __restrict__ out, int V, int n,
                        const int32_t* __restrict__ top_k, int k_all) {
  __shared__ TkSmem s;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const unsigned rank = sm100::cluster_ctarank();
  const int64_t row = blockIdx.x / n;
  const float* p = probs + row * (int64_t)V;
  float* o = out + row * (int64_t)V;
  // Positions: entry i of the row sits at position i + off from the 16-byte boundary at or
  // below the row's start, so that positions 4v .. 4v + 3 are one aligned vector; the row
  // is positions [off, span). This CTA holds the vectors rank * 4096 + j * 512 + t (a 16-byte
  // vector that holds one entry of the row lies in the row's pages, whatever it holds
  // besides). Positions past the cluster's registers (span > n * kTkChunk, only when n is
  // the maximum) are re-read from memory in every pass, warp by warp.
  const uintptr_t pa = reinterpret_cast<uintptr_t>(p);
  const int off = (int)((pa & 15u) >> 2);
  const float4* p4 = reinterpret_cast<const float4*>(pa - (pa & 15u));
  const int64_t span = (int64_t)off + V;
  const int64_t v0 = (int64_t)rank * (kTkChunk / 4) + t;
  const int64_t tail0 = (int64_t)n * kTkChunk + (int64_t)rank * kTkThreads + (t & ~31);
  const int64_t tail_step = (int64_t)n * kTkThreads;
  unsigned key[kTkPerThread];  // |p| bit patterns; 0 outside the row (counts as a zero entry)
#pragma unroll
  for (int j = 0; j < kTkVec; ++j) {
    const int64_t v = v0 + (int64_t)j * kTkThreads, q0 = 4 * v;
    float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
    if (q0 < span) f = __ldcs(p4 + v);
    const float e4[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
    for (int e = 0; e < 4; ++e)
      key[4 * j + e] = (q0 + e >= off && q0 + e < span) ? (__float_as_uint(e4[e]) & 0x7FFFFFFFu) : 0u;
  }
  auto tail_key = [&](int64_t q) -> unsigned {
    return q < span ? (__float_as_uint(__ldcs(p + (q - off))) & 0x7FFFFFFFu) : 0u;
  };
  // outputs: whole 16-byte vectors where the output row has the input's alignment and all
  // four positions are in the row, single entries elsewhere
  const uintptr_t oa = reinterpret_cast<uintptr_t>(o);
  const bool vec_out = (int)((oa & 15u) >> 2) == off;
  float4* o4 = reinterpret_cast<float4*>(oa - (oa & 15u));
  unsigned written = 0;  // bit j: vector j of this thread was stored early (all zeros)
  const int kk = top_k ? top_k[row] : k_all;
  unsigned pivot = 0;     // lowest kept bit pattern; 0 keeps everything
  bool have_inv = false;  // the candidate path delivered 1 / (kept sum) with the pivot
  float inv = 0.f;
  if (kk > 0 && kk < V) {
    // Zero entries outside the row only ever add zeros below a positive pivot, and a pivot
    // of zero keeps the zeros of the row anyway, so they change no selection.
    for (int b = t; b < kPasses * kBins; b += kTkThreads) (&s.hist[0][0])[b] = 0u;
    __syncthreads();
    // ---- first pass: bits 30..20
    unsigned k = (unsigned)kk;
    {
      unsigned* hist = s.hist[0];
#pragma unroll
      for (int j = 0; j < kTkPerThread; ++j) atomicAdd(&hist[key[j] >> 20], 1u);
      for (int64_t i = tail0 + lane; i < span; i += tail_step) atomicAdd(&hist[tail_key(i) >> 20], 1u);
    }
    __syncthreads();
    {
      // this CTA's count in each 256-bin slice: four bins a thread, two warps a slice
      const uint4 c = *reinterpret_cast<const uint4*>(&s.hist[0][4 * t]);
      const unsigned sum = __reduce_add_sync(0xffffffffu, c.x + c.y + c.z + c.w);
      if (lane == 0) s.wsum[warp] = sum;
      __syncthreads();
      if (t < kSlices) s.slice_tot[t] = s.wsum[2 * t] + s.wsum[2 * t + 1];
    }
    sm100::cluster_sync();  // every CTA's first-pass histogram and slice counts are complete
    // the cluster's count of each slice: eight threads, every CTA's count in one round
    if (t < kSlices) {
      unsigned v[kTkMaxCluster];
#pragma unroll
      for (int r = 0; r < kTkMaxCluster; ++r)
        v[r] = r < n ? sm100::ld_dsmem_u32(&s.slice_tot[t], (uint32_t)r) : 0u;
      unsigned a = 0;
#pragma unroll
      for (int r = 0; r < kTkMaxCluster; ++r) a += v[r];
      s.slice_all[t] = a;
    }
    __syncthreads();
    // the slice that holds the k-th largest entry (slices from the top), then its 256 bins
    // added up over the cluster (64 threads, four bins each, every CTA's counts in one round)
    int S = kSlices - 1;
    unsigned above_sl = 0;
    while (S > 0 && above_sl + s.slice_all[S] < k) above_sl += s.slice_all[S--];
    if (t < kSliceBins / 4) {
      const int b0 = S * kSliceBins + 4 * t;
      uint4 v[kTkMaxCluster];
#pragma unroll
      for (int r = 0; r < kTkMaxCluster; ++r)
        if (r < n) v[r] = sm100::ld_dsmem_v4(&s.hist[0][b0], (uint32_t)r);
      uint4 c = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int r = 0; r < kTkMaxCluster; ++r)
        if (r < n) {
          c.x += v[r].x;
          c.y += v[r].y;
          c.z += v[r].z;
          c.w += v[r].w;
        }
      *reinterpret_cast<uint4*>(&s.sel[4 * t]) = c;
    }
    __syncthreads();
    select_bin(s, s.sel, k - above_sl, kSliceBins);
    unsigned prefix = (unsigned)(S * kSliceBins + s.bin);  // the sign bit (0), then bits 30..20
    k -= above_sl + s.above;
    // Every entry below the selected bin is cut, whatever the rest of the selection finds:
    // whole vectors of such entries are stored (as zeros) now, while the cluster finishes
    // the selection, rather than all at the end.
    if (vec_out) {
#pragma unroll
      for (int j = 0; j < kTkVec; ++j) {
        const int64_t v = v0 + (int64_t)j * kTkThreads, q0 = 4 * v;
        const unsigned hi = max(max(key[4 * j], key[4 * j + 1]), max(key[4 * j + 2], key[4 * j + 3]));
        if (q0 >= off && q0 + 3 < span && (hi >> 20) < prefix) {
          __stcs(o4 + v, make_float4(0.f, 0.f, 0.f, 0.f));
          written |= 1u << j;
        }
      }
    }
    int done = 12;
    if (k == s.in_bin) {
      // the bin is kept whole: its lowest pattern is the pivot
      pivot = prefix << 20;
    } else if (s.in_bin <= (unsigned)kCandCap) {
      pivot = candidate_select(s, key, tail0, tail_step, lane, span, tail_key, rank, n, prefix, k, &inv);
      have_inv = true;
    } else {
      // ---- later passes over the whole cluster histograms (a bin too full for rank 0)
      __syncthreads();  // s.bin / s.above / s.in_bin are read before the next pass writes them
#pragma unroll
      for (int pass = 1; pass < kPasses; ++pass) {
        const int wbits = digit_width(pass), shift = 32 - done - wbits, nbins = 1 << wbits;
        unsigned* hist = s.hist[pass];
        auto count = [&](unsigned kv) {
          if ((kv >> (32 - done)) == prefix) atomicAdd(&hist[(kv >> shift) & (unsigned)(nbins - 1)], 1u);
        };
#pragma unroll
        for (int j = 0; j < kTkPerThread; ++j) count(key[j]);
        for (int64_t i = tail0 + lane; i < span; i += tail_step) count(tail_key(i));
        sm100::cluster_sync();  // every CTA's histogram of this pass is complete
        // four bins a thread; the remote loads go out four CTAs at a time, all issued before
        // the first add
        for (int b4 = t; b4 < nbins / 4; b4 += kTkThreads) {
          uint4 c = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int r0 = 0; r0 < kTkMaxCluster; r0 += 4) {
            uint4 v[4];
#pragma unroll
            for (int r = 0; r < 4; ++r)
              if (r0 + r < n) v[r] = sm100::ld_dsmem_v4(&hist[4 * b4], (uint32_t)(r0 + r));
#pragma unroll
            for (int r = 0; r < 4; ++r)
              if (r0 + r < n) {
                c.x += v[r].x;
                c.y += v[r].y;
                c.z += v[r].z;
                c.w += v[r].w;
              }
          }
          *reinterpret_cast<uint4*>(&s.tot[4 * b4]) = c;
        }
        __syncthreads();
        select_bin(s, s.tot, k, nbins);
        k -= s.above;
        prefix = (prefix << wbits) | (unsigned)s.bin;
        done += wbits;
        // the k-th largest is the smallest entry of the selected bin when the bin is kept
        // whole; the kept set is then every key from the bin's lower end up
        if (k == s.in_bin || pass == kPasses - 1) {
          pivot = prefix << (32 - done);
          break;
        }
        __syncthreads();  // s.bin / s.above / s.in_bin are read before the next pass writes them
      }
    }
  }
  if (!have_inv) {
    float kept = 0.f;
#pragma unroll
    for (int j = 0; j < kTkPerThread; ++j)
      if (key[j] >= pivot) kept += __uint_as_float(key[j]);
    for (int64_t i = tail0 + lane; i < span; i += tail_step) {
      const unsigned kv = tail_key(i);
      if (kv >= pivot) kept += __uint_as_float(kv);
    }
    kept = block_sum(s, kept);
    if (t == 0) s.part = kept;
    sm100::cluster_sync();  // every CTA's part is written (and the last pass's reads are done)
    float total = 0.f;
#pragma unroll
    for (int r0 = 0; r0 < kTkMaxCluster; r0 += 4) {
      float parts[4];
#pragma unroll
      for (int r = 0; r < 4; ++r)
        parts[r] = r0 + r < n ? __uint_as_float(sm100::ld_dsmem_u32(&s.part, (uint32_t)(r0 + r))) : 0.f;
#pragma unroll
      for (int r = 0; r < 4; ++r) total += parts[r];
    }
    inv = 1.f / total;
  }
#pragma unroll
  for (int j = 0; j < kTkVec; ++j) {
    const int64_t v = v0 + (int64_t)j * kTkThreads, q0 = 4 * v;
    if (q0 >= span || ((written >> j) & 1u)) continue;
    float r4[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const unsigned kv = key[4 * j + e];
      r4[e] = kv >= pivot ? __uint_as_float(kv) * inv : 0.f;
    }
    if (vec_out && q0 >= off && q0 + 3 < span) {
      __stcs(o4 + v, make_float4(r4[0], r4[1], r4[2], r4[3]));
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (q0 + e >= off && q0 + e < span) __stcs(o + (q0 + e - off), r4[e]);
    }
  }
  for (int64_t i = tail0 + lane; i < span; i += tail_step) {
    const unsigned kv = tail_key(i);
    __stcs(o + (i - off), kv >= pivot ? __uint_as_float(kv) * inv : 0.f);
  }
  // no CTA leaves while another may still read its shared memory (the candidate path reads
  // none after its last barrier)
  if (!have_inv) sm100::cluster_sync();
}

}  // namespace

cudaError_t launch_top_k_renorm(const float* probs, float* out, int B, int V, const int32_t* top_k,
                                int k_all, cudaStream_t s) {
  // positions: up to three before the row's first entry (16-byte alignment)
  int n = (int)(((int64_t)V + 3 + kTkChunk - 1) / kTkChunk);
  n = n < 1 ? 1 : (n > kTkMaxCluster ? kTkMaxCluster : n);
  if ((int64_t)B * n > 0x7FFFFFFF) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(B * n));
  cfg.blockDim = dim3(kTkThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)n;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, top_k_renorm_kernel, probs, out, V, n, top_k, k_all);
}

}  // namespace mla
