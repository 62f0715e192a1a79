// mla_attn_v0.cu -- straightforward CUDA-core MLA attention over the paged FP8 latent cache.
//
// One CTA handles one unit of work: a block of up to 64 query rows of one sequence and a
// range of keys. Keys are staged 64 at a time in shared memory, scores are FP32 dot
// products over all 576 entries, softmax is online (running max and sum per row), and
// the value accumulation keeps each thread's two output columns for every row in
// registers. Output is final bf16 + lse when the unit covers the whole sequence, else a
// normalised FP32 partial + lse for the merge.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <math.h>

#include "mla_internal.cuh"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kRowTile = 64;
constexpr int kKeys = 64;
constexpr int kQPitch = kD + 8;  // bf16 per staged query row (odd number of 16-byte chunks)

struct SmemV0 {
  uint16_t q[kRowTile][kQPitch];
  uint8_t kv[kKeys][kD];
  float pT[kKeys][kRowTile];  // scores, then probabilities, as [key][row]
  float m[kRowTile], l[kRowTile], alpha[kRowTile];
  int vis_end[kRowTile];
};

__device__ __forceinline__ float e4m3_to_float(uint8_t code) {
  __nv_fp8_e4m3 v;
  v.__x = code;
  return float(v);
}

__device__ __forceinline__ int seq_len_clamped(const AttnParams& p, int b) {
  int L = p.seq_lens[b];
  int64_t cap = p.pt_stride * (int64_t)p.page_size;
  if (L < 0) return 0;
  if ((int64_t)L > cap) return (int)cap;
  return L;
}

template <int RT>
__global__ void __launch_bounds__(kThreads) attn_v0_kernel(AttnParams p, int prefill_T) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  SmemV0& s = *reinterpret_cast<SmemV0*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  int b, row0, nr, key_lo, key_hi, unit = -1;
  bool final_out;
  if (prefill_T > 0) {
    b = 0;
    const int R = p.R;
    row0 = blockIdx.x * kRowTile;
    if (row0 >= R) return;
    nr = min(kRowTile, R - row0);
    int L = p.seq_lens[0];
    int64_t cap = p.pt_stride * (int64_t)p.page_size;
    if (L < 0 || (int64_t)L > cap) {
      if (tid == 0) report(p.hdr, MLA_ERR_BOUNDS);
      L = L < 0 ? 0 : (int)cap;
    }
    const int t_last = (row0 + nr - 1) / p.H;
    key_lo = 0;
    key_hi = max(0, min(L, L - p.n_q + t_last + 1));
    final_out = true;
  } else {
    unit = blockIdx.x;
    if (unit >= p.hdr->num_units) return;
    const Unit un = p.units[unit];
    b = un.b;
    row0 = 0;
    nr = p.R;
    key_lo = un.key_lo;
    key_hi = un.key_hi;
    final_out = p.seqs[b].count == 1;
  }
  const int L = seq_len_clamped(p, b);

  // Stage the query rows and the per-row visibility limit.
  for (int i = tid; i < nr * (kD / 8); i += kThreads) {
    const int r = i / (kD / 8), c = i % (kD / 8);
    const uint4* src = reinterpret_cast<const uint4*>(p.q + ((int64_t)b * p.R + row0 + r) * kD);
    *reinterpret_cast<uint4*>(&s.q[r][c * 8]) = src[c];
  }
  if (tid < kRowTile) {
    const int g = row0 + tid, j = g / p.H;
    s.vis_end[tid] = (tid < nr) ? min(key_hi, L - p.n_q + j + 1) : key_lo;
    s.m[tid] = -INFINITY;
    s.l[tid] = 0.f;
  }

  float o0[RT], o1[RT];
#pragma unroll
  for (int r = 0; r < RT; ++r) o0[r] = o1[r] = 0.f;
  const float score_scale = p.kv_scale * p.sm_scale;

  for (int k0 = key_lo; k0 < key_hi; k0 += kKeys) {
    const int nk = min(kKeys, key_hi - k0);
    __syncthreads();  // previous step done with kv / pT
    for (int i = tid; i < kKeys * (kD / 16); i += kThreads) {
      const int n = i / (kD / 16), c = i % (kD / 16);
      uint4 v = make_uint4(0, 0, 0, 0);
      if (n < nk) {
        const int a = k0 + n;
        const int page = p.page_table[(int64_t)b * p.pt_stride + a / p.page_size];
        if (page >= 0 && page < p.num_pages) {
          const uint4* src = reinterpret_cast<const uint4*>(
              p.pool + ((int64_t)page * p.page_size + a % p.page_size) * kD);
          v = src[c];
        } else if (c == 0) {
          report(p.hdr, MLA_ERR_BOUNDS);
        }
      }
      *reinterpret_cast<uint4*>(&s.kv[n][c * 16]) = v;
    }
    __syncthreads();
    // Scores: pair i -> key n = i / nr, row r = i % nr (rows fastest: broadcast key reads).
    for (int i = tid; i < kKeys * nr; i += kThreads) {
      const int n = i / nr, r = i % nr;
      float sc = -INFINITY;
      if (n < nk && k0 + n < s.vis_end[r]) {
        float acc = 0.f;
        const uint4* qv = reinterpret_cast<const uint4*>(&s.q[r][0]);
        const uint2* kv = reinterpret_cast<const uint2*>(&s.kv[n][0]);
#pragma unroll 4
        for (int c = 0; c < kD / 8; ++c) {
          const uint4 qq = qv[c];
          const uint2 kk = kv[c];
          const uint32_t qw[4] = {qq.x, qq.y, qq.z, qq.w};
          const uint32_t kw[2] = {kk.x, kk.y};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const uint16_t qb = (uint16_t)(qw[e >> 1] >> ((e & 1) * 16));
            const float qf = __uint_as_float(((uint32_t)qb) << 16);
            const uint8_t code = (uint8_t)(kw[e >> 2] >> ((e & 3) * 8));
            acc = fmaf(qf, e4m3_to_float(code), acc);
          }
        }
        sc = acc * score_scale;
      }
      s.pT[n][r] = sc;
    }
    __syncthreads();
    // Online softmax: one warp per row.
    for (int r = warp; r < nr; r += kThreads / 32) {
      const float s0 = s.pT[lane][r], s1 = s.pT[lane + 32][r];
      float tmax = fmaxf(s0, s1);
      for (int o = 16; o > 0; o >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
      const float m_old = s.m[r];
      const float m_new = fmaxf(m_old, tmax);
      float alpha, p0, p1;
      if (m_new == -INFINITY) {
        alpha = 1.f;
        p0 = p1 = 0.f;
      } else {
        alpha = (m_old == -INFINITY) ? 0.f : expf(m_old - m_new);
        p0 = (s0 == -INFINITY) ? 0.f : expf(s0 - m_new);
        p1 = (s1 == -INFINITY) ? 0.f : expf(s1 - m_new);
      }
      s.pT[lane][r] = p0;
      s.pT[lane + 32][r] = p1;
      float psum = p0 + p1;
      for (int o = 16; o > 0; o >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, o);
      if (lane == 0) {
        s.m[r] = m_new;
        s.l[r] = s.l[r] * alpha + psum;
        s.alpha[r] = alpha;
      }
    }
    __syncthreads();
    // Value accumulation: thread owns output columns tid and tid + 256.
#pragma unroll
    for (int r = 0; r < RT; ++r) {
      const float a = (r < nr) ? s.alpha[r] : 1.f;
      o0[r] *= a;
      o1[r] *= a;
    }
    for (int n = 0; n < nk; ++n) {
      const float v0 = e4m3_to_float(s.kv[n][tid]);
      const float v1 = e4m3_to_float(s.kv[n][tid + 256]);
      const float4* pr = reinterpret_cast<const float4*>(&s.pT[n][0]);
#pragma unroll
      for (int r4 = 0; r4 < RT / 4; ++r4) {
        const float4 pp = pr[r4];
        o0[4 * r4 + 0] = fmaf(pp.x, v0, o0[4 * r4 + 0]);
        o1[4 * r4 + 0] = fmaf(pp.x, v1, o1[4 * r4 + 0]);
        o0[4 * r4 + 1] = fmaf(pp.y, v0, o0[4 * r4 + 1]);
        o1[4 * r4 + 1] = fmaf(pp.y, v1, o1[4 * r4 + 1]);
        o0[4 * r4 + 2] = fmaf(pp.z, v0, o0[4 * r4 + 2]);
        o1[4 * r4 + 2] = fmaf(pp.z, v1, o1[4 * r4 + 2]);
        o0[4 * r4 + 3] = fmaf(pp.w, v0, o0[4 * r4 + 3]);
        o1[4 * r4 + 3] = fmaf(pp.w, v1, o1[4 * r4 + 3]);
      }
    }
  }
  __syncthreads();

  // Epilogue.
#pragma unroll
  for (int r = 0; r < RT; ++r) {
    if (r >= nr) break;
    const float l = s.l[r];
    const float inv = (l > 0.f) ? p.kv_scale / l : 0.f;
    const int64_t row = (int64_t)b * p.R + row0 + r;
    if (final_out) {
      p.out[row * kDV + tid] = __bfloat16_as_ushort(__float2bfloat16_rn(o0[r] * inv));
      p.out[row * kDV + tid + 256] = __bfloat16_as_ushort(__float2bfloat16_rn(o1[r] * inv));
    } else {
      float* po = p.part_out + ((int64_t)unit * p.R + r) * kDV;
      po[tid] = o0[r] * inv;
      po[tid + 256] = o1[r] * inv;
    }
  }
  if (tid < nr) {
    const float l = s.l[tid];
    const float lse = (l > 0.f) ? s.m[tid] + logf(l) : -INFINITY;
    if (final_out) {
      if (p.lse) p.lse[(int64_t)b * p.R + row0 + tid] = lse;
    } else {
      p.part_lse[(int64_t)unit * p.R + tid] = lse;
    }
  }
}

template <int RT>
cudaError_t launch_rt(const AttnParams& p, bool prefill, int T, cudaStream_t st) {
  const int smem = (int)sizeof(SmemV0);
  cudaError_t e = cudaFuncSetAttribute(attn_v0_kernel<RT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = prefill ? (unsigned)((p.R + kRowTile - 1) / kRowTile) : (unsigned)p.max_units;
  attn_v0_kernel<RT><<<grid, kThreads, smem, st>>>(p, prefill ? T : 0);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_v0(const AttnParams& p, bool prefill, int T, cudaStream_t s) {
  const int rows = prefill ? kRowTile : p.R;
  if (rows <= 16) return launch_rt<16>(p, prefill, T, s);
  if (rows <= 32) return launch_rt<32>(p, prefill, T, s);
  if (rows <= 48) return launch_rt<48>(p, prefill, T, s);
  return launch_rt<64>(p, prefill, T, s);
}

}  // namespace mla
