// mla_decode_tc.cu -- split-KV decode / speculative-verify attention on tcgen05 tensor cores.
//
// Work: one persistent CTA per SM walks the planner's units (keys [key_lo, key_hi) of one
// sequence, all of its query rows). Keys stream through shared memory 128 at a time
// (two 64-position pages, fetched by TMA straight from the paged pool) and every key is
// read from HBM exactly once per unit, whatever the head count or verify depth.
//
// Both contractions run on the FP8 cache bytes as they are, with no dequantisation pass:
//   scores  S^T[key][n] = sum_d code[key][d] * Qt[n][d]      tcgen05 kind::f8f6f4,
//           M = 128 keys, N = 2 x (padded rows), K = 576
//           The bf16 query row, scaled by a power of two, is split exactly into two e4m3
//           terms (bf16 has 8 significant bits, e4m3 4), stacked along N and summed after.
//   values  O^T[dv][n]  += sum_key code[key][dv] * Pt[n][key] tcgen05 kind::f8f6f4,
//           M = 128 dv (x4 chunks), N = rows, K = keys; the same FP8 tile read MN-major
//           The probabilities (scaled by 2^8) are split into three e4m3 terms, which
//           carries 12 significant bits, about what fp16 would.
// Keys sit on the MMA's M side ("swap A/B"): 8-16 heads x 1-4 positions are far below
// M = 128, so the few query rows take the narrow N side and nothing is padded in memory.
// Softmax is online over key tiles; one warpgroup owns one key per thread (its TMEM
// lane), so the running max per row needs a cross-warp reduction each tile.
//
// Roles (256 threads): warp 0 issues TMA, warp 1 owns TMEM and issues MMAs, warps 4-7
// stage queries, run the softmax and write the epilogue. Every wait is bounded.
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
constexpr int kTailOffset = 4 * kChunkBytes;            // 128 keys x 64 bytes, SW64
constexpr int kStageBytes = kTailOffset + 2 * 4096;     // 73,728
constexpr int kThreads = 256;
constexpr int kSoftmaxWarp0 = 4;
constexpr uint64_t kWaitLimitNs = 1000000000ull;        // 1 s
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kPScale = 8.0f;                         // P carried as 2^8 * p

template <int RP>
struct Cfg {
  static constexpr int NQK = 2 * RP;                    // two query terms per row
  static constexpr bool kStackP = RP <= 32;
  static constexpr int OCOLS = kStackP ? 3 * RP : RP;   // O^T columns per dv chunk
  static constexpr int NPV = OCOLS;
  static constexpr int kSCol = 0;                       // S^T buffers: [0, 2 NQK)
  static constexpr int kOCol = 2 * NQK;                 // O^T: 4 chunks of OCOLS
  static constexpr int kTmemUsed = 2 * NQK + 4 * OCOLS;
  static constexpr int kTmemCols = kTmemUsed <= 256 ? 256 : 512;
  static constexpr int kQBytes = NQK * kD;
  static constexpr int kPBytes = 3 * RP * kTileKeys;
  // shared memory layout (offsets from a 1024-aligned base)
  static constexpr int kOffStages = 0;
  static constexpr int kOffP = kStages * kStageBytes;
  static constexpr int kOffQ = kOffP + ((kPBytes + 1023) / 1024) * 1024;
  static constexpr int kOffMisc = kOffQ + kQBytes;
  static_assert(kTmemUsed <= 512, "TMEM budget");
  static_assert(kOffMisc % 16 == 0 && kOffQ % 1024 == 0 && kOffP % 1024 == 0, "alignment");
};

struct Misc {
  // float arrays first: they are read as float4 and must be 16-byte aligned
  alignas(16) float row_scale[48];
  alignas(16) float red[2][48 * 4];  // per-tile warp maxima, [row][warp]
  alignas(16) float lred[4][48];
  alignas(16) float alpha[4][48];    // per-warp copy of this tile's rescale factors
  alignas(16) int row_j[48];         // new-position index j of each row (very negative for padding)
  alignas(8) uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t s_full[2], s_empty[2];
  uint64_t p_full, pv_done, q_full;
  uint64_t wg_bar;  // bounded barrier of the softmax warpgroup (128 arrivals per phase)
  uint32_t tmem_base;
  int abort;
};
static_assert(offsetof(Misc, row_scale) % 16 == 0 && offsetof(Misc, red) % 16 == 0 &&
                  offsetof(Misc, lred) % 16 == 0 && offsetof(Misc, alpha) % 16 == 0,
              "vector-accessed arrays must be 16-byte aligned");
static_assert(offsetof(Misc, kv_full) % 8 == 0, "mbarriers must be 8-byte aligned");

template <int RP>
constexpr int smem_bytes() {
  return Cfg<RP>::kOffMisc + (int)sizeof(Misc) + 1024;
}

struct DecodeArgs {
  AttnParams p;
  int h0, Hs;  // heads [h0, h0 + Hs) handled by this launch
  int rows;    // n_q * Hs (<= RP)
  int total_rows_alloc;
};

__device__ __forceinline__ int seq_len_of(const AttnParams& p, int b) {
  int L = p.seq_lens[b];
  const int64_t cap = p.pt_stride * (int64_t)p.page_size;
  if (L < 0) return 0;
  if ((int64_t)L > cap) return (int)cap;
  return L;
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Misc* m,
                                              const AttnParams& p) {
  if (mbar_wait(bar, parity, kWaitLimitNs)) return true;
  m->abort = 1;
  report(p.hdr, MLA_ERR_TIMEOUT);
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
__device__ __forceinline__ uint32_t f16x2_to_e4m3x2(uint32_t h) {
  uint16_t c;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(c) : "r"(h));
  return c;
}
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t c) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)c));
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

template <int RP>
__global__ void __launch_bounds__(kThreads, 1)
    decode_tc_kernel(const __grid_constant__ DecodeArgs args,
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

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ms->kv_full[s], 1);
      mbar_init(&ms->kv_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ms->s_full[s], 1);
      mbar_init(&ms->s_empty[s], 128);
    }
    mbar_init(&ms->p_full, 128);
    mbar_init(&ms->pv_done, 1);
    mbar_init(&ms->q_full, 128);
    mbar_init(&ms->wg_bar, 128);
    ms->abort = 0;
    for (int r = 0; r < 48; ++r) ms->row_j[r] = (r < args.rows) ? r / args.Hs : -(1 << 30);
    fence_mbar_init();
    prefetch_tensormap(&map_main);
    prefetch_tensormap(&map_tail);
  }
  if (warp == 1) tmem_alloc(&ms->tmem_base, C::kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms->tmem_base;
  // Everything above overlapped the planner (programmatic dependent launch); from here on
  // the plan is read. The merge kernel may launch early and waits for this grid itself.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  const int num_units = p.hdr->num_units;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const int64_t rows64 = p.num_pages * (int64_t)p.page_size;
      const int total_rows = rows64 > 0x7fffff00 ? 0x7fffff00 : (int)rows64;
      uint32_t fill = 0;  // tiles issued so far
      for (int u = blockIdx.x; u < num_units && !aborted(ms); u += gridDim.x) {
        const Unit un = p.units[u];
        for (int k0 = un.key_lo; k0 < un.key_hi; k0 += kTileKeys) {
          const int s = fill % kStages;
          const uint32_t n = fill / kStages;
          if (!wait_or_abort(&ms->kv_empty[s], (n & 1) ^ 1, ms, p)) break;
          uint8_t* st = smem + C::kOffStages + s * kStageBytes;
          mbar_arrive_expect_tx(&ms->kv_full[s], kStageBytes);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int kk = k0 + 64 * h;
            int y = total_rows;  // fully out of range: TMA fills zeros
            if (kk < un.key_hi) {
              const int lp = kk / p.page_size;
              const int phys = p.page_table[(int64_t)un.b * p.pt_stride + lp];
              if (phys >= 0 && phys < p.num_pages)
                y = phys * p.page_size + (kk % p.page_size);
              else
                report(p.hdr, MLA_ERR_BOUNDS);
            }
#pragma unroll
            for (int c = 0; c < 4; ++c)
              tma_load_2d(st + c * kChunkBytes + h * 8192, &map_main, c * 128, y, &ms->kv_full[s]);
            tma_load_2d(st + kTailOffset + h * 4096, &map_tail, 0, y, &ms->kv_full[s]);
          }
          ++fill;
        }
      }
      // Drain: wait (bounded) until the consumer released every stage still holding a load.
      for (uint32_t f = (fill > kStages ? fill - kStages : 0); f < fill; ++f) {
        mbar_wait(&ms->kv_empty[f % kStages], (f / kStages) & 1, kWaitLimitNs);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // Two cursors over this CTA's tiles, polled without blocking: scores (QK) of tile g
    // may run ahead while values (PV) of tile g-1 wait for their probabilities, and a PV
    // is issued the moment its P is ready so its KV stage returns to the producer early.
    if (lane == 0) {
      constexpr uint32_t idesc_qk = instr_desc(0, 0, 0, 0, 128, C::NQK);
      constexpr uint32_t idesc_pv = instr_desc(0, 0, 1, 1, 128, C::NPV);
      const uint32_t q_s = smem_addr(qbuf), p_s = smem_addr(pbuf);
      auto tiles_of = [&](int u) {
        const Unit un = p.units[u];
        return (un.key_hi - un.key_lo + kTileKeys - 1) / kTileKeys;
      };
      // scores cursor
      int qu = blockIdx.x, qt = 0, qn = (qu < num_units) ? tiles_of(qu) : 0;
      uint32_t qg = 0, q_units = 0;
      bool q_ready = false;
      // values cursor
      int pu = blockIdx.x, pt = 0, pn = qn;
      uint32_t pg = 0;
      uint64_t idle_since = globaltimer_ns();
      while (pu < num_units) {
        bool progress = false;
        if (qu < num_units) {
          const int s = qg % kStages, sb = qg & 1;
          bool ready = true;
          if (qt == 0 && !q_ready) {
            q_ready = mbar_try_wait(&ms->q_full, q_units & 1);
            ready = q_ready;
          }
          ready = ready && mbar_try_wait(&ms->kv_full[s], (qg / kStages) & 1) &&
                  mbar_try_wait(&ms->s_empty[sb], ((qg >> 1) & 1) ^ 1);
          if (ready) {
            tc_fence_after();
            const uint32_t st = smem_addr(smem + C::kOffStages + s * kStageBytes);
            const uint32_t d = tmem + C::kSCol + sb * C::NQK;
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t a = smem_desc(st + c * kChunkBytes + kk * 32, 16, 1024, Swizzle::k128B);
                const uint64_t b = smem_desc(q_s + c * (C::NQK * 128) + kk * 32, 16, 1024, Swizzle::k128B);
                mma_f8f6f4(d, a, b, idesc_qk, (c | kk) != 0);
              }
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
              const uint64_t a = smem_desc(st + kTailOffset + kk * 32, 16, 512, Swizzle::k64B);
              const uint64_t b = smem_desc(q_s + 4 * (C::NQK * 128) + kk * 32, 16, 512, Swizzle::k64B);
              mma_f8f6f4(d, a, b, idesc_qk, 1);
            }
            mma_commit(&ms->s_full[sb]);
            ++qg;
            if (++qt == qn) {
              qu += gridDim.x;
              qt = 0;
              q_ready = false;
              ++q_units;
              qn = (qu < num_units) ? tiles_of(qu) : 0;
            }
            progress = true;
          }
        }
        if (pg < qg && mbar_try_wait(&ms->p_full, pg & 1)) {
          tc_fence_after();
          const int s = pg % kStages;
          const uint32_t st = smem_addr(smem + C::kOffStages + s * kStageBytes);
          const bool first = (pt == 0);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint32_t d = tmem + C::kOCol + c * C::OCOLS;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              const uint64_t a = smem_desc(st + c * kChunkBytes + ks * 4096, kChunkBytes, 1024, Swizzle::k128B);
              if (C::kStackP) {
                const uint64_t b = smem_desc(p_s + ks * 512, 128, 2048, Swizzle::kNone);
                mma_f8f6f4(d, a, b, idesc_pv, !first || ks > 0);
              } else {
#pragma unroll
                for (int term = 0; term < 3; ++term) {
                  const uint64_t b = smem_desc(p_s + term * (RP / 16) * 2048 + ks * 512, 128, 2048, Swizzle::kNone);
                  mma_f8f6f4(d, a, b, idesc_pv, !first || ks > 0 || term > 0);
                }
              }
            }
          }
          mma_commit(&ms->kv_empty[s]);
          mma_commit(&ms->pv_done);
          ++pg;
          if (++pt == pn) {
            pu += gridDim.x;
            pt = 0;
            pn = (pu < num_units) ? tiles_of(pu) : 0;
          }
          progress = true;
        }
        if (progress) {
          idle_since = globaltimer_ns();
        } else if (globaltimer_ns() - idle_since > kWaitLimitNs || aborted(ms)) {
          ms->abort = 1;
          report(p.hdr, MLA_ERR_TIMEOUT);
          break;
        }
      }
    }
  } else if (warp >= kSoftmaxWarp0) {
    // ------------------------------------------------------------------ softmax warpgroup
    const int wq = warp - kSoftmaxWarp0;  // TMEM lane quadrant
    const int i = wq * 32 + lane;         // key within the tile == TMEM lane
    const uint32_t lane_addr = (uint32_t)(wq * 32) << 16;
    const int R = args.rows;
    const float kv_scale = p.kv_scale;
    uint32_t tile = 0, pv_waits = 0, wg_phase = 0;
    // Bounded warpgroup barrier: every thread arrives, then waits for the phase.
    auto wg_sync = [&]() -> bool {
      mbar_arrive(&ms->wg_bar);
      const bool good = wait_or_abort(&ms->wg_bar, wg_phase & 1, ms, p);
      ++wg_phase;
      return good;
    };

    // Stage the query rows of unit u as two e4m3 terms with a per-row power-of-two scale.
    auto stage_q = [&](int u) {
      const Unit un = p.units[u];
      for (int r = wq; r < RP; r += 4) {
        float v[18];
        float amax = 0.f;
        const bool real = r < R;
        const int j = real ? r / args.Hs : 0, h = real ? args.h0 + r % args.Hs : 0;
        const uint16_t* src = p.q + (((int64_t)un.b * p.n_q + j) * p.H + h) * kD;
        // lane holds dims [16*lane, 16*lane+16) and, for lane < 4, [512 + 16*lane, ...)
#pragma unroll
        for (int e = 0; e < 18; ++e) v[e] = 0.f;
        if (real) {
          const uint4* s4 = reinterpret_cast<const uint4*>(src);
          uint4 a = s4[2 * lane], bq = s4[2 * lane + 1];
          uint32_t w[8] = {a.x, a.y, a.z, a.w, bq.x, bq.y, bq.z, bq.w};
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = __uint_as_float((w[e >> 1] >> ((e & 1) * 16)) << 16);
        }
        float tail[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) tail[e] = 0.f;
        if (real && lane < 4) {
          const uint4* s4 = reinterpret_cast<const uint4*>(src + 512);
          uint4 a = s4[2 * lane], bq = s4[2 * lane + 1];
          uint32_t w[8] = {a.x, a.y, a.z, a.w, bq.x, bq.y, bq.z, bq.w};
#pragma unroll
          for (int e = 0; e < 16; ++e) tail[e] = __uint_as_float((w[e >> 1] >> ((e & 1) * 16)) << 16);
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) amax = fmaxf(amax, fmaxf(fabsf(v[e]), fabsf(tail[e])));
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        // scale 2^e so that amax * 2^e lies in (224, 448]
        int ex = 0;
        if (amax > 0.f && isfinite(amax)) {
          int fe;
          frexpf(amax, &fe);           // amax = f * 2^fe, f in [0.5, 1)
          ex = 9 - fe;                 // amax * 2^ex in [256, 512) ... adjust below
          if (ldexpf(amax, ex) > 448.f) ex -= 1;
        }
        if (lane == 0) ms->row_scale[r] = real ? p.sm_scale * kv_scale * ldexpf(1.f, -ex) * kLog2e : 0.f;
        // two terms per value, packed 16 codes per 16-byte group
        auto emit = [&](const float* x, int w16) {
          uint32_t t1w[4], t2w[4];
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            const float a0 = ldexpf(x[e], ex), a1 = ldexpf(x[e + 1], ex);
            const uint16_t c1 = to_e4m3x2(a0, a1);
            const float2 b1 = from_e4m3x2(c1);
            const uint16_t c2 = to_e4m3x2(a0 - b1.x, a1 - b1.y);
            const int wi = e >> 2, sh = (e & 2) * 8;
            if ((e & 2) == 0) {
              t1w[wi] = c1;
              t2w[wi] = c2;
            } else {
              t1w[wi] |= (uint32_t)c1 << sh;
              t2w[wi] |= (uint32_t)c2 << sh;
            }
          }
          *reinterpret_cast<uint4*>(qbuf + q_offset<C::NQK>(r, w16)) = make_uint4(t1w[0], t1w[1], t1w[2], t1w[3]);
          *reinterpret_cast<uint4*>(qbuf + q_offset<C::NQK>(RP + r, w16)) = make_uint4(t2w[0], t2w[1], t2w[2], t2w[3]);
        };
        emit(v, lane);
        if (lane < 4) emit(tail, 32 + lane);
      }
      fence_proxy_async_smem();
      const bool good = wg_sync();  // row_scale visible to the whole warpgroup
      mbar_arrive(&ms->q_full);
      return good;
    };

    bool ok = true;
    if (blockIdx.x < num_units) ok = stage_q(blockIdx.x);

    for (int u = blockIdx.x; u < num_units && ok; u += gridDim.x) {
      const Unit un = p.units[u];
      const int L = seq_len_of(p, un.b);
      const int ntiles = (un.key_hi - un.key_lo + kTileKeys - 1) / kTileKeys;
      // last visible key of new position j is L - n_q + j (and the unit ends at key_hi)
      const int lim_cap = un.key_hi - 1;
      const int lim0 = min(lim_cap, L - p.n_q);
      float m[RP], l[RP];
#pragma unroll
      for (int r = 0; r < RP; ++r) {
        m[r] = -INFINITY;
        l[r] = 0.f;
      }
      for (int t = 0; t < ntiles; ++t, ++tile) {
        const int sb = tile & 1;
        const int s = tile % kStages;
        const int k0 = un.key_lo + t * kTileKeys;
        const int kabs = k0 + i;
        if (!(ok = wait_or_abort(&ms->s_full[sb], (tile >> 1) & 1, ms, p))) break;
        tc_fence_after();
        float x[RP];
        {
          const uint32_t base = tmem + lane_addr + C::kSCol + sb * C::NQK;
#pragma unroll
          for (int c = 0; c < RP; c += 16) {
            float a[16], b2[16];
            tmem_ld16(base + c, a);
            tmem_ld16(base + RP + c, b2);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) x[c + e] = a[e] + b2[e];
          }
        }
        tc_fence_before();
        mbar_arrive(&ms->s_empty[sb]);
        // to log2 units (per-row scale folds sm_scale, kv_scale, the query term scale, log2 e)
#pragma unroll
        for (int r = 0; r < RP; r += 4) {
          const float4 sc = *reinterpret_cast<const float4*>(&ms->row_scale[r]);
          x[r] *= sc.x;
          x[r + 1] *= sc.y;
          x[r + 2] *= sc.z;
          x[r + 3] *= sc.w;
        }
        // masking only on tiles that reach past the first new position's last visible key
        if (k0 + kTileKeys - 1 > lim0) {
#pragma unroll
          for (int r = 0; r < RP; ++r) {
            const int lim = min(lim_cap, lim0 + ms->row_j[r]);
            if (kabs > lim) x[r] = -INFINITY;
          }
        }
        // tile max per row: warp max in hardware, then the four warps through shared memory
        float* red = &ms->red[tile & 1][0];
#pragma unroll
        for (int r = 0; r < RP; ++r) {
          const float v = warp_max(x[r]);
          if (lane == 0) red[r * 4 + wq] = v;
        }
        if (!(ok = wg_sync())) break;
        bool need_rescale = false;
        float moff[RP];
#pragma unroll
        for (int r = 0; r < RP; ++r) {
          const float4 t4 = *reinterpret_cast<const float4*>(&red[r * 4]);
          const float tm = fmaxf(fmaxf(t4.x, t4.y), fmaxf(t4.z, t4.w));
          float al = 1.f;
          if (tm > m[r]) {
            al = ex2(m[r] - tm);  // 0 when m was -inf (nothing accumulated yet)
            need_rescale |= (m[r] != -INFINITY);
            l[r] *= al;
            m[r] = tm;
          }
          if (lane == 0) ms->alpha[wq][r] = al;
          moff[r] = (m[r] == -INFINITY) ? 0.f : m[r] - kPScale;
        }
        // p = 2^(x - m + 8) rounded to fp16, carried exactly by three e4m3 terms
        uint32_t w1[RP / 4], w2[RP / 4], w3[RP / 4];
#pragma unroll
        for (int r = 0; r < RP; r += 2) {
          const float p0 = ex2(x[r] - moff[r]);
          const float p1 = ex2(x[r + 1] - moff[r + 1]);
          l[r] += p0;
          l[r + 1] += p1;
          const uint32_t h = f32x2_to_f16x2(p0, p1);
          const uint32_t c1 = f16x2_to_e4m3x2(h);
          const uint32_t r1 = hsub2(h, e4m3x2_to_f16x2(c1));
          const uint32_t c2 = f16x2_to_e4m3x2(r1);
          const uint32_t r2 = hsub2(r1, e4m3x2_to_f16x2(c2));
          const uint32_t c3 = f16x2_to_e4m3x2(r2);
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
        // the previous tile's PV must be done before P and O are touched
        if (t > 0) {
          if (!(ok = wait_or_abort(&ms->pv_done, pv_waits & 1, ms, p))) break;
          ++pv_waits;
          tc_fence_after();
          if (need_rescale) {
            __syncwarp();
            const float* al = &ms->alpha[wq][0];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
#pragma unroll
              for (int cc = 0; cc < C::OCOLS; cc += 16) {
                const uint32_t a = tmem + lane_addr + C::kOCol + c * C::OCOLS + cc;
                float v[16];
                tmem_ld16(a, v);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) v[e] *= al[(cc + e) % RP];
                tmem_st16(a, v);
              }
            }
            tmem_wait_st();
          }
        }
        // keys past this unit's range: zero their V bytes so 0 * garbage cannot be NaN
        if (kabs >= un.key_hi) {
          uint8_t* st = smem + C::kOffStages + s * kStageBytes + (i >> 6) * 8192 + (i & 63) * 128;
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int e = 0; e < 8; ++e)
              reinterpret_cast<uint4*>(st + c * kChunkBytes)[e] = make_uint4(0, 0, 0, 0);
        }
        // P^T: MN-major, 16 rows x 8 keys core matrices; term t, row group g at
        // (t * RP/16 + g) * 2048, key i at (i / 8) * 128 + (i % 8) * 16.
        const int off = (i >> 3) * 128 + (i & 7) * 16;
#pragma unroll
        for (int g = 0; g < RP / 16; ++g) {
          *reinterpret_cast<uint4*>(pbuf + (0 * (RP / 16) + g) * 2048 + off) =
              make_uint4(w1[4 * g], w1[4 * g + 1], w1[4 * g + 2], w1[4 * g + 3]);
          *reinterpret_cast<uint4*>(pbuf + (1 * (RP / 16) + g) * 2048 + off) =
              make_uint4(w2[4 * g], w2[4 * g + 1], w2[4 * g + 2], w2[4 * g + 3]);
          *reinterpret_cast<uint4*>(pbuf + (2 * (RP / 16) + g) * 2048 + off) =
              make_uint4(w3[4 * g], w3[4 * g + 1], w3[4 * g + 2], w3[4 * g + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&ms->p_full);
      }
      if (!ok) break;
      // next unit's queries can go in now: all QK of this unit are complete
      const int un_next = u + gridDim.x;
      if (un_next < num_units && !(ok = stage_q(un_next))) break;
      // ---- epilogue: row sums, then O / l
      float* lred = &ms->lred[0][0];
#pragma unroll
      for (int r = 0; r < RP; ++r) {
        float v = l[r];
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) lred[wq * 48 + r] = v;
      }
      if (!(ok = wg_sync())) break;
      float inv[RP];
#pragma unroll
      for (int r = 0; r < RP; ++r) {
        const float lt = lred[r] + lred[48 + r] + lred[96 + r] + lred[144 + r];
        l[r] = lt;
        inv[r] = lt > 0.f ? kv_scale / lt : 0.f;
      }
      if (!(ok = wait_or_abort(&ms->pv_done, pv_waits & 1, ms, p))) break;
      ++pv_waits;
      tc_fence_after();
      const bool final_out = p.seqs[un.b].count == 1;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        float o[C::OCOLS];
#pragma unroll
        for (int cc = 0; cc < C::OCOLS; cc += 16) {
          float v[16];
          tmem_ld16(tmem + lane_addr + C::kOCol + c * C::OCOLS + cc, v);
#pragma unroll
          for (int e = 0; e < 16; ++e) o[cc + e] = v[e];
        }
        tmem_wait_ld();
#pragma unroll
        for (int r = 0; r < RP; ++r) {
          if (r >= R) break;
          float acc = o[r];
          if (C::kStackP) acc += o[RP + r] + o[2 * RP + r];
          const int j = r / args.Hs, h = args.h0 + r % args.Hs;
          const int64_t orow = ((int64_t)un.b * p.n_q + j) * p.H + h;
          const int dv = c * 128 + i;
          if (final_out) {
            p.out[orow * kDV + dv] = __bfloat16_as_ushort(__float2bfloat16_rn(acc * inv[r]));
          } else {
            p.part_out[((int64_t)u * p.R + j * p.H + h) * kDV + dv] = acc * inv[r];
          }
        }
      }
      tc_fence_before();
      if (i < R) {
        float lt = 0.f, mm = -INFINITY;
#pragma unroll
        for (int r = 0; r < RP; ++r)
          if (r == i) {
            lt = l[r];
            mm = m[r];
          }
        const float lse = (lt > 0.f) ? 0.6931471805599453f * (mm - kPScale + log2f(lt)) : -INFINITY;
        const int j = i / args.Hs, h = args.h0 + i % args.Hs;
        if (final_out) {
          if (p.lse) p.lse[((int64_t)un.b * p.n_q + j) * p.H + h] = lse;
        } else {
          p.part_lse[(int64_t)u * p.R + j * p.H + h] = lse;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
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

template <int RP>
cudaError_t launch_rp(const DecodeArgs& a, const CUtensorMap& mm, const CUtensorMap& mt,
                      int grid, cudaStream_t s) {
  constexpr int smem = smem_bytes<RP>();
  cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<RP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_tc_kernel<RP>, a, mm, mt);
}

}  // namespace

// Decode / verify attention for every unit of the plan. Rows per launch are limited to 48
// (three query terms of 48 rows fit TMEM); 16 heads x 4 positions run as two head halves.
cudaError_t launch_decode_tc(const AttnParams& p, int num_sms, cudaStream_t s, int* launches) {
  CUtensorMap mm, mt;
  if (!encode_pool_maps(p, &mm, &mt)) return cudaErrorInvalidValue;
  const int grid = min(num_sms, p.max_units);
  const int groups = (p.R > 48) ? 2 : 1;
  for (int gi = 0; gi < groups; ++gi) {
    DecodeArgs a;
    a.p = p;
    a.Hs = p.H / groups;
    a.h0 = gi * a.Hs;
    if (gi == groups - 1) a.Hs = p.H - a.h0;
    a.rows = p.n_q * a.Hs;
    a.total_rows_alloc = p.R;
    cudaError_t e;
    if (a.rows <= 16)
      e = launch_rp<16>(a, mm, mt, grid, s);
    else if (a.rows <= 32)
      e = launch_rp<32>(a, mm, mt, grid, s);
    else
      e = launch_rp<48>(a, mm, mt, grid, s);
    if (e != cudaSuccess) return e;
    ++*launches;
  }
  return cudaSuccess;
}

}  // namespace mla
