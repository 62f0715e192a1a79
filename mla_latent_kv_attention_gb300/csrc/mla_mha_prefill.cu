// mla_mha_prefill.cu -- causal prefill of one sequence in the MHA (non-absorbed) form.
//
// Keys and values of every head come from the one shared latent ("MI355X Kimi K2.5 vLLM
// AITER 7x speedup", section "PR #35850 修复了什么"): key_h(n) = [c_n W_UK_h ; r_n] (192
// wide: 128 up-projected dims, then the 64 RoPE dims every head shares), value_h(n) =
// c_n W_UV_h (128 wide), with c_n the 512-wide latent and r_n the RoPE part of cached row n,
// both dequantised from e4m3 under kv_scale. New position t of the T (the last T of the L
// cached) attends causally: keys n <= L - T + t. In this form the attention costs
// 2 x (192 + 128) flops per (query, key, head) instead of 2 x (576 + 512), at the price of
// one up-projection GEMM over the cached rows.
//
// Three steps:
//   1. mha_dequant_kernel: cached rows -> latent [L][512] bf16 (e4m3 values, exact; the
//      scale goes into the GEMM) and RoPE rows [L][64] bf16 (scaled).
//   2. mha_proj_kernel (mla_mha_proj.cu, tcgen05): kvup [L][H][256] = kv_scale * latent @ W_ukv.
//   3. mha_attn_kernel: flash attention on tcgen05. One persistent CTA per SM walks units
//      of (128 new positions, one head), longest first. Per 128-key tile: S = Q K^T
//      (M = 128 queries, N = 128 keys, K = 192; twelve kind::f16 MMAs) into the TMEM score
//      buffer of the tile's parity. Two softmax warpgroups take the tiles of one parity each,
//      a whole 128-key row a thread, with a running max, sum and O accumulator of their own
//      (the key axis split in two interleaved halves, merged by their maxima once per unit),
//      so no tile needs an exchange between them. Probabilities go back as bf16 over the
//      scores they came from; O_parity += P V with P read from TMEM (A operand) and V from
//      shared memory (MN-major). Lazy rescale: an O is rescaled only when its row maximum
//      grows by more than 2^8.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>

#include "mla_internal.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kBM = 128;                       // new positions per unit
constexpr int kBox = 128 * 128;                // one 64-wide 16-bit box of 128 rows (16 KB)
constexpr int kQBytes = 3 * kBox;              // q: dims 0..63, 64..127, 128..191
constexpr int kStages = 2;                     // key ring and value ring, two buffers each
static_assert(kStages == 2, "s_full / pv_done double as the rings' release barriers");
constexpr int kThreads = 384;                  // warp 0 TMA (q, keys), 1 MMA, 2 TMA (values), 4..11 softmax
constexpr uint32_t kTmemCols = 512;            // S0 at 0, S1 at 128; O0 at 256, O1 at 384
constexpr uint32_t kColO = 256;
constexpr uint64_t kWaitNs = 1000000000ull;    // every wait gives up after 1 s

// The two forms of the attention (the host picks one per call).
//   bf16 (PREC = false): keys [c W_UK ; r] x kv_scale and values in bf16, probabilities in
//     bf16; 128-key tiles of three 64-wide key boxes.
//   precise (PREC = true): keys as a bf16 pair hi + lo of c W_UK and the exact e4m3 RoPE
//     values, all without kv_scale (it goes into the softmax scale), so the scores carry
//     about 16 bits; values (x kv_scale) and probabilities in fp16; 96-key tiles of five
//     key boxes (hi 0..63, hi 64..127, lo 0..63, lo 64..127, RoPE) so that the rings fit.
template <bool PREC>
struct MhaCfg {
  static constexpr int kBN = PREC ? 96 : 128;    // keys per tile
  static constexpr int kKBox = kBN * 128;        // one 64-wide 16-bit box of kBN keys
  static constexpr int kKBytes = (PREC ? 5 : 3) * kKBox;
  static constexpr int kVBytes = 2 * kKBox;      // values: dims 0..63, 64..127
  static constexpr int kOffK = kQBytes;
  static constexpr int kOffV = kOffK + kStages * kKBytes;
  static constexpr int kOffMisc = kOffV + kStages * kVBytes;
  static constexpr int kQKSteps = PREC ? 20 : 12;  // K = 16 MMAs of the scores
  static constexpr int kValCol = PREC ? 256 : 128;  // first value column of a head in kvup
  static constexpr uint32_t kPType = PREC ? 0 : 1;  // instruction type code: f16 : bf16
};
constexpr float kRescale = 8.f;                // log2 growth of a row maximum that forces a rescale

struct Misc {
  // keys are released when their scores MMA completes (s_full), values when their values
  // MMA does (pv_done), so the next keys load while a tile's softmax runs. One commit
  // serves both waiters: every tcgen05.commit costs the issuing thread time.
  uint64_t k_full[kStages], v_full[kStages];
  uint64_t s_full[2], p_full[2], pv_done[2];
  uint64_t q_full, q_free;
  uint64_t pair_bar;  // bounded barrier of the two softmax warpgroups (256 arrivals)
  uint32_t tmem_base;
  int abort;
  unsigned status;
  float red_max[2][2][kBM];  // [tile parity][warpgroup][row]
  float red_sum[2][kBM];
};

template <bool PREC>
constexpr int mha_smem_bytes() {
  return MhaCfg<PREC>::kOffMisc + (int)sizeof(Misc) + 1024;  // + alignment slack
}
static_assert(mha_smem_bytes<false>() <= 232448 && mha_smem_bytes<true>() <= 232448, "shared memory");

// 2^x on the SFU (the PTX instruction; inputs are <= 0 or -inf here)
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct MhaParams {
  int L, T, H;
  int bn;            // keys per tile (MhaCfg<PREC>::kBN)
  float scale_log2;  // sm_scale * log2(e) (precise form: times kv_scale too)
  uint16_t* out;     // [T][H][128]
  float* lse;        // [T][H] or null
  unsigned* status;  // [gridDim.x]
  WsHeader* hdr;
  float* part_out;   // [chunks][2][128][128]: normalised partial outputs of split units
  float* part_lse;   // [chunks][2][128]
};

__device__ __forceinline__ void report(Misc* m, mla_status_t code) {
  atomicCAS(&m->status, 0u, (unsigned)code);
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Misc* m) {
  if (mbar_wait(bar, parity, kWaitNs)) return true;
  m->abort = 1;
  report(m, MLA_ERR_TIMEOUT);
  return false;
}

// Units: a pair of adjacent query tiles (2i, 2i+1) of one head, taken by two neighbouring
// CTAs 2c and 2c + 1 (rank 0 the later tile, rank 1 the earlier), which stream the same key
// and value tiles, each into its own shared memory (the second read of a tile is served by
// L2). The pair covers the later tile's keys; for the earlier tile the extra last tile is
// fully masked. Pairs are
// ordered longest first and dealt to the clusters in a snake: round r gives pair r*G + c to
// cluster c for even r and to cluster G-1-c for odd r. With an odd number of query tiles
// the last pair holds one tile, which rank 1 repeats without writing it.
struct Unit {
  int q0, h, ntiles;
  bool write;
};

__device__ __forceinline__ int num_qtiles(const MhaParams& p) { return (p.T + kBM - 1) / kBM; }
__device__ __forceinline__ int num_pairs(const MhaParams& p) { return (num_qtiles(p) + 1) / 2; }

__device__ __forceinline__ Unit unit_at(const MhaParams& p, int u, int rank, int bn) {
  const int nq = num_qtiles(p);
  const int qp = num_pairs(p) - 1 - u / p.H;
  const int hi = min(2 * qp + 1, nq - 1);         // the pair's later query tile
  Unit x;
  x.h = u % p.H;
  x.q0 = (rank == 0 ? hi : 2 * qp) * kBM;
  x.write = rank == 0 || hi != 2 * qp;
  const int last = min(hi * kBM + kBM, p.T) - 1;  // last new position of the later tile
  const int keys = p.L - p.T + last + 1;           // keys it sees
  x.ntiles = (keys + bn - 1) / bn;
  return x;
}

__device__ __forceinline__ int unit_of(int r, int c, int G) {
  return r * G + ((r & 1) ? G - 1 - c : c);
}

// The work of a cluster: whole units for the full rounds of the snake; the units left over
// for a last, part-full round are cut along the key axis instead, into as many chunks as
// fit one per cluster (chunk c of leftover unit c % lo: key tiles [kc n / nch,
// (kc + 1) n / nch), kc = c / lo), each writing a normalised partial and its LSE to slot
// c, merged afterwards. This keeps every cluster busy to the end.
struct Split {
  int full_rounds, leftover, chunks_per_unit;  // chunks_per_unit < 2: leftovers run whole
};

__host__ __device__ __forceinline__ int mha_ntiles(int L, int T, int hi_tile, int bn) {
  const int last = (hi_tile * kBM + kBM < T ? hi_tile * kBM + kBM : T) - 1;
  return (L - T + last + 1 + bn - 1) / bn;
}

__host__ __device__ __forceinline__ Split split_of(int L, int T, int H, int clusters, int bn) {
  const int nq = (T + kBM - 1) / kBM, npairs = (nq + 1) / 2;
  const int U = npairs * H;
  Split sp;
  sp.full_rounds = U / clusters;
  sp.leftover = U % clusters;
  sp.chunks_per_unit = 1;
  if (sp.leftover > 0) {
    // the last unit (the smallest pair, 2 * 0 and 1) bounds how finely a unit can be cut
    const int fewest = mha_ntiles(L, T, nq > 1 ? 1 : 0, bn);
    const int c = clusters / sp.leftover;
    sp.chunks_per_unit = c < fewest ? c : fewest;
  }
  return sp;
}

struct Work {
  Unit x;
  int j0, j1;  // key tiles [j0, j1)
  int slot;    // -1: the whole unit, written as the final output; else a partial slot
  bool valid;
};

__device__ __forceinline__ Work work_at(const MhaParams& p, const Split& sp, int i, int c, int NC,
                                        int rank, int bn) {
  Work w;
  w.valid = false;
  w.slot = -1;
  if (i < sp.full_rounds) {
    w.x = unit_at(p, unit_of(i, c, NC), rank, bn);
    w.j0 = 0;
    w.j1 = w.x.ntiles;
    w.valid = true;
    return w;
  }
  if (i > sp.full_rounds || sp.leftover == 0) return w;
  const int base = sp.full_rounds * NC;
  if (sp.chunks_per_unit < 2) {
    if (c >= sp.leftover) return w;
    w.x = unit_at(p, base + c, rank, bn);
    w.j0 = 0;
    w.j1 = w.x.ntiles;
    w.valid = true;
    return w;
  }
  if (c >= sp.leftover * sp.chunks_per_unit) return w;
  const int lu = c % sp.leftover, kc = c / sp.leftover;
  w.x = unit_at(p, base + lu, rank, bn);
  w.j0 = kc * w.x.ntiles / sp.chunks_per_unit;
  w.j1 = (kc + 1) * w.x.ntiles / sp.chunks_per_unit;
  w.slot = c;
  w.valid = true;
  return w;
}

template <bool PREC>
__global__ void __launch_bounds__(kThreads, 1)
    mha_attn_kernel(const MhaParams p, const __grid_constant__ CUtensorMap map_q,
                    const __grid_constant__ CUtensorMap map_kv,
                    const __grid_constant__ CUtensorMap map_rope) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  using C = MhaCfg<PREC>;
  constexpr int kBN = C::kBN;
  Misc* ms = reinterpret_cast<Misc*>(smem + C::kOffMisc);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x / 2, c = blockIdx.x / 2;  // pairs of neighbouring CTAs
  const int rank = (int)(blockIdx.x & 1);
  const Split sp = split_of(p.L, p.T, p.H, G, kBN);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ms->k_full[s], 1);
      mbar_init(&ms->v_full[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ms->s_full[i], 1);
      mbar_init(&ms->p_full[i], 128);
      mbar_init(&ms->pv_done[i], 1);
    }
    mbar_init(&ms->q_full, 1);
    mbar_init(&ms->q_free, 1);
    mbar_init(&ms->pair_bar, 256);
    ms->abort = 0;
    ms->status = 0;
    fence_mbar_init();
    prefetch_tensormap(&map_q);
    prefetch_tensormap(&map_kv);
    prefetch_tensormap(&map_rope);
    if (blockIdx.x == 0) p.hdr->num_ctas = gridDim.x + 1;  // + the dequantisation's status word
  }
  if (warp == 1) tmem_alloc(&ms->tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms->tmem_base;

  if (warp == 0) {
    // ---- TMA producer ----
    if (lane == 0) {
      int g = 0, k = 0;
      for (int r = 0;; ++r) {
        const Work wk = work_at(p, sp, r, c, G, rank, kBN);
        if (!wk.valid || ms->abort) break;
        const Unit& x = wk.x;
        if (k > 0 && !wait_or_abort(&ms->q_free, (k - 1) & 1, ms)) break;
        mbar_arrive_expect_tx(&ms->q_full, kQBytes);
        for (int b = 0; b < 3; ++b) tma_load_3d(smem + b * kBox, &map_q, 64 * b, x.h, x.q0, &ms->q_full);
        bool ok = true;
        for (int j = wk.j0; j < wk.j1; ++j, ++g) {
          const int s = g & 1;
          if (g >= 2 && !(ok = wait_or_abort(&ms->s_full[s], ((g >> 1) & 1) ^ 1, ms))) break;
          uint8_t* kb = smem + C::kOffK + s * C::kKBytes;
          mbar_arrive_expect_tx(&ms->k_full[s], C::kKBytes);
          const int n0 = j * kBN;
          // the up-projected boxes (bf16: two; precise: hi, hi, lo, lo), then RoPE
          constexpr int kUp = PREC ? 4 : 2;
#pragma unroll
          for (int bx = 0; bx < kUp; ++bx)
            tma_load_3d(kb + bx * C::kKBox, &map_kv, 64 * bx, x.h, n0, &ms->k_full[s]);
          tma_load_2d(kb + kUp * C::kKBox, &map_rope, 0, n0, &ms->k_full[s]);
        }
        if (!ok) break;
        ++k;
      }
    }
  } else if (warp == 2) {
    // ---- TMA producer of the values ----
    if (lane == 0) {
      int g = 0;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const Work wk = work_at(p, sp, r, c, G, rank, kBN);
        if (!wk.valid || ms->abort) break;
        const Unit& x = wk.x;
        for (int j = wk.j0; j < wk.j1; ++j, ++g) {
          const int s = g & 1;
          if (g >= 2 && !(ok = wait_or_abort(&ms->pv_done[s], ((g >> 1) & 1) ^ 1, ms))) break;
          uint8_t* vb = smem + C::kOffV + s * C::kVBytes;
          mbar_arrive_expect_tx(&ms->v_full[s], C::kVBytes);
          tma_load_3d(vb, &map_kv, C::kValCol, x.h, j * kBN, &ms->v_full[s]);
          tma_load_3d(vb + C::kKBox, &map_kv, C::kValCol + 64, x.h, j * kBN, &ms->v_full[s]);
        }
      }
    }
  } else if (warp == 1) {
    // ---- MMA issuer ----
    if (lane == 0) {
      constexpr uint32_t idesc_qk = instr_desc(1, 1, 0, 0, 128, kBN);  // bf16, both K-major
      // P from TMEM, V MN-major from shared memory (both bf16, or both f16 when precise)
      constexpr uint32_t idesc_pv = instr_desc(C::kPType, C::kPType, 0, 1, 128, 128);
      const uint32_t q_addr = smem_addr(smem);
      const uint32_t k_base = smem_addr(smem + C::kOffK);
      const uint32_t v_base = smem_addr(smem + C::kOffV);
      // values MMA of tile gx: P from the score buffer of parity gx & 1 into that parity's
      // O accumulator; `first`: the first tile of this parity in the unit
      auto pv = [&](int gx, bool first) -> bool {
        if (!wait_or_abort(&ms->p_full[gx & 1], (gx >> 1) & 1, ms)) return false;
        if (!wait_or_abort(&ms->v_full[gx & 1], (gx >> 1) & 1, ms)) return false;
        tc_fence_after();
        const uint32_t v_addr = v_base + (gx & 1) * C::kVBytes;
        const uint32_t pcol = tmem + (gx & 1) * 128;
        const uint32_t ocol = tmem + kColO + (gx & 1) * 128;
#pragma unroll
        for (int ks = 0; ks < kBN / 16; ++ks) {
          const uint64_t b = smem_desc(v_addr + ks * 2048, C::kKBox, 1024, Swizzle::k128B);
          mma_f16_tmem_a(ocol, pcol + ks * 8, b, idesc_pv, (first && ks == 0) ? 0u : 1u);
        }
        mma_commit(&ms->pv_done[gx & 1]);
        return true;
      };
      int g = 0, k = 0;
      bool ok = true;
      for (int r = 0; ok; ++r) {
        const Work wk = work_at(p, sp, r, c, G, rank, kBN);
        if (!wk.valid || ms->abort) break;
        const int n = wk.j1 - wk.j0;  // tiles of this work item
        if (!(ok = wait_or_abort(&ms->q_full, k & 1, ms))) break;
        for (int j = 0; j < n; ++j, ++g) {
          const int s = g & 1;
          if (!(ok = wait_or_abort(&ms->k_full[s], (g >> 1) & 1, ms))) break;
          tc_fence_after();
          const uint32_t k_addr = k_base + s * C::kKBytes;
#pragma unroll
          for (int kk = 0; kk < C::kQKSteps; ++kk) {
            // k-step kk: query box qb against key box kb (precise: dims 0..127 against the
            // hi boxes, again against the lo boxes, then the RoPE dims)
            const int qb = PREC ? (kk < 16 ? (kk & 7) >> 2 : 2) : kk >> 2;
            const int kb = PREC ? (kk < 16 ? kk >> 2 : 4) : kk >> 2;
            const uint32_t in_box = (kk & 3) * 32;
            const uint64_t a = smem_desc(q_addr + qb * kBox + in_box, 16, 1024, Swizzle::k128B);
            const uint64_t b = smem_desc(k_addr + kb * C::kKBox + in_box, 16, 1024, Swizzle::k128B);
            mma_f16(tmem + s * 128, a, b, idesc_qk, kk > 0 ? 1u : 0u);
          }
          mma_commit(&ms->s_full[s]);
          if (j == n - 1) mma_commit(&ms->q_free);
          if (j >= 1 && !(ok = pv(g - 1, j <= 2))) break;
        }
        if (!ok) break;
        if (!(ok = pv(g - 1, n <= 2))) break;
        ++k;
      }
    }
  } else if (warp >= 4) {
    // ---- softmax: warpgroup wg takes the tiles of parity wg, a whole 128-key row a thread,
    // with its own running max, sum and O accumulator; the two merge once per unit ----
    const int wg = (warp - 4) >> 2;
    const int row = ((warp & 3) << 5) + lane;  // TMEM lane = query row of the tile
    const uint32_t lane_addr = (uint32_t)((warp & 3) << 5) << 16;
    const uint32_t s_col = tmem + lane_addr + wg * 128;       // this warpgroup's score buffer
    const uint32_t o_col = tmem + lane_addr + kColO + wg * 128;  // and its O accumulator
    const int prefix = p.L - p.T;
    int g = 0, mine = 0, pair_phase = 0;  // mine: tiles of this parity so far (pv_done phases)
    auto pair_sync = [&]() -> bool {
      mbar_arrive(&ms->pair_bar);
      return wait_or_abort(&ms->pair_bar, (pair_phase++) & 1, ms);
    };
    bool ok = true;
    for (int r = 0; ok; ++r) {
      const Work wk = work_at(p, sp, r, c, G, rank, kBN);
      if (!wk.valid || ms->abort) break;
      const Unit& x = wk.x;
      const int t = x.q0 + row;          // new position of this thread's row
      const int last_key = prefix + t;   // keys 0..last_key are visible
      float m_run = -INFINITY, l = 0.f;
      bool have = false;                 // this warpgroup took a tile of the work item
      for (int j = wk.j0; j < wk.j1; ++j, ++g) {
        if ((g & 1) != wg) continue;
        // the k-th tile of this parity is phase k of this parity's barriers
        if (!(ok = wait_or_abort(&ms->s_full[wg], mine & 1, ms))) break;
        // this warpgroup's previous values MMA (it wrote O and read P from the buffer about
        // to be overwritten) finished before these scores were computed; confirm its phase
        if (mine > 0 && !(ok = wait_or_abort(&ms->pv_done[wg], (mine - 1) & 1, ms))) break;
        tc_fence_after();
        const int k0 = j * kBN;
        const bool edge = k0 + kBN - 1 > last_key;  // the causal edge crosses this tile
        // pass 1: the row maximum (log2 units)
        float mt = -INFINITY;
#pragma unroll
        for (int q = 0; q < kBN / 32; ++q) {
          float a[16], b[16];
          tmem_ld16(s_col + 32 * q, a);
          tmem_ld16(s_col + 32 * q + 16, b);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const bool va = !edge || k0 + 32 * q + e <= last_key;
            const bool vb = !edge || k0 + 32 * q + 16 + e <= last_key;
            mt = fmaxf(mt, va ? a[e] : -INFINITY);
            mt = fmaxf(mt, vb ? b[e] : -INFINITY);
          }
        }
        mt *= p.scale_log2;
        if (mt > m_run + kRescale) {  // first tile, or a large jump: rescale this O
          if (have) {
            const float f = ex2(m_run - mt);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              float w[16];
              tmem_ld16(o_col + 16 * q, w);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 16; ++e) w[e] *= f;
              tmem_st16(o_col + 16 * q, w);
            }
            l *= f;
          }
          m_run = mt;
        }
        // pass 2: probabilities, packed two 16-bit values per column over the first kBN / 2
        // score columns (column 16q + i holds keys 32q + 2i, 32q + 2i + 1; chunk q's packed
        // columns only overlap score columns already read)
        float sum = 0.f;
#pragma unroll
        for (int q = 0; q < kBN / 32; ++q) {
          float a[16], b[16];
          tmem_ld16(s_col + 32 * q, a);
          tmem_ld16(s_col + 32 * q + 16, b);
          tmem_wait_ld();
          float pk[16];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            float x0 = a[2 * e] * p.scale_log2 - m_run, x1 = a[2 * e + 1] * p.scale_log2 - m_run;
            float y0 = b[2 * e] * p.scale_log2 - m_run, y1 = b[2 * e + 1] * p.scale_log2 - m_run;
            if (edge) {
              const int kb = k0 + 32 * q + 2 * e;
              if (kb > last_key) x0 = -INFINITY;
              if (kb + 1 > last_key) x1 = -INFINITY;
              if (kb + 16 > last_key) y0 = -INFINITY;
              if (kb + 17 > last_key) y1 = -INFINITY;
            }
            const float p0 = ex2(x0), p1 = ex2(x1), p2 = ex2(y0), p3 = ex2(y1);
            sum += (p0 + p1) + (p2 + p3);
            if constexpr (PREC) {
              const __half2 h0 = __floats2half2_rn(p0, p1), h1 = __floats2half2_rn(p2, p3);
              pk[e] = __uint_as_float(*reinterpret_cast<const uint32_t*>(&h0));
              pk[8 + e] = __uint_as_float(*reinterpret_cast<const uint32_t*>(&h1));
            } else {
              const __nv_bfloat162 h0 = __floats2bfloat162_rn(p0, p1);
              const __nv_bfloat162 h1 = __floats2bfloat162_rn(p2, p3);
              pk[e] = __uint_as_float(*reinterpret_cast<const uint32_t*>(&h0));
              pk[8 + e] = __uint_as_float(*reinterpret_cast<const uint32_t*>(&h1));
            }
          }
          tmem_st16(s_col + 16 * q, pk);
        }
        l += sum;
        have = true;
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&ms->p_full[wg]);
        ++mine;
      }
      if (!ok) break;
      // ---- epilogue: both warpgroups' (m, l, O) merge; warpgroup wg writes dims 64 wg.. ----
      if (have && !(ok = wait_or_abort(&ms->pv_done[wg], (mine - 1) & 1, ms))) break;
      tc_fence_before();
      ms->red_max[0][wg][row] = have ? m_run : -INFINITY;
      ms->red_sum[wg][row] = have ? l : 0.f;
      if (!(ok = pair_sync())) break;
      tc_fence_after();
      const float m0 = ms->red_max[0][0][row], m1 = ms->red_max[0][1][row];
      const float mm = fmaxf(m0, m1);
      const float f0 = (m0 == -INFINITY) ? 0.f : ex2(m0 - mm);
      const float f1 = (m1 == -INFINITY) ? 0.f : ex2(m1 - mm);
      const float lt = ms->red_sum[0][row] * f0 + ms->red_sum[1][row] * f1;
      // a key chunk can hold no visible key for a row: partial 0 with lse -inf (weight 0)
      const float inv = lt > 0.f ? 1.f / lt : 0.f;
      const float w0 = f0 * inv, w1 = f1 * inv;
      uint16_t* orow = p.out + ((int64_t)t * p.H + x.h) * 128 + wg * 64;
      const uint32_t oa = tmem + lane_addr + kColO + wg * 64;  // O0, dims of this warpgroup
      float* prow = wk.slot >= 0
                        ? p.part_out + (((int64_t)wk.slot * 2 + rank) * kBM + row) * 128 + wg * 64
                        : nullptr;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float a[16], b[16];
        tmem_ld16(oa + 16 * q, a);
        tmem_ld16(oa + 128 + 16 * q, b);
        tmem_wait_ld();
        if (prow) {  // a partial of a split unit, float32, normalised by its own sum
#pragma unroll
          for (int e = 0; e < 16; e += 4) {
            float4 v4;
            v4.x = (w0 != 0.f ? a[e] * w0 : 0.f) + (w1 != 0.f ? b[e] * w1 : 0.f);
            v4.y = (w0 != 0.f ? a[e + 1] * w0 : 0.f) + (w1 != 0.f ? b[e + 1] * w1 : 0.f);
            v4.z = (w0 != 0.f ? a[e + 2] * w0 : 0.f) + (w1 != 0.f ? b[e + 2] * w1 : 0.f);
            v4.w = (w0 != 0.f ? a[e + 3] * w0 : 0.f) + (w1 != 0.f ? b[e + 3] * w1 : 0.f);
            *reinterpret_cast<float4*>(prow + 16 * q + e) = v4;
          }
        } else if (x.write && t < p.T) {
          uint32_t pkd[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            // an accumulator that took no tile holds stale values: its weight is exactly 0
            const float v0 = (w0 != 0.f ? a[2 * e] * w0 : 0.f) + (w1 != 0.f ? b[2 * e] * w1 : 0.f);
            const float v1 = (w0 != 0.f ? a[2 * e + 1] * w0 : 0.f) + (w1 != 0.f ? b[2 * e + 1] * w1 : 0.f);
            const __nv_bfloat162 h2 = __floats2bfloat162_rn(v0, v1);
            pkd[e] = *reinterpret_cast<const uint32_t*>(&h2);
          }
          uint4* dst = reinterpret_cast<uint4*>(orow + 16 * q);
          dst[0] = make_uint4(pkd[0], pkd[1], pkd[2], pkd[3]);
          dst[1] = make_uint4(pkd[4], pkd[5], pkd[6], pkd[7]);
        }
      }
      if (wg == 0 && wk.slot >= 0)
        p.part_lse[((int64_t)wk.slot * 2 + rank) * kBM + row] =
            lt > 0.f ? 0.6931471805599453f * (mm + log2f(lt)) : -INFINITY;
      else if (wg == 0 && x.write && t < p.T && p.lse)
        p.lse[(int64_t)t * p.H + x.h] = 0.6931471805599453f * (mm + log2f(lt));
      tc_fence_before();
      if (!(ok = pair_sync())) break;  // both have read the shared (m, l) and both O's
    }
  }

  tc_fence_before();
  __syncthreads();
  // after an abort, give loads already in flight a moment to land
  if (ms->abort && threadIdx.x == 0) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 50000) {
    }
  }
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  if (threadIdx.x == 0) p.status[blockIdx.x] = ms->status;
}

// The split units' partials, merged by their LSE: one warp per query row of a split unit
// (4 of the 128 dims a lane); lse = m + ln sum_c exp(lse_c - m), out = sum_c exp(lse_c -
// lse) out_c.
__global__ void __launch_bounds__(256) mha_chunk_merge_kernel(const MhaParams p, Split sp, int NC) {
  const int wid = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (wid >= sp.leftover * 2 * kBM) return;
  const int lu = wid / (2 * kBM), rank = (wid / kBM) & 1, row = wid % kBM;
  const Unit x = unit_at(p, sp.full_rounds * NC + lu, rank, p.bn);
  const int t = x.q0 + row;
  if (!x.write || t >= p.T) return;
  const int nch = sp.chunks_per_unit;
  float m = -INFINITY;
  for (int kc = 0; kc < nch; ++kc)
    m = fmaxf(m, p.part_lse[((int64_t)(kc * sp.leftover + lu) * 2 + rank) * kBM + row]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float sum = 0.f;
  for (int kc = 0; kc < nch; ++kc) {
    const int64_t sr = ((int64_t)(kc * sp.leftover + lu) * 2 + rank) * kBM + row;
    const float ls = p.part_lse[sr];
    if (ls == -INFINITY) continue;
    const float w = expf(ls - m);
    const float4 v = *reinterpret_cast<const float4*>(p.part_out + sr * 128 + 4 * lane);
    acc.x += w * v.x;
    acc.y += w * v.y;
    acc.z += w * v.z;
    acc.w += w * v.w;
    sum += w;
  }
  const float inv = sum > 0.f ? 1.f / sum : 0.f;
  const __nv_bfloat162 h0 = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  const __nv_bfloat162 h1 = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  *reinterpret_cast<uint2*>(p.out + ((int64_t)t * p.H + x.h) * 128 + 4 * lane) =
      make_uint2(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1));
  if (lane == 0 && p.lse) p.lse[(int64_t)t * p.H + x.h] = sum > 0.f ? m + logf(sum) : -INFINITY;
}

// Cached rows -> latent [L][512] bf16 (the e4m3 values; exact) and RoPE rows [L][64] bf16
// (e4m3 value x rope_scale: kv_scale, one rounding, for the bf16 form; 1, exact, for the
// precise one). One thread per 8 codes of a row.
__global__ void mha_dequant_kernel(const uint8_t* __restrict__ pool, int64_t num_pages,
                                   int page_size, const int32_t* __restrict__ page_table, int L,
                                   float rope_scale, __nv_bfloat16* __restrict__ latent,
                                   __nv_bfloat16* __restrict__ rope, unsigned* status) {
  const int64_t items = (int64_t)L * (kD / 8);
  for (int64_t it = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; it < items;
       it += (int64_t)gridDim.x * blockDim.x) {
    const int n = (int)(it / (kD / 8));
    const int c8 = (int)(it % (kD / 8));
    const int32_t page = page_table[n / page_size];
    uint2 raw = make_uint2(0u, 0u);
    if (page < 0 || page >= num_pages) {
      atomicCAS(status, 0u, (unsigned)MLA_ERR_BOUNDS);
    } else {
      raw = *reinterpret_cast<const uint2*>(pool + ((int64_t)page * page_size + n % page_size) * kD +
                                            c8 * 8);
    }
    float f[8];
    const uint32_t w[2] = {raw.x, raw.y};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(
          (__nv_fp8x2_storage_t)((w[i >> 1] >> (16 * (i & 1))) & 0xFFFFu), __NV_E4M3);
      const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&h));
      f[2 * i] = x.x;
      f[2 * i + 1] = x.y;
    }
    uint32_t o[4];
    if (c8 < kDV / 8) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
        o[i] = *reinterpret_cast<const uint32_t*>(&b);
      }
      *reinterpret_cast<uint4*>(latent + (int64_t)n * kDV + c8 * 8) = make_uint4(o[0], o[1], o[2], o[3]);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * i] * rope_scale, f[2 * i + 1] * rope_scale);
        o[i] = *reinterpret_cast<const uint32_t*>(&b);
      }
      *reinterpret_cast<uint4*>(rope + (int64_t)n * 64 + (c8 - kDV / 8) * 8) =
          make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
}

}  // namespace

typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                             const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                             CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                             CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link-time dependency on
// the driver library).
static EncodeFn tensor_map_encoder() {
  static EncodeFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(ptr);
    else
      cudaGetLastError();
  }
  return fn;
}

// The attention launch of one form: tensor maps over q, kvup and the RoPE rows, the
// attention kernel, and the merge of key-split units when the last round was cut.
template <bool PREC>
static cudaError_t launch_mha_attn(const MhaArgs& a, int grid, cudaStream_t s, int* launches) {
  using C = MhaCfg<PREC>;
  const EncodeFn encode = tensor_map_encoder();
  if (!encode) return cudaErrorInvalidValue;
  CUtensorMap mq, mkv, mr;
  cuuint32_t estr[3] = {1, 1, 1};
  {
    cuuint64_t dims[3] = {192, (cuuint64_t)a.H, (cuuint64_t)a.T};
    cuuint64_t strides[2] = {192 * 2, (cuuint64_t)a.H * 192 * 2};
    cuuint32_t box[3] = {64, 1, 128};
    if (encode(&mq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.q), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    // kvup [L][H][width] 16-bit (precise: hi, lo, then fp16 values; the map moves bytes
    // only, so one 16-bit element type serves all of them)
    const cuuint64_t width = mha_up_width(PREC);
    cuuint64_t dims[3] = {width, (cuuint64_t)a.H, (cuuint64_t)a.L};
    cuuint64_t strides[2] = {width * 2, (cuuint64_t)a.H * width * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)C::kBN};
    if (encode(&mkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.kvup, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[2] = {64, (cuuint64_t)a.L};
    cuuint64_t strides[1] = {64 * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)C::kBN};
    if (encode(&mr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, a.rope, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  MhaParams p;
  p.L = a.L;
  p.T = a.T;
  p.H = a.H;
  p.bn = C::kBN;
  p.scale_log2 = a.sm_scale * (PREC ? a.kv_scale : 1.f) * 1.4426950408889634f;
  p.out = a.out;
  p.lse = a.lse;
  p.status = a.status;
  p.hdr = a.hdr;
  p.part_out = static_cast<float*>(a.part_out);
  p.part_lse = static_cast<float*>(a.part_lse);
  constexpr int smem = mha_smem_bytes<PREC>();
  cudaError_t e = cudaFuncSetAttribute(mha_attn_kernel<PREC>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const bool prof = a.prof_start && a.prof_stop;
  if (prof) cudaEventRecord(a.prof_start, s);
  mha_attn_kernel<PREC><<<grid, kThreads, smem, s>>>(p, mq, mkv, mr);
  e = cudaGetLastError();
  if (e == cudaSuccess) ++*launches;
  if (prof) cudaEventRecord(a.prof_stop, s);
  // the split units' partials (only when the last round was cut into chunks)
  const Split sp = split_of(a.L, a.T, a.H, grid / 2, C::kBN);
  if (e == cudaSuccess && sp.leftover > 0 && sp.chunks_per_unit >= 2) {
    const int warps = sp.leftover * 2 * kBM;
    mha_chunk_merge_kernel<<<(warps + 7) / 8, 256, 0, s>>>(p, sp, grid / 2);
    e = cudaGetLastError();
    if (e == cudaSuccess) ++*launches;
  }
  return e;
}

cudaError_t launch_mha_prefill(const MhaArgs& a, int num_sms, cudaStream_t s, int* launches) {
  const int pairs = (((a.T + kBM - 1) / kBM) + 1) / 2 * a.H;
  const int grid = 2 * std::min(num_sms / 2, pairs);  // pairs of CTAs
  // 1. dequantise (its status word follows the attention CTAs' words and is cleared first);
  //    the precise form keeps the RoPE values exact and applies kv_scale in the softmax
  unsigned* dq_status = a.status + grid;
  cudaError_t e = cudaMemsetAsync(dq_status, 0, sizeof(unsigned), s);
  if (e != cudaSuccess) return e;
  const int64_t items = (int64_t)a.L * (kD / 8);
  const int grid1 = (int)std::min<int64_t>((items + 255) / 256, (int64_t)num_sms * 8);
  mha_dequant_kernel<<<grid1, 256, 0, s>>>(a.pool, a.num_pages, a.page_size, a.page_table, a.L,
                                           a.precise ? 1.f : a.kv_scale,
                                           reinterpret_cast<__nv_bfloat16*>(a.latent),
                                           reinterpret_cast<__nv_bfloat16*>(a.rope), dq_status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ++*launches;
  // 2. up-projection: latent [L][512] @ w_ukv [512][H*256] into kvup [L][H][width]
  e = launch_mha_projection(a.latent, a.w_ukv, a.kvup, a.L, a.H, a.kv_scale, a.precise, dq_status, s);
  if (e != cudaSuccess) return e;
  ++*launches;
  // 3. attention
  return a.precise ? launch_mha_attn<true>(a, grid, s, launches)
                   : launch_mha_attn<false>(a, grid, s, launches);
}

}  // namespace mla
