// mla_mha_proj.cu -- the up-projection of the MHA-form prefill, on tcgen05.
//
// Keys and values of every head come from the one shared latent ("MI355X Kimi K2.5 vLLM
// AITER 7x speedup", section "PR #35850 修复了什么"): for cached row n and column c of head h,
//     acc[n][h][c] = sum_k latent[n][k] * w_ukv[k][h][c]
// with latent [L][512] bf16 (the rows' e4m3 values, exact) and w_ukv [512][H][256] bf16 (per
// head 128 key columns, then 128 value columns). kvup [L][H][width] receives
//   bf16 form (width 256): kv_scale * acc rounded to bf16, keys and values alike;
//   precise form (width 384): for the key columns acc itself as a bf16 pair, hi = bf16(acc)
//     in columns 0..127 and lo = bf16(acc - hi) in 128..255 (about 16 bits; kv_scale is
//     applied with the softmax scale), for the value columns kv_scale * acc rounded to fp16
//     in 256..383.
//
// One CTA per 128 x 256 output tile. TMA brings 64-wide k-blocks of both operands into a
// two-stage ring (the latent tile K-major, the weight tile MN-major, both 128-byte
// swizzled); one thread issues M = 128, N = 256, K = 16 bf16 MMAs into a 256-column TMEM
// accumulator; the four warps read it back (one row per thread), round as above and store.
// Two CTAs fit an SM, so one tile's epilogue overlaps another's loads.
// Every wait is bounded; a wait that gives up reports MLA_ERR_TIMEOUT in the status word.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mla_internal.cuh"
#include "sm100.cuh"

namespace mla {
namespace {

using namespace sm100;

constexpr int kPM = 128;                    // rows (cached positions) per tile
constexpr int kPN = 256;                    // output columns per tile
constexpr int kPK = 64;                     // k per stage: 128 bytes of bf16, one swizzle row
constexpr int kPKTotal = 512;               // latent width
constexpr int kPStages = 2;
constexpr int kPABytes = kPM * kPK * 2;     // 16 KB
constexpr int kPBBox = kPK * 64 * 2;        // one 64-column weight box: 8 KB
constexpr int kPBBytes = 4 * kPBBox;        // 32 KB
constexpr int kPStage = kPABytes + kPBBytes;
constexpr uint32_t kPTmemCols = 256;
constexpr uint64_t kPWaitNs = 1000000000ull;

struct ProjMisc {
  uint64_t full[kPStages], empty[kPStages], done;
  uint32_t tmem_base;
  int abort;
};

constexpr int kPSmem = kPStages * kPStage + (int)sizeof(ProjMisc) + 1024;
static_assert(2 * kPSmem <= 232448, "two CTAs per SM");

__global__ void __launch_bounds__(128, 2)
    mha_proj_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                    int L, int N, float scale, int precise, uint16_t* __restrict__ out, unsigned* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  ProjMisc* ms = reinterpret_cast<ProjMisc*>(smem + kPStages * kPStage);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles_n = N / kPN;
  const int m0 = (blockIdx.x / tiles_n) * kPM;
  const int n0 = (blockIdx.x % tiles_n) * kPN;
  constexpr int kBlocks = kPKTotal / kPK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(&ms->full[s], 1);
      mbar_init(&ms->empty[s], 1);
    }
    mbar_init(&ms->done, 1);
    ms->abort = 0;
    fence_mbar_init();
    prefetch_tensormap(&map_a);
    prefetch_tensormap(&map_b);
  }
  if (warp == 1) tmem_alloc(&ms->tmem_base, kPTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ms->tmem_base;

  if (warp == 0 && lane == 0) {
    // ---- TMA producer: k-block kb into stage kb % 2 once the MMAs of kb - 2 released it
    for (int kb = 0; kb < kBlocks; ++kb) {
      const int s = kb % kPStages;
      if (kb >= kPStages && !mbar_wait(&ms->empty[s], ((kb / kPStages) - 1) & 1, kPWaitNs)) {
        ms->abort = 1;
        break;
      }
      uint8_t* st = smem + s * kPStage;
      mbar_arrive_expect_tx(&ms->full[s], kPStage);
      tma_load_2d(st, &map_a, kb * kPK, m0, &ms->full[s]);
      for (int j = 0; j < 4; ++j)
        tma_load_2d(st + kPABytes + j * kPBBox, &map_b, n0 + 64 * j, kb * kPK, &ms->full[s]);
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer: bf16 x bf16 -> f32; A (latent) K-major, B (weights) MN-major
    constexpr uint32_t idesc = instr_desc(1, 1, 0, 1, kPM, kPN);
    for (int kb = 0; kb < kBlocks; ++kb) {
      const int s = kb % kPStages;
      if (!mbar_wait(&ms->full[s], (kb / kPStages) & 1, kPWaitNs)) {
        ms->abort = 1;
        break;
      }
      tc_fence_after();
      const uint32_t a = smem_addr(smem + s * kPStage);
      const uint32_t b = a + kPABytes;
#pragma unroll
      for (int kk = 0; kk < kPK / 16; ++kk) {
        // A: 16 k values = 32 bytes along the swizzled row; 8-row groups 1024 bytes apart.
        // B: 16 k rows of 128 bytes; 64-column boxes kPBBox apart, 8-row groups 1024 apart.
        const uint64_t da = smem_desc(a + kk * 32, 16, 1024, Swizzle::k128B);
        const uint64_t db = smem_desc(b + kk * 2048, kPBBox, 1024, Swizzle::k128B);
        mma_f16(tmem, da, db, idesc, (kb | kk) != 0 ? 1u : 0u);
      }
      mma_commit(&ms->empty[s]);
    }
    mma_commit(&ms->done);  // completes once every MMA issued above has
  }
  __syncwarp();

  // ---- epilogue: thread t of warp w holds row m0 + 32 w + t of the tile
  const bool ok = mbar_wait(&ms->done, 0, kPWaitNs) && !*reinterpret_cast<volatile int*>(&ms->abort);
  tc_fence_after();
  const int row = m0 + warp * 32 + lane;
  if (ok) {
    const uint32_t base = tmem + ((uint32_t)(warp * 32) << 16);
    // a tile is one head's 256 columns (n0 = 256 h)
    const int width = precise ? 384 : 256, H = N / kPN;
    uint16_t* dst = out + ((int64_t)row * H + n0 / kPN) * width;
#pragma unroll 1
    for (int c = 0; c < kPN; c += 16) {
      float v[16];
      tmem_ld16(base + c, v);
      tmem_wait_ld();
      uint32_t w[8], lo[8];
      const bool key = c < kPN / 2;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (!precise) {
          const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * e] * scale, v[2 * e + 1] * scale);
          w[e] = *reinterpret_cast<const uint32_t*>(&h);
        } else if (key) {
          const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
          const float2 hf = __bfloat1622float2(h);
          const __nv_bfloat162 l = __floats2bfloat162_rn(v[2 * e] - hf.x, v[2 * e + 1] - hf.y);
          w[e] = *reinterpret_cast<const uint32_t*>(&h);
          lo[e] = *reinterpret_cast<const uint32_t*>(&l);
        } else {
          const __half2 h = __floats2half2_rn(v[2 * e] * scale, v[2 * e + 1] * scale);
          w[e] = *reinterpret_cast<const uint32_t*>(&h);
        }
      }
      if (row < L) {
        // bf16 form: column c; precise form: keys hi at c and lo at 128 + c, values at 128 + c
        uint4* d4 = reinterpret_cast<uint4*>(dst + ((precise && !key) ? c + 128 : c));
        d4[0] = make_uint4(w[0], w[1], w[2], w[3]);
        d4[1] = make_uint4(w[4], w[5], w[6], w[7]);
        if (precise && key) {
          uint4* l4 = reinterpret_cast<uint4*>(dst + 128 + c);
          l4[0] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
          l4[1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
        }
      }
    }
  } else if (threadIdx.x == 0 && status) {
    atomicCAS(status, 0u, (unsigned)MLA_ERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (!ok && threadIdx.x == 0) {  // let loads already in flight land before the CTA leaves
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 50000) {
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kPTmemCols);
  }
}

typedef CUresult (*EncodeFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                             const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                             CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                             CUtensorMapFloatOOBfill);

EncodeFn proj_encoder() {
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

}  // namespace

// latent [L][512] @ w [512][H][256] into kvup [L][H][mha_up_width(precise)] (see the top of
// this file); pointers 16-byte aligned. One launch.
cudaError_t launch_mha_projection(const void* latent, const void* w, void* kvup, int L, int H,
                                  float kv_scale, int precise, unsigned* status, cudaStream_t s) {
  if (L <= 0) return cudaSuccess;
  const int N = H * kPN;
  if (H <= 0) return cudaErrorInvalidValue;
  const EncodeFn encode = proj_encoder();
  if (!encode) return cudaErrorInvalidValue;
  CUtensorMap ma, mb;
  cuuint32_t estr[2] = {1, 1};
  {
    cuuint64_t dims[2] = {(cuuint64_t)kPKTotal, (cuuint64_t)L};
    cuuint64_t strides[1] = {(cuuint64_t)kPKTotal * 2};
    cuuint32_t box[2] = {(cuuint32_t)kPK, (cuuint32_t)kPM};
    if (encode(&ma, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(latent), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[2] = {(cuuint64_t)N, (cuuint64_t)kPKTotal};
    cuuint64_t strides[1] = {(cuuint64_t)N * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)kPK};
    if (encode(&mb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(w), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  cudaError_t e = cudaFuncSetAttribute(mha_proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmem);
  if (e != cudaSuccess) return e;
  const int64_t tiles = (int64_t)((L + kPM - 1) / kPM) * (N / kPN);
  mha_proj_kernel<<<(unsigned)tiles, 128, kPSmem, s>>>(ma, mb, L, N, kv_scale, precise,
                                                        static_cast<uint16_t*>(kvup), status);
  return cudaGetLastError();
}

}  // namespace mla
