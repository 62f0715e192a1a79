// mla_cache.cu -- appending new latent rows to the paged FP8 cache.
//
// The step in front of decode, verify and prefill: the new positions' latent rows (576
// wide: 512 latent + 64 RoPE) are written into their cache slots as e4m3 codes under the
// cache's per-tensor scale, so that the attention kernels read them like every other
// cached row ("MI355X Kimi K2.5 vLLM AITER 7x speedup", section "PR #35850 修复了什么":
// the FP8 KV cache handled natively; "Scaling Kimi K3 on AMD Instinct MI355X", section
// "缓存可复用，还要能一致地恢复": 576 FP8 bytes per position).
//
// code = e4m3(x * inv_scale), both the reciprocal and the product rounded to binary32,
// the conversion rounding to nearest even and saturating at +-448. HBM-bound: 1,152 bytes
// read and 576 written per row, one warp per row, every access 16 bytes wide.
#include <cuda_fp8.h>

#include "mla_internal.cuh"

namespace mla {
namespace {

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

// bf16 pair (lo in the low half) scaled by inv -> two e4m3 codes (lo in the low byte)
__device__ __forceinline__ uint32_t quant2(uint32_t w, float inv) {
  const float lo = __uint_as_float(w << 16) * inv;
  const float hi = __uint_as_float(w & 0xFFFF0000u) * inv;
  return e4m3x2(lo, hi);
}

__global__ void __launch_bounds__(256) cache_append_kernel(uint8_t* __restrict__ pool,
                                                           int64_t pool_rows,
                                                           const uint16_t* __restrict__ x,
                                                           const int64_t* __restrict__ slots,
                                                           int64_t n, float inv,
                                                           unsigned* status) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; i < n; i += nwarps) {
    const int64_t s = slots[i];
    if (s < 0) continue;  // padding: nothing to write
    if (s >= pool_rows) {
      if (lane == 0 && status) atomicCAS(status, 0u, (unsigned)MLA_ERR_BOUNDS);
      continue;
    }
    // 36 groups of 16 values: 32 bytes of bf16 in, 16 bytes of codes out
    const uint4* src = reinterpret_cast<const uint4*>(x + i * kD);
    uint4* dst = reinterpret_cast<uint4*>(pool + s * kD);
    for (int g = lane; g < kD / 16; g += 32) {
      const uint4 a = src[2 * g], b = src[2 * g + 1];
      uint4 c;
      c.x = quant2(a.x, inv) | (quant2(a.y, inv) << 16);
      c.y = quant2(a.z, inv) | (quant2(a.w, inv) << 16);
      c.z = quant2(b.x, inv) | (quant2(b.y, inv) << 16);
      c.w = quant2(b.z, inv) | (quant2(b.w, inv) << 16);
      dst[g] = c;
    }
  }
}

}  // namespace

cudaError_t launch_cache_append(uint8_t* pool, int64_t pool_rows, const uint16_t* x,
                                const int64_t* slots, int64_t n, float inv, unsigned* status,
                                int num_sms, cudaStream_t s) {
  const int64_t blocks = (n * 32 + 255) / 256;  // one warp per row, at most 8 CTAs per SM
  const int grid = (int)(blocks < (int64_t)num_sms * 8 ? blocks : (int64_t)num_sms * 8);
  cache_append_kernel<<<grid, 256, 0, s>>>(pool, pool_rows, x, slots, n, inv, status);
  return cudaGetLastError();
}

}  // namespace mla
