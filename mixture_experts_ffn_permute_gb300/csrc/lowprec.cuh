// FP8 (E4M3) / NVFP4 (E2M1) conversions and the bulk-copy helpers the
// low-precision grouped GEMMs share (grouped_gemm_fp4.cu, grouped_gemm_fp4_pair.cu).
// Lane layouts: the low nibble / low byte is the lower-indexed element, and
// cvt.rn.satfinite.e4m3x2.f32 takes the higher element first.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ptx.cuh"

namespace moe {

__device__ __forceinline__ void bulk_load(void* smem_dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(smem_dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Two E2M1 codes (low nibble = lower element) -> f16x2.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(r)
      : "r"(byte));
  return r;
}

// Two E4M3 codes (low byte = lower element) -> f16x2.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two) {
  uint32_t r;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
      : "=r"(r)
      : "r"(two));
  return r;
}

// (lo, hi) fp32 -> two E4M3 codes, round-to-nearest-even, saturating.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  __half2 x = *reinterpret_cast<__half2*>(&a);
  __half2 y = *reinterpret_cast<__half2*>(&b);
  __half2 z = __hmul2(x, y);
  return *reinterpret_cast<uint32_t*>(&z);
}

}  // namespace moe
