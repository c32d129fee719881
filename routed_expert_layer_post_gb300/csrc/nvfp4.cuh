// Device helpers for NVFP4 blocks (E2M1 values, one E4M3 scale per 16 values,
// an FP32 scale on top): the block scale and the element codes, each step an
// FP32 operation in a fixed order, so that every kernel that quantizes takes
// the same decisions.
//
// TokenSpeed blog, "Model architecture and precision -> NVFP4 and FP8
// checkpoints": E2M1 weights, an E4M3 scale per 16, an FP32 scale per expert;
// expert inputs quantized in the same format at runtime.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

namespace beam {

__device__ __forceinline__ float e4m3_value(uint32_t code) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(code), __NV_E4M3);
  return __half2float(__half(h));
}

// Scale code of a block with largest magnitude `amax` under FP32 scale g, and
// the FP32 divisor s * g of its values (0 when the scale is 0).
__device__ __forceinline__ uint32_t block_scale(float amax, float g, float* divisor) {
  const float r = __fdiv_rn(amax, __fmul_rn(6.0f, g));
  const uint32_t code = __nv_cvt_float_to_fp8(r, __NV_SATFINITE, __NV_E4M3);
  *divisor = __fmul_rn(e4m3_value(code), g);
  return code;
}

__device__ __forceinline__ uint32_t e2m1_code(float x, float divisor) {
  if (!(divisor > 0.0f)) return 0u;
  return static_cast<uint32_t>(__nv_cvt_float_to_fp4(__fdiv_rn(x, divisor), __NV_E2M1, cudaRoundNearest)) & 15u;
}

}  // namespace beam
