// NVFP4 quantizers: expert weights (offline conversion from bf16) and the
// expert inputs (at runtime).
//
// TokenSpeed blog, "Model architecture and precision -> NVFP4 and FP8
// checkpoints": each expert weight is a 4-bit E2M1 value, every 16 weights
// share an E4M3 scale and each expert has an additional FP32 scale; expert
// inputs are quantized in the same format at runtime, so the expert GEMMs run
// FP4 x FP4 ("TensorRT-LLM NVFP4 MoE": input quantization does not depend on
// routing).
//
// One block of 16 values along the reduction dimension, with FP32 scale g:
//   s = E4M3(amax / (6 g))        (round to nearest even, saturating at 448)
//   q = E2M1(x / (s g))           (round to nearest even, saturating at 6)
// each product and quotient an FP32 operation; a block with s = 0 codes all
// zeros. An expert's g is its largest |w| over gate, up and down divided by
// 6 * 448, so the block holding that weight gets scale 448.
//
// Layouts (see beam.h): codes two per byte, element 2j in the low nibble;
// weight scales in 512-byte atoms that tcgen05.cp copies to tensor memory as
// the block-scaled MMA reads them; activation scales one 16-byte slot per 64
// values (the four scales in its first bytes).
#include "common.cuh"
#include "kernels.h"
#include "nvfp4.cuh"
#include "ptx.cuh"

namespace beam {

namespace {

constexpr int kThreads = 256;

// 16 bf16 values -> 8 bytes of codes (element 2j in the low nibble); returns the scale code.
__device__ __forceinline__ uint32_t quantize16(const uint4& lo, const uint4& hi, float g, uint2* packed) {
  float f[16];
  unpack8(lo, *reinterpret_cast<float(*)[8]>(&f[0]));
  unpack8(hi, *reinterpret_cast<float(*)[8]>(&f[8]));
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
  float d;
  const uint32_t s = block_scale(amax, g, &d);
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 16; ++i) w[i >> 3] |= e2m1_code(f[i], d) << (4 * (i & 7));
  *packed = make_uint2(w[0], w[1]);
  return s;
}

// ------------------------------------------------------------------ expert weights
// Per-expert largest |w| over gate, up and down, as float bits (non-negative
// floats order like unsigned integers). blockIdx.y = expert.
__global__ void __launch_bounds__(kThreads)
    expert_amax_kernel(const uint4* __restrict__ w_gu, const uint4* __restrict__ w_d, size_t gu_vec, size_t d_vec,
                       unsigned* __restrict__ amax_bits) {
  const int e = blockIdx.y;
  const uint4* a = w_gu + static_cast<size_t>(e) * gu_vec;
  const uint4* b = w_d + static_cast<size_t>(e) * d_vec;
  float m = 0.0f;
  for (size_t i = static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x; i < gu_vec + d_vec;
       i += static_cast<size_t>(gridDim.x) * kThreads) {
    float f[8];
    unpack8(i < gu_vec ? a[i] : b[i - gu_vec], f);
#pragma unroll
    for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(f[j]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFullMask, m, o));
  if ((threadIdx.x & 31) == 0) atomicMax(&amax_bits[e], __float_as_uint(m));
}

// Offset of the scale of (row r of a plane of `rows` rows, 16-value group kb
// along a reduction of K) in the 512-byte-atom layout:
// [plane][rows/128][K/256][4 chunks][512], byte (r%32)*16 + (r/32)*4 + j.
__device__ __forceinline__ size_t atom_offset(int plane, int rows, int K, int row, int kb) {
  const int b = row >> 7, r = row & 127;
  const int s = kb >> 4, c = (kb >> 2) & 3, j = kb & 3;
  const size_t atom = (static_cast<size_t>(plane) * (rows >> 7) + b) * (K >> 8) + s;
  return atom * 2048 + c * 512 + (r & 31) * 16 + (r >> 5) * 4 + j;
}

// One thread per 16-weight group. Matrix 0: the [E][2F][H] gate/up weights
// (planes 2e, 2e+1 of F rows); matrix 1: the [E][H][F] down weights.
__global__ void __launch_bounds__(kThreads)
    quantize_experts_kernel(const uint4* __restrict__ w_gu, const uint4* __restrict__ w_d, int E, int H, int F,
                            const unsigned* __restrict__ amax_bits, uint2* __restrict__ q_gu,
                            uint8_t* __restrict__ sf_gu, uint2* __restrict__ q_d, uint8_t* __restrict__ sf_d) {
  const size_t n_gu = static_cast<size_t>(E) * 2 * F * (H / 16);
  const size_t n_d = static_cast<size_t>(E) * H * (F / 16);
  for (size_t i = static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x; i < n_gu + n_d;
       i += static_cast<size_t>(gridDim.x) * kThreads) {
    const bool gu = i < n_gu;
    const size_t v = gu ? i : i - n_gu;
    const int K = gu ? H : F;
    const size_t row = v / (K / 16);   // row over all experts' rows of this matrix
    const int kb = static_cast<int>(v - row * (K / 16));
    const int rows_per_e = gu ? 2 * F : H;
    const int e = static_cast<int>(row / rows_per_e);
    const float g = __fdiv_rn(__uint_as_float(amax_bits[e]), 2688.0f);
    const uint4* src = (gu ? w_gu : w_d) + v * 2;
    uint2 packed;
    const uint32_t s = quantize16(src[0], src[1], g, &packed);
    (gu ? q_gu : q_d)[v] = packed;
    const int r = static_cast<int>(row - static_cast<size_t>(e) * rows_per_e);  // row within the expert
    if (gu)  // gate rows 0..F-1 form plane 2e, up rows F..2F-1 plane 2e+1
      sf_gu[atom_offset(2 * e + (r >= F ? 1 : 0), F, H, r % F, kb)] = static_cast<uint8_t>(s);
    else
      sf_d[atom_offset(e, H, F, r, kb)] = static_cast<uint8_t>(s);
  }
}

__global__ void expert_scale_kernel(float* __restrict__ scale, int E) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e < E) scale[e] = __fdiv_rn(scale[e], 2688.0f);  // amax (bits written as float) -> g
}

// ------------------------------------------------------------------ activations
// One thread per 16-value group of a row; the four threads of a 64-value
// chunk gather their scale codes into one 16-byte slot.
__global__ void __launch_bounds__(kThreads)
    quantize_rows_kernel(const uint4* __restrict__ x, int rows, int K, float g, uint2* __restrict__ q,
                         uint4* __restrict__ sf) {
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int groups = K / 16;
  const size_t n = static_cast<size_t>(rows) * groups;
  const size_t i = static_cast<size_t>(blockIdx.x) * kThreads + threadIdx.x;  // groups % 4 == 0: a chunk's
  if (i >= n) return;                                                          // four threads share a warp
  uint2 packed;
  const uint32_t s = quantize16(x[2 * i], x[2 * i + 1], g, &packed);
  q[i] = packed;
  const int lane = threadIdx.x & 31;
  const unsigned quad = 0xFu << (lane & ~3);
  uint32_t word = s << (8 * (lane & 3));
  word |= __shfl_xor_sync(quad, word, 1);
  word |= __shfl_xor_sync(quad, word, 2);
  if ((lane & 3) == 0) sf[i >> 2] = make_uint4(word, 0u, 0u, 0u);
}

}  // namespace

bool nvfp4_experts_supported(int E, int H, int F) {
  return E >= 1 && E <= 256 && H % 256 == 0 && F % 256 == 0;
}

cudaError_t launch_quantize_experts(const uint16_t* w_gu, const uint16_t* w_d, int E, int H, int F, uint8_t* q_gu,
                                    uint8_t* sf_gu, uint8_t* q_d, uint8_t* sf_d, float* expert_scale, int num_sms,
                                    cudaStream_t stream) {
  // the scales array first holds each expert's largest |w| (as float bits)
  cudaError_t err = cudaMemsetAsync(expert_scale, 0, sizeof(float) * E, stream);
  if (err != cudaSuccess) return err;
  const size_t gu_vec = static_cast<size_t>(2) * F * H / 8, d_vec = static_cast<size_t>(H) * F / 8;
  expert_amax_kernel<<<dim3(64, E), kThreads, 0, stream>>>(reinterpret_cast<const uint4*>(w_gu),
                                                           reinterpret_cast<const uint4*>(w_d), gu_vec, d_vec,
                                                           reinterpret_cast<unsigned*>(expert_scale));
  ++launch_counter();
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  quantize_experts_kernel<<<num_sms * 8, kThreads, 0, stream>>>(
      reinterpret_cast<const uint4*>(w_gu), reinterpret_cast<const uint4*>(w_d), E, H, F,
      reinterpret_cast<const unsigned*>(expert_scale), reinterpret_cast<uint2*>(q_gu), sf_gu,
      reinterpret_cast<uint2*>(q_d), sf_d);
  ++launch_counter();
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  expert_scale_kernel<<<(E + 255) / 256, 256, 0, stream>>>(expert_scale, E);
  ++launch_counter();
  return cudaGetLastError();
}

cudaError_t launch_quantize_rows(const uint16_t* x, int rows, int K, float g, uint8_t* q, uint8_t* sf,
                                 cudaStream_t stream, bool pdl) {
  const size_t n = static_cast<size_t>(rows) * (K / 16);
  const int blocks = static_cast<int>((n + kThreads - 1) / kThreads);
  const cudaError_t err = launch_kernel(quantize_rows_kernel, dim3(blocks), dim3(kThreads), 0, stream, pdl,
                                        reinterpret_cast<const uint4*>(x), rows, K, g, reinterpret_cast<uint2*>(q),
                                        reinterpret_cast<uint4*>(sf));
  ++launch_counter();
  return err;
}

}  // namespace beam
