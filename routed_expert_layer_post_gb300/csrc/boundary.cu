// Sandwich-norm boundary: post-RMSNorm of the previous sublayer's output,
// depth-scaled residual add, next pre-RMSNorm, in one pass.
//
// vLLM Beam summary, section "MoE and residual stream" (RMSNorm before and
// after every sublayer; h <- sqrt((n-1)/n) h + x / sqrt(n)) and kernel change
// 1 (norm, residual, norm fused with FP32 math and the reference's BF16
// rounding points); TokenSpeed blog, "MNNVL all-reduce and SandwichNorm
// fusion" (post-norm, depth-scaled residual, next pre-norm); Gaudi cookbook
// port, "What was built -> Model code" (bf16 rounding after the norms and the
// residual).
//
//   y  = bf16(x * w_post / sqrt(mean(x^2) + eps))
//   h' = bf16((sqrt(n-1) h + y) / sqrt(n))
//   z  = bf16(h' * w_pre / sqrt(mean(h'^2) + eps))
//
// Numerics. Every rounding point gets the correctly rounded bf16 value (up to
// values within ~2^-40 of a bf16 midpoint). Squares of bf16 values are exact
// in fp32 and are summed with TwoSum; the per-token 1/sqrt runs once in fp64.
// Each output is first evaluated in plain fp32 together with a rigorous error
// bound; when the bound shows the bf16 rounding is already decided (nearly
// always) that value is kept, otherwise the element is recomputed in
// double-float form: products with the normaliser and the residual
// coefficients as error-free pairs (FMA gives the exact product error), and
// the pair rounded to bf16 by looking at the low word only when the high word
// sits exactly on a midpoint. Plain fp32 alone is not enough: when h and y
// nearly cancel (exactly, for n - 1 a perfect square), a one-ulp change in y or
// in a rounded coefficient moves h' by thousands of bf16 ulps. The __f*_rn
// intrinsics keep the compiler from contracting the error-free steps into FMAs.
//
// Schedule: one block per token, one thread per 8-element chunk (128-bit
// loads and stores), two block reductions in a fixed order (deterministic).
// A decode token's loads are all in flight at once, and the kernel body stays
// small. The warp-per-token alternative (each lane holding 20 chunks in
// registers) measured 4-5x slower on GB300 at 2048 and 16384 tokens: its
// unrolled body overflowed the instruction cache and 186 registers per thread
// left 8 warps per SM.
#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

#include <cmath>

namespace beam {

namespace {

struct F2 {
  float hi, lo;
};

__device__ __forceinline__ F2 two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bp = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
  return {s, e};
}

__device__ __forceinline__ void acc_add(F2& acc, float v) {
  const F2 t = two_sum(acc.hi, v);
  acc.hi = t.hi;
  acc.lo = __fadd_rn(acc.lo, t.lo);
}

// symmetric in its arguments, so butterfly reductions agree bit for bit on every lane
__device__ __forceinline__ F2 f2_add(F2 a, F2 b) {
  const F2 t = two_sum(a.hi, b.hi);
  const float lo = __fadd_rn(__fadd_rn(a.lo, b.lo), t.lo);
  const float hi = __fadd_rn(t.hi, lo);
  return {hi, __fsub_rn(lo, __fsub_rn(hi, t.hi))};
}

__device__ __forceinline__ F2 warp_sum_f2(F2 v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    F2 w;
    w.hi = __shfl_xor_sync(kFullMask, v.hi, o);
    w.lo = __shfl_xor_sync(kFullMask, v.lo, o);
    v = f2_add(v, w);
  }
  return v;
}

// 1/sqrt(sum/H + eps) as an fp32 pair, from a double-float sum of squares.
// GB300 runs fp64 at a small fraction of the fp32 rate, so one thread per
// token evaluates this and the result is broadcast.
__device__ __forceinline__ F2 rsqrt_mean(F2 sum, double inv_h, double eps) {
  const double ms = (static_cast<double>(sum.hi) + static_cast<double>(sum.lo)) * inv_h + eps;
  const double r = 1.0 / sqrt(ms);
  const float hi = static_cast<float>(r);
  return {hi, static_cast<float>(r - static_cast<double>(hi))};
}

// bf16 bits of the exact value hi + lo, where |lo| <= half an fp32 ulp of hi
__device__ __forceinline__ uint32_t round_pair(float hi, float lo) {
  const uint32_t b = __float_as_uint(hi);
  if ((b & 0xffffu) == 0x8000u && lo != 0.0f) {
    const bool grow = (lo > 0.0f) == (hi > 0.0f);
    return (b >> 16) + (grow ? 1u : 0u);
  }
  return f2bf(hi);
}

// bf16 bits of a * b * r with a, b bf16 values (a * b exact in fp32) and r a pair
__device__ __forceinline__ uint32_t scaled_bf16(float a, float b, const F2& r) {
  const float ab = __fmul_rn(a, b);
  const float p = __fmul_rn(ab, r.hi);
  float pe = fmaf(ab, r.hi, -p);
  pe = fmaf(ab, r.lo, pe);
  const float hi = __fadd_rn(p, pe);
  return round_pair(hi, __fsub_rn(pe, __fsub_rn(hi, p)));
}

// Coefficients of the residual add as fp32 pairs: sqrt(n-1) = cm_hi + cm_lo,
// 1/sqrt(n) = c_hi + c_lo.
struct ResidualCoef {
  float cm_hi, cm_lo, c_hi, c_lo;
};

// bf16 bits of (sqrt(n-1) h + y) / sqrt(n)
__device__ __forceinline__ uint32_t residual_bf16(float h, float y, const ResidualCoef& k) {
  const float p = __fmul_rn(k.cm_hi, h);
  float pe = fmaf(k.cm_hi, h, -p);
  pe = fmaf(k.cm_lo, h, pe);
  const F2 s = two_sum(p, y);
  float u_lo = __fadd_rn(s.lo, pe);
  const float u_hi = __fadd_rn(s.hi, u_lo);
  u_lo = __fsub_rn(u_lo, __fsub_rn(u_hi, s.hi));
  const float v = __fmul_rn(u_hi, k.c_hi);
  float ve = fmaf(u_hi, k.c_hi, -v);
  ve = fmaf(u_hi, k.c_lo, ve);
  ve = fmaf(u_lo, k.c_hi, ve);
  const float v_hi = __fadd_rn(v, ve);
  return round_pair(v_hi, __fsub_rn(ve, __fsub_rn(v_hi, v)));
}

__device__ __forceinline__ void acc_squares(F2& acc, const uint4& v) {
  float f[8];
  unpack8(v, f);
#pragma unroll
  for (int i = 0; i < 8; ++i) acc_add(acc, __fmul_rn(f[i], f[i]));  // exact square of a bf16 value
}

// Adaptive precision: the plain fp32 value v is used when every value within
// its error bound e rounds to the same bf16 number (the usual case); only
// values whose interval [v - e, v + e] straddles a rounding midpoint take the
// exact double-float path above. The bounds are deliberately loose (about
// four times the worst-case fp32 error), so the fast path never decides a
// case the exact path would decide differently.
__device__ __forceinline__ bool rounds_alike(float v, float e) {
  return f2bf(__fsub_rn(v, e)) == f2bf(__fadd_rn(v, e));
}

// bf16(a * b * r), a and b bf16 values, r a pair with |r.lo| <= 2^-24 |r.hi|
__device__ __forceinline__ uint32_t scaled_bf16_fast(float a, float b, const F2& r) {
  const float v = __fmul_rn(__fmul_rn(a, b), r.hi);  // a * b is exact
  if (rounds_alike(v, fabsf(v) * 0x1p-21f)) return f2bf(v);
  return scaled_bf16(a, b, r);
}

// bf16((sqrt(n-1) h + y) / sqrt(n)); the error of the fp32 evaluation is
// bounded by a few ulps of c * (|sqrt(n-1) h| + |y|), which covers cancellation
__device__ __forceinline__ uint32_t residual_bf16_fast(float h, float y, const ResidualCoef& k) {
  const float ch = __fmul_rn(k.cm_hi, h);
  const float v = __fmul_rn(fmaf(k.cm_hi, h, y), k.c_hi);
  const float e = __fmul_rn(__fadd_rn(fabsf(ch), fabsf(y)), k.c_hi) * 0x1p-20f;
  if (rounds_alike(v, e)) return f2bf(v);
  return residual_bf16(h, y, k);
}

// y and h' for one 8-element chunk; returns h' packed, accumulates its squares
__device__ __forceinline__ uint4 chunk_residual(const uint4& xv, const uint4& hv, const uint4& wv, const F2& r,
                                                const ResidualCoef& coef, F2& acc) {
  float fx[8], fh[8], fw[8], hn[8];
  unpack8(xv, fx);
  unpack8(hv, fh);
  unpack8(wv, fw);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float y = __uint_as_float(scaled_bf16_fast(fx[i], fw[i], r) << 16);
    hn[i] = __uint_as_float(residual_bf16_fast(fh[i], y, coef) << 16);
    acc_add(acc, __fmul_rn(hn[i], hn[i]));
  }
  return pack8(hn);
}

__device__ __forceinline__ uint4 chunk_scale(const uint4& hv, const uint4& wv, const F2& r) {
  float fh[8], fw[8];
  unpack8(hv, fh);
  unpack8(wv, fw);
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i] = scaled_bf16_fast(fh[i], fw[i], r);
  return make_uint4(o[0] | (o[1] << 16), o[2] | (o[3] << 16), o[4] | (o[5] << 16), o[6] | (o[7] << 16));
}

// ------------------------------------------------------------------ block per token
// block-wide sum of squares -> 1/sqrt(mean + eps), evaluated by thread 0
__device__ __forceinline__ F2 block_rsqrt_mean(F2 v, F2* red, int nwarps, double inv_h, double eps) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  v = warp_sum_f2(v);
  if (lane == 0) red[w] = v;
  __syncthreads();
  if (w == 0) {
    F2 t = (lane < nwarps) ? red[lane] : F2{0.f, 0.f};
    t = warp_sum_f2(t);
    if (lane == 0) red[32] = rsqrt_mean(t, inv_h, eps);
  }
  __syncthreads();
  const F2 r = red[32];
  __syncthreads();  // red is reused by the next reduction
  return r;
}

__global__ void __launch_bounds__(1024)
    boundary_block_kernel(const uint4* h, const uint4* __restrict__ x, const uint4* __restrict__ w_post,
                          const uint4* __restrict__ w_pre, int nc, double inv_h, double eps, ResidualCoef coef,
                          uint4* h_out, uint4* __restrict__ z_out, int* zero_slot) {
  __shared__ F2 red[33];
  ptx::griddep_wait();  // inputs come from the previous kernel
  ptx::griddep_launch_dependents();
  if (zero_slot != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *zero_slot = 0;
  const int c = threadIdx.x;  // chunk owned by this thread
  const int nwarps = blockDim.x >> 5;
  const size_t idx = static_cast<size_t>(blockIdx.x) * nc + c;
  const uint4 xv = x[idx];
  const uint4 hv = h[idx];
  const uint4 wp = w_post[c];
  const uint4 wq = w_pre[c];
  F2 acc{0.f, 0.f};
  acc_squares(acc, xv);
  const F2 r = block_rsqrt_mean(acc, red, nwarps, inv_h, eps);
  F2 acc2{0.f, 0.f};
  const uint4 hn = chunk_residual(xv, hv, wp, r, coef, acc2);
  h_out[idx] = hn;
  const F2 r2 = block_rsqrt_mean(acc2, red, nwarps, inv_h, eps);
  z_out[idx] = chunk_scale(hn, wq, r2);
}

}  // namespace

bool boundary_supported(int H) { return H > 0 && H % 256 == 0 && H <= 8192; }

cudaError_t launch_boundary(const uint16_t* h, const uint16_t* x, const uint16_t* w_post, const uint16_t* w_pre,
                            int T, int H, float eps, int n, uint16_t* h_out, uint16_t* z_out, cudaStream_t stream,
                            bool pdl, int* zero_slot) {
  const double cm = std::sqrt(static_cast<double>(n - 1)), c = 1.0 / std::sqrt(static_cast<double>(n));
  ResidualCoef coef;
  coef.cm_hi = static_cast<float>(cm);
  coef.cm_lo = static_cast<float>(cm - static_cast<double>(coef.cm_hi));
  coef.c_hi = static_cast<float>(c);
  coef.c_lo = static_cast<float>(c - static_cast<double>(coef.c_hi));
  const double inv_h = 1.0 / H, e = static_cast<double>(eps);
  const uint4* hp = reinterpret_cast<const uint4*>(h);
  const uint4* xp = reinterpret_cast<const uint4*>(x);
  const uint4* wp = reinterpret_cast<const uint4*>(w_post);
  const uint4* wq = reinterpret_cast<const uint4*>(w_pre);
  uint4* ho = reinterpret_cast<uint4*>(h_out);
  uint4* zo = reinterpret_cast<uint4*>(z_out);
  const cudaError_t err = launch_kernel(boundary_block_kernel, dim3(T), dim3(H / 8), 0, stream, pdl, hp, xp, wp, wq,
                                        H / 8, inv_h, e, coef, ho, zo, zero_slot);
  ++launch_counter();
  return err;
}

}  // namespace beam
