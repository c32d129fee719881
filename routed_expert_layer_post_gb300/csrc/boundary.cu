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
// values within ~2^-40 of a bf16 midpoint), using fp32 instructions in
// double-float form: squares of bf16 values are exact in fp32 and are summed
// with TwoSum; the per-token 1/sqrt runs once in fp64; products with the
// normaliser and the residual coefficients are error-free pairs (FMA gives
// the exact product error); a pair is rounded to bf16 by looking at the low
// word only when the high word sits exactly on a midpoint. Plain fp32 is not
// enough here: when h and y nearly cancel (exactly, for n - 1 a perfect
// square), a one-ulp change in y or in a rounded coefficient moves h' by
// thousands of bf16 ulps. The __f*_rn intrinsics keep the compiler from
// contracting the error-free steps into FMAs.
//
// Two schedules with the same arithmetic: one warp per token (lane l owns the
// 8-element chunks l, l+32, ...) when there are enough tokens to fill the
// GPU, and one block per token (one thread per chunk) for small batches, so
// that a decode token's loads are all in flight at once. 128-bit loads and
// stores throughout; reductions run in a fixed order (deterministic).
#include "common.cuh"
#include "kernels.h"

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

// 1/sqrt(sum/H + eps) as an fp32 pair, from a double-float sum of squares
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

// y and h' for one 8-element chunk; returns h' packed, accumulates its squares
__device__ __forceinline__ uint4 chunk_residual(const uint4& xv, const uint4& hv, const uint4& wv, const F2& r,
                                                const ResidualCoef& coef, F2& acc) {
  float fx[8], fh[8], fw[8], hn[8];
  unpack8(xv, fx);
  unpack8(hv, fh);
  unpack8(wv, fw);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float y = __uint_as_float(scaled_bf16(fx[i], fw[i], r) << 16);
    hn[i] = __uint_as_float(residual_bf16(fh[i], y, coef) << 16);
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
  for (int i = 0; i < 8; ++i) o[i] = scaled_bf16(fh[i], fw[i], r);
  return make_uint4(o[0] | (o[1] << 16), o[2] | (o[3] << 16), o[4] | (o[5] << 16), o[6] | (o[7] << 16));
}

// ------------------------------------------------------------------ warp per token
constexpr int kWarps = 4;

template <int NCMAX>
__global__ void __launch_bounds__(kWarps * 32)
    boundary_warp_kernel(const uint4* h, const uint4* __restrict__ x, const uint4* __restrict__ w_post,
                         const uint4* __restrict__ w_pre, int T, int nc, double inv_h, double eps,
                         ResidualCoef coef, uint4* h_out, uint4* __restrict__ z_out) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  const size_t row = static_cast<size_t>(t) * nc * 32;

  uint4 v[NCMAX], hv[NCMAX];
#pragma unroll
  for (int j = 0; j < NCMAX; ++j) {
    if (j < nc) {
      v[j] = x[row + j * 32 + lane];
      hv[j] = h[row + j * 32 + lane];  // read before any h_out store: h_out may alias h
    }
  }
  F2 acc{0.f, 0.f};
#pragma unroll
  for (int j = 0; j < NCMAX; ++j)
    if (j < nc) acc_squares(acc, v[j]);
  const F2 r = rsqrt_mean(warp_sum_f2(acc), inv_h, eps);

  F2 acc2{0.f, 0.f};
#pragma unroll
  for (int j = 0; j < NCMAX; ++j) {
    if (j < nc) {
      v[j] = chunk_residual(v[j], hv[j], w_post[j * 32 + lane], r, coef, acc2);
      h_out[row + j * 32 + lane] = v[j];
    }
  }
  const F2 r2 = rsqrt_mean(warp_sum_f2(acc2), inv_h, eps);
#pragma unroll
  for (int j = 0; j < NCMAX; ++j)
    if (j < nc) z_out[row + j * 32 + lane] = chunk_scale(v[j], w_pre[j * 32 + lane], r2);
}

// ------------------------------------------------------------------ block per token
__device__ __forceinline__ F2 block_sum_f2(F2 v, F2* red, int nwarps) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  v = warp_sum_f2(v);
  if (lane == 0) red[w] = v;
  __syncthreads();
  F2 t = (lane < nwarps) ? red[lane] : F2{0.f, 0.f};
  t = warp_sum_f2(t);
  __syncthreads();  // red is reused by the next reduction
  return t;
}

__global__ void __launch_bounds__(1024)
    boundary_block_kernel(const uint4* h, const uint4* __restrict__ x, const uint4* __restrict__ w_post,
                          const uint4* __restrict__ w_pre, int nc, double inv_h, double eps, ResidualCoef coef,
                          uint4* h_out, uint4* __restrict__ z_out) {
  __shared__ F2 red[32];
  const int c = threadIdx.x;  // chunk owned by this thread
  const int nwarps = blockDim.x >> 5;
  const size_t idx = static_cast<size_t>(blockIdx.x) * nc + c;
  const uint4 xv = x[idx];
  const uint4 hv = h[idx];
  const uint4 wp = w_post[c];
  const uint4 wq = w_pre[c];
  F2 acc{0.f, 0.f};
  acc_squares(acc, xv);
  const F2 r = rsqrt_mean(block_sum_f2(acc, red, nwarps), inv_h, eps);
  F2 acc2{0.f, 0.f};
  const uint4 hn = chunk_residual(xv, hv, wp, r, coef, acc2);
  h_out[idx] = hn;
  const F2 r2 = rsqrt_mean(block_sum_f2(acc2, red, nwarps), inv_h, eps);
  z_out[idx] = chunk_scale(hn, wq, r2);
}

template <int NCMAX>
void launch_warp(const uint4* h, const uint4* x, const uint4* wp, const uint4* wq, int T, int nc, double inv_h,
                 double eps, const ResidualCoef& coef, uint4* h_out, uint4* z_out, cudaStream_t stream) {
  const int blocks = (T + kWarps - 1) / kWarps;
  boundary_warp_kernel<NCMAX><<<blocks, kWarps * 32, 0, stream>>>(h, x, wp, wq, T, nc, inv_h, eps, coef, h_out,
                                                                   z_out);
}

// below this many tokens one block per token beats one warp per token
constexpr int kBlockPerTokenMaxT = 256;

}  // namespace

bool boundary_supported(int H) { return H > 0 && H % 256 == 0 && H <= 8192; }

cudaError_t launch_boundary(const uint16_t* h, const uint16_t* x, const uint16_t* w_post, const uint16_t* w_pre,
                            int T, int H, float eps, int n, uint16_t* h_out, uint16_t* z_out, cudaStream_t stream) {
  const int nc = H / 256;  // chunks per lane in the warp schedule
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
  if (T <= kBlockPerTokenMaxT) {
    boundary_block_kernel<<<T, H / 8, 0, stream>>>(hp, xp, wp, wq, H / 8, inv_h, e, coef, ho, zo);
  } else if (nc <= 4) {
    launch_warp<4>(hp, xp, wp, wq, T, nc, inv_h, e, coef, ho, zo, stream);
  } else if (nc <= 8) {
    launch_warp<8>(hp, xp, wp, wq, T, nc, inv_h, e, coef, ho, zo, stream);
  } else if (nc <= 16) {
    launch_warp<16>(hp, xp, wp, wq, T, nc, inv_h, e, coef, ho, zo, stream);
  } else if (nc <= 20) {
    launch_warp<20>(hp, xp, wp, wq, T, nc, inv_h, e, coef, ho, zo, stream);
  } else {
    launch_warp<32>(hp, xp, wp, wq, T, nc, inv_h, e, coef, ho, zo, stream);
  }
  ++launch_counter();
  return cudaGetLastError();
}

}  // namespace beam
