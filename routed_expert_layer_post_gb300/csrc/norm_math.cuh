// Device arithmetic of the sandwich-norm boundary, shared by the boundary
// kernel and the fused decode routing kernel: double-float sums of squares,
// the per-token normaliser, and bf16 rounding of the three outputs with a
// rigorous fp32 fast path and an exact double-float fallback (see
// boundary.cu for the numerics).
#pragma once

#include "common.cuh"

#include <cmath>

namespace beam {
namespace norm {

struct F2 {
  float hi, lo;
};

__device__ __forceinline__ F2 two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bp = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
  return {s, e};
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

// 1/sqrt(sum/H + eps) as an fp32 pair, in double-float arithmetic (GB300
// runs fp64 at a small fraction of the fp32 rate: one fp64 1/sqrt takes about
// fifteen times as long as this). m = sum * (1/H) + eps is formed as a pair
// with error-free products; r0 = rsqrtf(m) is within 2^-22 of 1/sqrt(m), and
// one Newton step carried to second order, r0 (1 + e/2 + 3e^2/8) with
// e = 1 - m r0^2, leaves a truncation error below 2^-64. The fp32 product
// a = m_hi r0^2 lies within 2^-21 of 1, so 1 - a is exact and e carries
// about 2^-46 relative error; so does the pair (2^-48 for a pair rounded from
// an fp64 1/sqrt).
__device__ __forceinline__ F2 rsqrt_mean(F2 sum, F2 inv_h, float eps) {
  const float p = __fmul_rn(sum.hi, inv_h.hi);
  float pe = fmaf(sum.hi, inv_h.hi, -p);
  pe = fmaf(sum.hi, inv_h.lo, pe);
  pe = fmaf(sum.lo, inv_h.hi, pe);
  const F2 s = two_sum(p, eps);
  float m_lo = __fadd_rn(s.lo, pe);
  const float m_hi = __fadd_rn(s.hi, m_lo);
  m_lo = __fsub_rn(m_lo, __fsub_rn(m_hi, s.hi));
  const float r0 = rsqrtf(m_hi);
  const float q = __fmul_rn(r0, r0);
  const float qe = fmaf(r0, r0, -q);
  const float a = __fmul_rn(m_hi, q);
  float ae = fmaf(m_hi, q, -a);
  ae = fmaf(m_hi, qe, ae);
  ae = fmaf(m_lo, q, ae);
  const float e = __fsub_rn(__fsub_rn(1.0f, a), ae);
  const float corr = __fmul_rn(r0, __fmul_rn(e, fmaf(0.375f, e, 0.5f)));
  const float hi = __fadd_rn(r0, corr);
  return {hi, __fsub_rn(corr, __fsub_rn(hi, r0))};
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

// Adaptive precision: the plain fp32 value v is used when every value within
// its error bound e rounds to the same bf16 number (the usual case); only
// values whose interval [v - e, v + e] straddles a rounding midpoint take the
// exact double-float paths above. The bounds are deliberately loose (about
// four times the worst-case fp32 error), so the fast path never decides a
// case the exact path would decide differently.
//
// The fast paths and the sums of squares work on element pairs with
// Blackwell's packed fp32 arithmetic: each lane of __fmul2_rn / __fadd2_rn /
// __ffma2_rn is one IEEE round-to-nearest operation, the value of the scalar
// form, at half the issue slots (the boundary is issue-bound). An element
// whose rounding the check leaves open falls back alone to the exact path.

__device__ __forceinline__ float2 neg2(float2 v) { return make_float2(-v.x, -v.y); }
__device__ __forceinline__ float2 abs2(float2 v) { return make_float2(fabsf(v.x), fabsf(v.y)); }

// bf16x2 bits (element 0 in the low half) of a pair
__device__ __forceinline__ uint32_t bf16x2_bits(float2 v) {
  const __nv_bfloat162 b = __float22bfloat162_rn(v);
  return *reinterpret_cast<const uint32_t*>(&b);
}

// Pair of double-float accumulators (element 0 and element 1 sums)
struct F2x2 {
  float2 hi, lo;
};

__device__ __forceinline__ void acc_add2(F2x2& acc, float2 v) {
  const float2 s = __fadd2_rn(acc.hi, v);
  const float2 bp = __fadd2_rn(s, neg2(acc.hi));
  const float2 e = __fadd2_rn(__fadd2_rn(acc.hi, neg2(__fadd2_rn(s, neg2(bp)))), __fadd2_rn(v, neg2(bp)));
  acc.hi = s;
  acc.lo = __fadd2_rn(acc.lo, e);
}

// the two lanes' sums as one pair
__device__ __forceinline__ F2 fold(const F2x2& a) { return f2_add(F2{a.hi.x, a.lo.x}, F2{a.hi.y, a.lo.y}); }

// bf16x2 of a * b * r for a pair: a, b bf16 values (a * b exact in fp32), r a
// pair with |r.lo| <= 2^-24 |r.hi|, so v = fl(a b r.hi) is within about
// |v| 2^-23 of the exact value (the check allows |v| 2^-21)
__device__ __forceinline__ uint32_t scaled_bf16x2_fast(float2 a, float2 b, const F2& r) {
  const float2 v = __fmul2_rn(__fmul2_rn(a, b), make_float2(r.hi, r.hi));
  const float2 e = __fmul2_rn(abs2(v), make_float2(0x1p-21f, 0x1p-21f));
  const uint32_t lo = bf16x2_bits(__fadd2_rn(v, neg2(e)));
  const uint32_t hi = bf16x2_bits(__fadd2_rn(v, e));
  if (lo == hi) return bf16x2_bits(v);
  uint32_t out = 0;
  out |= ((lo & 0xffffu) == (hi & 0xffffu)) ? f2bf(v.x) : scaled_bf16(a.x, b.x, r);
  out |= (((lo >> 16) == (hi >> 16)) ? f2bf(v.y) : scaled_bf16(a.y, b.y, r)) << 16;
  return out;
}

// bf16x2 of (sqrt(n-1) h + y) / sqrt(n) for a pair; the error of the fp32
// evaluation is bounded by a few ulps of c (|sqrt(n-1) h| + |y|), which covers
// cancellation
__device__ __forceinline__ uint32_t residual_bf16x2_fast(float2 h, float2 y, const ResidualCoef& k) {
  const float2 cm = make_float2(k.cm_hi, k.cm_hi), c = make_float2(k.c_hi, k.c_hi);
  const float2 ch = __fmul2_rn(cm, h);
  const float2 v = __fmul2_rn(__ffma2_rn(cm, h, y), c);
  const float2 e =
      __fmul2_rn(__fmul2_rn(__fadd2_rn(abs2(ch), abs2(y)), c), make_float2(0x1p-20f, 0x1p-20f));
  const uint32_t lo = bf16x2_bits(__fadd2_rn(v, neg2(e)));
  const uint32_t hi = bf16x2_bits(__fadd2_rn(v, e));
  if (lo == hi) return bf16x2_bits(v);
  uint32_t out = 0;
  out |= ((lo & 0xffffu) == (hi & 0xffffu)) ? f2bf(v.x) : residual_bf16(h.x, y.x, k);
  out |= (((lo >> 16) == (hi >> 16)) ? f2bf(v.y) : residual_bf16(h.y, y.y, k)) << 16;
  return out;
}

__device__ __forceinline__ void acc_squares2(F2x2& acc, const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = make_float2(bf16_lo(w[i]), bf16_hi(w[i]));
    acc_add2(acc, __fmul2_rn(f, f));  // exact squares of bf16 values
  }
}

// y and h' for one 8-element chunk; returns h' packed, accumulates its squares
__device__ __forceinline__ uint4 chunk_residual(const uint4& xv, const uint4& hv, const uint4& wv, const F2& r,
                                                const ResidualCoef& coef, F2x2& acc) {
  const uint32_t x[4] = {xv.x, xv.y, xv.z, xv.w};
  const uint32_t h[4] = {hv.x, hv.y, hv.z, hv.w};
  const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t yb = scaled_bf16x2_fast(make_float2(bf16_lo(x[i]), bf16_hi(x[i])),
                                           make_float2(bf16_lo(w[i]), bf16_hi(w[i])), r);
    o[i] = residual_bf16x2_fast(make_float2(bf16_lo(h[i]), bf16_hi(h[i])), make_float2(bf16_lo(yb), bf16_hi(yb)),
                                coef);
    const float2 hn = make_float2(bf16_lo(o[i]), bf16_hi(o[i]));
    acc_add2(acc, __fmul2_rn(hn, hn));
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ uint4 chunk_scale(const uint4& hv, const uint4& wv, const F2& r) {
  const uint32_t h[4] = {hv.x, hv.y, hv.z, hv.w};
  const uint32_t w[4] = {wv.x, wv.y, wv.z, wv.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    o[i] = scaled_bf16x2_fast(make_float2(bf16_lo(h[i]), bf16_hi(h[i])), make_float2(bf16_lo(w[i]), bf16_hi(w[i])),
                              r);
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// block-wide sum of squares -> 1/sqrt(mean + eps), evaluated by one thread;
// red needs 33 entries
__device__ __forceinline__ F2 block_rsqrt_mean(F2 v, F2* red, int nwarps, F2 inv_h, float eps) {
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

// 1/H as an fp32 pair
inline F2 inv_hidden(int H) {
  const double v = 1.0 / H;
  const float hi = static_cast<float>(v);
  return {hi, static_cast<float>(v - static_cast<double>(hi))};
}

// coefficients of the residual add for boundary index n
inline ResidualCoef residual_coef(int n) {
  const double cm = std::sqrt(static_cast<double>(n - 1)), c = 1.0 / std::sqrt(static_cast<double>(n));
  ResidualCoef coef;
  coef.cm_hi = static_cast<float>(cm);
  coef.cm_lo = static_cast<float>(cm - static_cast<double>(coef.cm_hi));
  coef.c_hi = static_cast<float>(c);
  coef.c_lo = static_cast<float>(c - static_cast<double>(coef.c_hi));
  return coef;
}

}  // namespace norm
}  // namespace beam
