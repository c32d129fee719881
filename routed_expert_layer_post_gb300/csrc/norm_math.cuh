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
// 1/sqrt(n) = c_hi + c_lo; c_bnd = c_hi 2^-20 scales the bracket of the
// fp32 residual (residual_bracket).
struct ResidualCoef {
  float cm_hi, cm_lo, c_hi, c_lo, c_bnd;
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

// ---------------------------------------------------------------- bracketed chunks
// The boundary kernel's form of the adaptive scheme, with fewer instructions
// per element. Each output is bracketed by two fp32 numbers that provably
// enclose its exact value; when both round to the same bf16 number, so does
// the exact value (rounding is monotone), and that number is the result. The
// pairs of an 8-element chunk OR their differences into one word, so a chunk
// takes a single branch; a chunk left open re-checks its elements out of line
// and sends the open ones alone to the exact paths above.

// a - b per lane, one IEEE rounding each
__device__ __forceinline__ float2 fsub2(float2 a, float2 b) {
  uint64_t d;
  asm("{\n\t.reg .b64 pa, pb;\n\t"
      "mov.b64 pa, {%1, %2};\n\t"
      "mov.b64 pb, {%3, %4};\n\t"
      "sub.rn.f32x2 %0, pa, pb;\n\t}"
      : "=l"(d)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(d));
  return r;
}

// acc_add2 with subtractions in place of additions of negated copies (the
// same IEEE operations, so the same sums)
__device__ __forceinline__ void acc_add2s(F2x2& acc, float2 v) {
  const float2 s = __fadd2_rn(acc.hi, v);
  const float2 bp = fsub2(s, acc.hi);
  const float2 e = __fadd2_rn(fsub2(acc.hi, fsub2(s, bp)), fsub2(v, bp));
  acc.hi = s;
  acc.lo = __fadd2_rn(acc.lo, e);
}

__device__ __forceinline__ float2 unpack2(uint32_t w) { return make_float2(bf16_lo(w), bf16_hi(w)); }

// The products of both lanes of two bf16x2 words, exact in fp32 (8-bit
// significands), each by one mixed-precision multiply-add straight from the
// packed halves: no unpacking. Adding -0 keeps the sign of a zero product.
__device__ __forceinline__ float2 mul_bf16x2(uint32_t a, uint32_t b) {
  float2 r;
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %2;\n\t"
      "mov.b32 {bl, bh}, %3;\n\t"
      "fma.rn.f32.bf16 %0, al, bl, 0f80000000;\n\t"
      "fma.rn.f32.bf16 %1, ah, bh, 0f80000000;\n\t}"
      : "=f"(r.x), "=f"(r.y)
      : "r"(a), "r"(b));
  return r;
}

// Ends of the bracket of a * b * r: the scale r.hi (1 -+ 2^-21), rounded.
// The pair r is within 2^-45 of 1/sqrt(mean + eps) and r.hi within 2^-24 of
// it, so the ends lie at least 2^-21.4 (relative) below and above the exact
// scale.
struct ScaleBracket {
  float lo, hi;
};
__device__ __forceinline__ ScaleBracket scale_bracket(const F2& r) {
  return {__fmul_rn(r.hi, 1.0f - 0x1p-21f), __fmul_rn(r.hi, 1.0f + 0x1p-21f)};
}

// Bracket of a * b * r for a pair, given the exact products ab = a * b: the
// rounded products fl(ab s.lo) and fl(ab s.hi) keep the exact value between
// them (each end's rounding, 2^-24, is well inside its scale's 2^-21.4
// margin) for every result in the normal range. Returns the bf16x2 of the s.hi end;
// open collects the bits in which the two ends' roundings differ.
__device__ __forceinline__ uint32_t scaled_bracket(float2 ab, const ScaleBracket& s, uint32_t& open) {
  const uint32_t lo = bf16x2_bits(__fmul2_rn(ab, make_float2(s.lo, s.lo)));
  const uint32_t hi = bf16x2_bits(__fmul2_rn(ab, make_float2(s.hi, s.hi)));
  open |= lo ^ hi;
  return hi;
}

// Bracket of (sqrt(n-1) h + y) / sqrt(n) for a pair. With S = |sqrt(n-1) h| +
// |y|, v = fl(fl(cm_hi h + y) c_hi) is within c S 2^-21.9 of the exact value
// (two roundings and the two rounded coefficients), cancellation included;
// v -+ fl(|h| cm_hi + |y|) c_bnd (c_bnd = c_hi 2^-20), each formed by one
// fused multiply-add, stays beyond that after its own rounding.
__device__ __forceinline__ uint32_t residual_bracket(float2 h, float2 y, const ResidualCoef& k, uint32_t& open) {
  const float2 cm = make_float2(k.cm_hi, k.cm_hi);
  const float2 v = __fmul2_rn(__ffma2_rn(cm, h, y), make_float2(k.c_hi, k.c_hi));
  const float2 m = __ffma2_rn(abs2(h), cm, abs2(y));
  const uint32_t lo = bf16x2_bits(__ffma2_rn(m, make_float2(-k.c_bnd, -k.c_bnd), v));
  const uint32_t hi = bf16x2_bits(__ffma2_rn(m, make_float2(k.c_bnd, k.c_bnd), v));
  open |= lo ^ hi;
  return hi;
}

// an open chunk of a * b * r: each element re-checked, the open ones exact
static __device__ __noinline__ uint4 reopen_scaled(uint4 av, uint4 bv, F2 r, ScaleBracket sb, uint4 ov) {
  const uint32_t a[4] = {av.x, av.y, av.z, av.w};
  const uint32_t b[4] = {bv.x, bv.y, bv.z, bv.w};
  uint32_t o[4] = {ov.x, ov.y, ov.z, ov.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 pa = unpack2(a[i]), pb = unpack2(b[i]);
    uint32_t open = 0;
    scaled_bracket(__fmul2_rn(pa, pb), sb, open);
    if (open & 0xffffu) o[i] = (o[i] & 0xffff0000u) | scaled_bf16(pa.x, pb.x, r);
    if (open >> 16) o[i] = (o[i] & 0xffffu) | (scaled_bf16(pa.y, pb.y, r) << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// an open chunk of the residual add: each element re-checked, the open ones exact
static __device__ __noinline__ uint4 reopen_residual(uint4 hv, uint4 yv, ResidualCoef k, uint4 ov) {
  const uint32_t h[4] = {hv.x, hv.y, hv.z, hv.w};
  const uint32_t y[4] = {yv.x, yv.y, yv.z, yv.w};
  uint32_t o[4] = {ov.x, ov.y, ov.z, ov.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 ph = unpack2(h[i]), py = unpack2(y[i]);
    uint32_t open = 0;
    residual_bracket(ph, py, k, open);
    if (open & 0xffffu) o[i] = (o[i] & 0xffff0000u) | residual_bf16(ph.x, py.x, k);
    if (open >> 16) o[i] = (o[i] & 0xffffu) | (residual_bf16(ph.y, py.y, k) << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// bf16 of a * b * r for a chunk (sb = scale_bracket(r))
__device__ __forceinline__ uint4 chunk_scaled(const uint4& av, const uint4& bv, const F2& r, const ScaleBracket& sb) {
  uint32_t open = 0;
  const uint4 o = make_uint4(scaled_bracket(mul_bf16x2(av.x, bv.x), sb, open),
                             scaled_bracket(mul_bf16x2(av.y, bv.y), sb, open),
                             scaled_bracket(mul_bf16x2(av.z, bv.z), sb, open),
                             scaled_bracket(mul_bf16x2(av.w, bv.w), sb, open));
  return open == 0 ? o : reopen_scaled(av, bv, r, sb, o);
}

// y = bf16(x w_post r), then h' = bf16((sqrt(n-1) h + y) / sqrt(n)) for a
// chunk; returns h' and accumulates its squares (in element order, as
// chunk_residual)
__device__ __forceinline__ uint4 chunk_residual_bracketed(const uint4& xv, const uint4& hv, const uint4& wv,
                                                          const F2& r, const ScaleBracket& sb, const ResidualCoef& k,
                                                          F2x2& acc) {
  const uint4 y = chunk_scaled(xv, wv, r, sb);
  uint32_t open = 0;
  uint4 o = make_uint4(residual_bracket(unpack2(hv.x), unpack2(y.x), k, open),
                       residual_bracket(unpack2(hv.y), unpack2(y.y), k, open),
                       residual_bracket(unpack2(hv.z), unpack2(y.z), k, open),
                       residual_bracket(unpack2(hv.w), unpack2(y.w), k, open));
  if (open != 0) o = reopen_residual(hv, y, k, o);
  const uint32_t w[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) acc_add2s(acc, mul_bf16x2(w[i], w[i]));
  return o;
}

// squares of a chunk of bf16 values into a pair of double-float sums
__device__ __forceinline__ void acc_squares2s(F2x2& acc, const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) acc_add2s(acc, mul_bf16x2(w[i], w[i]));
}

// block_rsqrt_mean without the closing barrier: each of the kernel's
// reductions has a red array of its own
__device__ __forceinline__ F2 block_rsqrt_mean_once(F2 v, F2* red, int nwarps, F2 inv_h, float eps) {
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
  return red[32];
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
  coef.c_bnd = std::ldexp(coef.c_hi, -20);
  return coef;
}

}  // namespace norm
}  // namespace beam
