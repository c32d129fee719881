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
// values within ~2^-40 of a bf16 midpoint, and for results in the fp32 normal
// range). Squares and products of bf16 values are exact in fp32 (mixed
// bf16 x bf16 -> fp32 multiply-adds straight from the packed halves); the
// squares are summed with TwoSum and the per-token 1/sqrt is taken in
// double-float arithmetic. Each output is first evaluated in plain fp32 and
// bracketed by two fp32 numbers that provably enclose the exact value; when
// both ends round to the same bf16 number (nearly always) that number is the
// result. The brackets of a chunk's eight elements are checked together, one
// branch per chunk; an open chunk is re-checked element by element out of
// line, and each open element is recomputed in double-float form: products
// with the normaliser and the residual coefficients as error-free pairs (FMA
// gives the exact product error), and the pair rounded to bf16 by looking at
// the low word only when the high word sits exactly on a midpoint. Plain fp32
// alone is not enough: when h and y nearly cancel (exactly, for n - 1 a
// perfect square), a one-ulp change in y or in a rounded coefficient moves h'
// by thousands of bf16 ulps. The __f*_rn intrinsics keep the compiler from
// contracting the error-free steps into FMAs.
//
// Schedule: one block per token, each thread owning one to four 8-element
// chunks (128-bit loads and stores), two block reductions in a fixed order
// (deterministic). A decode token's loads are all in flight at once, and the
// kernel body stays small. The warp-per-token alternative (each lane holding
// 20 chunks in registers) measured 4-5x slower on GB300 at 2048 and 16384
// tokens: its unrolled body overflowed the instruction cache and 186 registers
// per thread left 8 warps per SM.
#include "common.cuh"
#include "kernels.h"
#include "norm_math.cuh"
#include "ptx.cuh"

#include <cmath>

namespace beam {

namespace {

using namespace norm;

// ------------------------------------------------------------------ block per token
// NCH chunks per thread: chunks c, c + width, ... (width = THREADS, or
// blockDim.x when THREADS is 0). More chunks per thread share the two block
// reductions and their barriers among more elements; each thread's chunks
// enter its double-float sum in chunk order before the reduction, so the sums
// are exact whatever NCH is. A compile-time width turns the chunk offsets
// into immediates, and MINB blocks per SM caps the registers (64 for the
// hidden size 5120: 160 threads, 6 blocks, 30 warps per SM).
template <int NCH, int THREADS, int MINB>
__global__ void __launch_bounds__(THREADS > 0 ? THREADS : 1024, MINB)
    boundary_block_kernel(const uint4* h, const uint4* __restrict__ x, const uint4* __restrict__ w_post,
                          const uint4* __restrict__ w_pre, int nc, F2 inv_h, float eps, ResidualCoef coef,
                          uint4* h_out, uint4* __restrict__ z_out, int* zero_slot) {
  __shared__ F2 red[2][33];  // one per reduction: no barrier before reuse
  const int width = THREADS > 0 ? THREADS : static_cast<int>(blockDim.x);
  if constexpr (THREADS > 0) nc = NCH * THREADS;
  ptx::griddep_wait();  // inputs come from the previous kernel
  ptx::griddep_launch_dependents();
  if (zero_slot != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *zero_slot = 0;
  const size_t base = static_cast<size_t>(blockIdx.x) * nc + threadIdx.x;
  uint4 xv[NCH], hv[NCH];
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    xv[i] = x[base + i * width];
    hv[i] = h[base + i * width];
  }
  F2x2 acc{{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
  for (int i = 0; i < NCH; ++i) acc_squares2s(acc, xv[i]);
  const F2 r = block_rsqrt_mean_once(fold(acc), red[0], width >> 5, inv_h, eps);
  const ScaleBracket sb = scale_bracket(r);
  F2x2 acc2{{0.f, 0.f}, {0.f, 0.f}};
  uint4 hn[NCH];
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    hn[i] = chunk_residual_bracketed(xv[i], hv[i], w_post[threadIdx.x + i * width], r, sb, coef, acc2);
    h_out[base + i * width] = hn[i];
  }
  const F2 r2 = block_rsqrt_mean_once(fold(acc2), red[1], width >> 5, inv_h, eps);
  const ScaleBracket sb2 = scale_bracket(r2);
#pragma unroll
  for (int i = 0; i < NCH; ++i)
    z_out[base + i * width] = chunk_scaled(hn[i], w_pre[threadIdx.x + i * width], r2, sb2);
}

// ------------------------------------------------------------------ with the combine fused in
// The boundary after the MoE sublayer takes as x the weighted sum of the
// token's K expert outputs (vLLM Beam summary, kernel change list: the norm
// kernel after the MoE also combines the top-8 outputs). x is formed in
// registers exactly as the separate combine forms it -- every row requested
// before the first is used, fp32 FMA in slot order from zero, one bf16
// rounding -- so the outputs are the bits of combine followed by the
// boundary, without writing or reading y. KMAX bounds K (register arrays).
template <int KMAX>
__global__ void __launch_bounds__(1024)
    boundary_combine_kernel(const uint4* h, const uint4* __restrict__ y_perm, const float* __restrict__ topk_w,
                            const int32_t* __restrict__ inv, int K, const uint4* __restrict__ w_post,
                            const uint4* __restrict__ w_pre, int nc, F2 inv_h, float eps, ResidualCoef coef,
                            uint4* h_out, uint4* __restrict__ z_out) {
  __shared__ F2 red[2][33];  // one per reduction: no barrier before reuse
  const int c = threadIdx.x;  // chunk owned by this thread
  const int t = blockIdx.x;
  const int nwarps = blockDim.x >> 5;
  const uint4 wp = w_post[c];  // weights do not come from the previous kernel
  const uint4 wq = w_pre[c];
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const size_t idx = static_cast<size_t>(t) * nc + c;
  const uint4 hv = h[idx];
  uint4 rows[KMAX];
  float wk[KMAX];
#pragma unroll
  for (int k = 0; k < KMAX; ++k) {
    rows[k] = make_uint4(0u, 0u, 0u, 0u);
    wk[k] = 0.f;
    if (k < K) {
      const int p = inv[static_cast<size_t>(t) * K + k];
      if (p >= 0) {
        wk[k] = topk_w[static_cast<size_t>(t) * K + k];
        rows[k] = y_perm[static_cast<size_t>(p) * nc + c];
      }
    }
  }
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int k = 0; k < KMAX; ++k) {
    if (k < K) {
      float f[8];
      unpack8(rows[k], f);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(wk[k], f[i], acc[i]);
    }
  }
  const uint4 xv = pack8(acc);
  F2x2 sq{{0.f, 0.f}, {0.f, 0.f}};
  acc_squares2s(sq, xv);
  const F2 r = block_rsqrt_mean_once(fold(sq), red[0], nwarps, inv_h, eps);
  F2x2 sq2{{0.f, 0.f}, {0.f, 0.f}};
  const uint4 hn = chunk_residual_bracketed(xv, hv, wp, r, scale_bracket(r), coef, sq2);
  h_out[idx] = hn;
  const F2 r2 = block_rsqrt_mean_once(fold(sq2), red[1], nwarps, inv_h, eps);
  z_out[idx] = chunk_scaled(hn, wq, r2, scale_bracket(r2));
}

}  // namespace

bool boundary_supported(int H) { return H > 0 && H % 256 == 0 && H <= 8192; }

cudaError_t launch_boundary_combine(const uint16_t* h, const uint16_t* y_perm, const float* topk_w,
                                    const int32_t* inv_perm, int K, const uint16_t* w_post, const uint16_t* w_pre,
                                    int T, int H, float eps, int n, uint16_t* h_out, uint16_t* z_out,
                                    cudaStream_t stream, bool pdl) {
  const ResidualCoef coef = residual_coef(n);
  const F2 inv_h = inv_hidden(H);
  auto kernel = K <= 8 ? boundary_combine_kernel<8> : boundary_combine_kernel<16>;
  const cudaError_t err = launch_kernel(
      kernel, dim3(T), dim3(H / 8), 0, stream, pdl, reinterpret_cast<const uint4*>(h),
      reinterpret_cast<const uint4*>(y_perm), topk_w, inv_perm, K, reinterpret_cast<const uint4*>(w_post),
      reinterpret_cast<const uint4*>(w_pre), H / 8, inv_h, eps, coef, reinterpret_cast<uint4*>(h_out),
      reinterpret_cast<uint4*>(z_out));
  ++launch_counter();
  return err;
}

cudaError_t launch_boundary(const uint16_t* h, const uint16_t* x, const uint16_t* w_post, const uint16_t* w_pre,
                            int T, int H, float eps, int n, uint16_t* h_out, uint16_t* z_out, cudaStream_t stream,
                            bool pdl, int* zero_slot) {
  const ResidualCoef coef = residual_coef(n);
  const F2 inv_h = inv_hidden(H);
  const uint4* hp = reinterpret_cast<const uint4*>(h);
  const uint4* xp = reinterpret_cast<const uint4*>(x);
  const uint4* wp = reinterpret_cast<const uint4*>(w_post);
  const uint4* wq = reinterpret_cast<const uint4*>(w_pre);
  uint4* ho = reinterpret_cast<uint4*>(h_out);
  uint4* zo = reinterpret_cast<uint4*>(z_out);
  // hidden size 5120 from 1024 tokens: four chunks per thread, 160 threads,
  // six blocks per SM (timed alone: 16384 tokens 193 -> 125 us, 2048 tokens
  // 26.7 -> 20.6 us against two chunks of per-element checks);
  // other sizes two chunks per thread from 1024 tokens when that still fills
  // whole warps; below 1024 tokens one chunk per thread, which keeps more
  // loads in flight (64 tokens 6.2 us against 8.2 us with four)
  cudaError_t err;
  if (T >= 1024 && H == 5120)
    err = launch_kernel(boundary_block_kernel<4, 160, 6>, dim3(T), dim3(160), 0, stream, pdl, hp, xp, wp, wq, H / 8,
                        inv_h, eps, coef, ho, zo, zero_slot);
  else if (T >= 1024 && H % 512 == 0)
    err = launch_kernel(boundary_block_kernel<2, 0, 1>, dim3(T), dim3(H / 16), 0, stream, pdl, hp, xp, wp, wq, H / 8,
                        inv_h, eps, coef, ho, zo, zero_slot);
  else
    err = launch_kernel(boundary_block_kernel<1, 0, 1>, dim3(T), dim3(H / 8), 0, stream, pdl, hp, xp, wp, wq, H / 8,
                        inv_h, eps, coef, ho, zo, zero_slot);
  ++launch_counter();
  return err;
}

}  // namespace beam
