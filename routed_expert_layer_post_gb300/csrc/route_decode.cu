// Decode-size routing in one launch: boundary -> FP32 router -> group top-k
// -> permutation -> row gather, for up to kMaxT tokens with Beam's expert
// layout (256 experts in 8 groups).
//
// Same arithmetic as the separate kernels (boundary.cu, router.cu,
// permute.cu; their page citations apply): the sandwich-norm boundary with
// bf16 rounding points, FP32 router logits with fp32 FMA, sigmoid + bias,
// top-2-sum group scores, TG groups, K experts, weights * routed_scale, and
// the stable (expert, token) order.
//
// One block per SM (one or two experts each), one thread per 8 hidden
// elements. At decode the token rows are ~10 KB, so every block recomputes the
// boundary for the tokens (it removes a launch and a round trip of z; one
// block per SM keeps the redundant arithmetic at one copy per SM), then dots z
// with its experts' router rows. The last block to finish (ticket counter)
// writes h' and z, runs the top-k for every token with the whole block and the
// permutation of the T*K pairs, clears the expert GEMMs' counters and
// tickets, raises the first ready flag (offsets and scratch valid), copies the
// permuted rows from the z it holds in registers and raises the second (rows
// valid). The experts launch that follows polls those flags instead of waiting
// for this kernel to end. With NVFP4 experts the permuted rows are written
// quantized instead (E2M1 codes and E4M3 block scales under the FP32 input
// scale, the same arithmetic as the standalone quantizer: TokenSpeed blog,
// "TensorRT-LLM NVFP4 MoE", input quantization does not depend on routing). Only the last block writes h': h' may alias h, and
// by then every block has read h. Ticket and flags are zeroed by the host
// before the launch; the ticket is left zero.
#include "common.cuh"
#include "kernels.h"
#include "norm_math.cuh"
#include "nvfp4.cuh"
#include "ptx.cuh"

namespace beam {

namespace {

using namespace norm;

constexpr int kMaxT = 8;
constexpr int kMaxPairs = 64;
constexpr int kMaxThreads = 640;  // H <= 5120
constexpr int kE = 256;           // experts (8 groups of 32)
constexpr int kMaxK = 16;

__device__ __forceinline__ void red_release(int* p, int v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Shared memory of the block top-k: up to two tokens at once (256 threads each)
struct TopkSmem {
  float sb[2][kE];       // biased scores
  float gs[2][8];        // group scores
  float slot_s[2][kMaxK];
  int slot_id[2][kMaxK];
};

// Group-limited top-k of token t over 256 experts in 8 groups of 32, one
// thread per expert (q) and one warp per group, by ranks: a candidate in the
// TG chosen groups takes slot r = the number of chosen candidates that beat
// it (higher biased score, ties to the lower index), which is the order K
// rounds of argmax would pick. Same values as the warp version (topk.cuh):
// the same sigmoid, group scores as the sum of the group's two largest biased
// scores (with multiplicity), weights normalised in slot order.
__device__ __forceinline__ void topk_block_phase1(const float* logits, float bias_q, int t, int q, int gi,
                                                  TopkSmem& sm, float& s_out) {
  const int lane = q & 31;
  const float l = __ldcg(logits + static_cast<size_t>(t) * kE + q);
  const float s = 1.0f / (1.0f + expf(-l));
  const float sb = s + bias_q;
  sm.sb[gi][q] = sb;
  float top1 = sb;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) top1 = fmaxf(top1, __shfl_xor_sync(kFullMask, top1, o));
  const unsigned eq = __ballot_sync(kFullMask, sb == top1);
  float v = (eq != 0u && lane == __ffs(eq) - 1) ? -INFINITY : sb;  // drop one instance of the maximum
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFullMask, v, o));
  if (lane == 0) sm.gs[gi][q >> 5] = top1 + v;
  if (q < kMaxK) {  // a slot no candidate takes (non-finite scores) reads as a dropped pair
    sm.slot_id[gi][q] = -1;
    sm.slot_s[gi][q] = 0.f;
  }
  s_out = s;
}

__device__ __forceinline__ void topk_block_phase2(int q, int gi, int TG, int K, float s, TopkSmem& sm) {
  unsigned chosen = 0;
#pragma unroll
  for (int g = 0; g < 8; ++g) {
    const float gv = sm.gs[gi][g];
    int rank = 0;
#pragma unroll
    for (int o = 0; o < 8; ++o) {
      const float ov = sm.gs[gi][o];
      rank += (ov > gv) || (ov == gv && o < g);
    }
    if (rank < TG) chosen |= 1u << g;
  }
  if (!((chosen >> (q >> 5)) & 1u)) return;
  const float sb = sm.sb[gi][q];
  int rank = 0;
  for (int g = 0; g < 8; ++g) {
    if (!((chosen >> g) & 1u)) continue;
    const float4* row = reinterpret_cast<const float4*>(&sm.sb[gi][g * 32]);
#pragma unroll
    for (int j4 = 0; j4 < 8; ++j4) {
      const float4 o = row[j4];
      const int j = g * 32 + j4 * 4;
      rank += (o.x > sb) || (o.x == sb && j < q);
      rank += (o.y > sb) || (o.y == sb && j + 1 < q);
      rank += (o.z > sb) || (o.z == sb && j + 2 < q);
      rank += (o.w > sb) || (o.w == sb && j + 3 < q);
    }
  }
  if (rank < K) {
    sm.slot_id[gi][rank] = q;
    sm.slot_s[gi][rank] = s;
  }
}

// One thread's 8 values (chunk c of a row) of an NVFP4 row: 16-value blocks
// are chunk pairs (c, c + 1), and the four scales of a 64-value slot come
// from chunks 8j .. 8j + 7 (lanes 8i .. 8i + 7 of a warp, since a warp's
// chunks are 32-aligned). Codes two per byte, element 2i in the low nibble.
// Every lane of the warp calls it.
__device__ __forceinline__ void store_row_fp4(const uint4& v, float g, int c, uint8_t* q_row, uint4* sf_row) {
  float f[8];
  unpack8(v, f);
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(f[i]));
  a = fmaxf(a, __shfl_xor_sync(kFullMask, a, 1));
  float d;
  const uint32_t sc = block_scale(a, g, &d);
  uint32_t word = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) word |= e2m1_code(f[i], d) << (4 * i);
  reinterpret_cast<uint32_t*>(q_row)[c] = word;
  // scale byte of block c / 2 at byte (c % 8) / 2 of slot c / 8
  uint32_t sw = (c & 1) ? 0u : sc << (8 * ((c & 7) >> 1));
  sw |= __shfl_xor_sync(kFullMask, sw, 2);
  sw |= __shfl_xor_sync(kFullMask, sw, 4);
  if ((c & 7) == 0) sf_row[c >> 3] = make_uint4(sw, 0u, 0u, 0u);
}

// TMAX: token capacity of the register arrays
template <int TMAX>
__global__ void __launch_bounds__(kMaxThreads, 1)
    route_decode_kernel(const uint4* h, const uint4* __restrict__ x, const uint4* __restrict__ w_post,
                        const uint4* __restrict__ w_pre, const float* __restrict__ W, const float* __restrict__ bias,
                        int T, int E, int G, int TG, int K, float scale, F2 inv_h, float eps, ResidualCoef coef,
                        uint4* h_out, uint4* __restrict__ z_out, float* __restrict__ logits,
                        int32_t* __restrict__ ids, float* __restrict__ wout, int32_t* __restrict__ offsets,
                        int32_t* __restrict__ perm_token, int32_t* __restrict__ inv_perm, uint4* __restrict__ x_perm,
                        uint8_t* __restrict__ xq, uint4* __restrict__ xsf, float g_in, int* sync,
                        int* __restrict__ clear, int clear_ints) {
  __shared__ F2 red[2][33];  // one per norm reduction
  __shared__ float fred[32], fred2[32];
  __shared__ int hist[256];
  __shared__ int s_pos[kMaxPairs];
  __shared__ int s_ids[kMaxPairs];
  __shared__ __align__(16) TopkSmem tk;
  __shared__ int s_last;
  const int c = threadIdx.x;  // 8-element chunk owned by this thread
  const int nc = blockDim.x;
  const int nwarps = nc >> 5;
  const int lane = c & 31, warp = c >> 5;
  // experts of this block: e0 and e1 (e1 < E for the first E - gridDim.x blocks)
  const int e0 = blockIdx.x, e1 = blockIdx.x + gridDim.x;
  const bool two = e1 < E;

  // constants first: they do not depend on the previous kernel
  const float4* wrow0 = reinterpret_cast<const float4*>(W + static_cast<size_t>(e0) * nc * 8);
  const float4* wrow1 = reinterpret_cast<const float4*>(W + static_cast<size_t>(two ? e1 : e0) * nc * 8);
  const float4 wa0 = __ldg(wrow0 + 2 * c), wb0 = __ldg(wrow0 + 2 * c + 1);
  const float4 wa1 = __ldg(wrow1 + 2 * c), wb1 = __ldg(wrow1 + 2 * c + 1);
  const uint4 wp = w_post[c];
  const uint4 wq = w_pre[c];
  const float bias_q = c < 2 * kE ? __ldg(bias + c % kE) : 0.f;  // the top-k's expert c % 256
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();

  uint4 hc[TMAX], zc[TMAX];
#pragma unroll
  for (int t = 0; t < TMAX; ++t) {
    hc[t] = make_uint4(0u, 0u, 0u, 0u);
    zc[t] = hc[t];
    if (t < T) {
      const size_t idx = static_cast<size_t>(t) * nc + c;
      const uint4 xv = x[idx];
      const uint4 hv = h[idx];
      F2x2 acc{{0.f, 0.f}, {0.f, 0.f}};
      F2x2 acc2{{0.f, 0.f}, {0.f, 0.f}};
      if constexpr (TMAX <= 4) {
        // the boundary kernel's bracketed chunks (the same bits); red[0] is
        // written again only after the next reduction's barriers
        acc_squares2s(acc, xv);
        const F2 r = block_rsqrt_mean_once(fold(acc), red[0], nwarps, inv_h, eps);
        hc[t] = chunk_residual_bracketed(xv, hv, wp, r, scale_bracket(r), coef, acc2);
        const F2 r2 = block_rsqrt_mean_once(fold(acc2), red[1], nwarps, inv_h, eps);
        zc[t] = chunk_scaled(hc[t], wq, r2, scale_bracket(r2));
      } else {
        // per-pair checks: with eight tokens' h' and z held in registers the
        // out-of-line calls of the bracketed form spill
        acc_squares2(acc, xv);
        const F2 r = block_rsqrt_mean(fold(acc), red[0], nwarps, inv_h, eps);
        hc[t] = chunk_residual(xv, hv, wp, r, coef, acc2);
        const F2 r2 = block_rsqrt_mean(fold(acc2), red[0], nwarps, inv_h, eps);
        zc[t] = chunk_scale(hc[t], wq, r2);
      }
      // router logits of the block's experts: z . W_r[e] in fp32 FMA, fixed reduction order
      float zf[8];
      unpack8(zc[t], zf);
      float d0 = 0.f, d1 = 0.f;
      d0 = fmaf(zf[0], wa0.x, d0);
      d0 = fmaf(zf[1], wa0.y, d0);
      d0 = fmaf(zf[2], wa0.z, d0);
      d0 = fmaf(zf[3], wa0.w, d0);
      d0 = fmaf(zf[4], wb0.x, d0);
      d0 = fmaf(zf[5], wb0.y, d0);
      d0 = fmaf(zf[6], wb0.z, d0);
      d0 = fmaf(zf[7], wb0.w, d0);
      d1 = fmaf(zf[0], wa1.x, d1);
      d1 = fmaf(zf[1], wa1.y, d1);
      d1 = fmaf(zf[2], wa1.z, d1);
      d1 = fmaf(zf[3], wa1.w, d1);
      d1 = fmaf(zf[4], wb1.x, d1);
      d1 = fmaf(zf[5], wb1.y, d1);
      d1 = fmaf(zf[6], wb1.z, d1);
      d1 = fmaf(zf[7], wb1.w, d1);
      d0 = warp_sum(d0);
      d1 = warp_sum(d1);
      if (lane == 0) {
        fred[warp] = d0;
        fred2[warp] = d1;
      }
      __syncthreads();
      if (warp == 0) {
        const float s0 = warp_sum(lane < nwarps ? fred[lane] : 0.f);
        const float s1 = warp_sum(lane < nwarps ? fred2[lane] : 0.f);
        if (lane == 0) {
          logits[static_cast<size_t>(t) * E + e0] = s0;
          if (two) logits[static_cast<size_t>(t) * E + e1] = s1;
        }
      }
      __syncthreads();
    }
  }

  // the last block to finish sees every expert's logits
  __threadfence();
  __syncthreads();
  int* ticket = sync;
  if (c == 0) s_last = (atomicAdd(ticket, 1) == static_cast<int>(gridDim.x) - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();

#pragma unroll
  for (int t = 0; t < TMAX; ++t) {
    if (t < T) {
      const size_t idx = static_cast<size_t>(t) * nc + c;
      h_out[idx] = hc[t];
      z_out[idx] = zc[t];
    }
  }

  // top-k, up to two tokens at once (256 threads each)
  const int ngrp = nc >= 2 * kE ? 2 : 1;
  const int gi = c / kE, q = c % kE;
  for (int t0 = 0; t0 < T; t0 += ngrp) {
    const int t = t0 + gi;
    const bool act = gi < ngrp && t < T;
    float s = 0.f;
    if (act) topk_block_phase1(logits, bias_q, t, q, gi, tk, s);
    __syncthreads();
    if (act) topk_block_phase2(q, gi, TG, K, s, tk);
    __syncthreads();
    if (act && q < K) {
      float total = 0.f;
      for (int k = 0; k < K; ++k) total += tk.slot_s[gi][k];
      const int id = tk.slot_id[gi][q];
      ids[static_cast<size_t>(t) * K + q] = id;
      wout[static_cast<size_t>(t) * K + q] = scale * tk.slot_s[gi][q] / total;
      s_ids[t * K + q] = id;
    }
    __syncthreads();
  }

  const int pairs = T * K;
  if (warp == 0) {
    // counts, exclusive scan over experts, stable positions in (expert, pair) order
    for (int i = lane; i < 256; i += 32) hist[i] = 0;
    __syncwarp();
    int my_e[2], my_i[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      my_i[q] = lane + 32 * q;
      my_e[q] = my_i[q] < pairs ? s_ids[my_i[q]] : -1;
      if (my_e[q] >= E) my_e[q] = -1;  // no valid choice (non-finite scores): dropped
      if (my_e[q] >= 0) atomicAdd(&hist[my_e[q]], 1);
    }
    __syncwarp();
    const int per_lane = (E + 31) / 32;
    int local = 0;
    for (int j = 0; j < per_lane; ++j) {
      const int ee = lane * per_lane + j;
      if (ee < E) local += hist[ee];
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(kFullMask, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - local;
    __syncwarp();
    for (int j = 0; j < per_lane; ++j) {
      const int ee = lane * per_lane + j;
      if (ee < E) {
        const int cnt = hist[ee];
        offsets[ee] = run;
        hist[ee] = run;  // becomes the expert's first position
        run += cnt;
      }
    }
    if (lane == 31) offsets[E] = incl;
    __syncwarp();
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      if (my_i[q] < pairs) {
        int pos = -1;
        if (my_e[q] >= 0) {
          int before = 0;  // earlier pairs with the same expert
          for (int j = 0; j < my_i[q]; ++j) before += (s_ids[j] == my_e[q]);
          pos = hist[my_e[q]] + before;
          perm_token[pos] = my_i[q] / K;
        }
        s_pos[my_i[q]] = pos;
        inv_perm[my_i[q]] = pos;
      }
    }
  }
  for (int j = c; j < clear_ints; j += nc) clear[j] = 0;
  // offsets, permutation and cleared scratch are published together (the
  // barrier orders every thread's stores before thread 0's release)
  __syncthreads();
  if (c == 0) red_release(sync + 1, 1);
  // permuted rows straight from the z this block holds (bf16, or NVFP4 codes and scales)
  for (int i = 0; i < pairs; ++i) {
    if (s_pos[i] < 0) continue;
    const int t = i / K;
    uint4 v = zc[0];
#pragma unroll
    for (int tt = 1; tt < TMAX; ++tt)
      if (tt == t) v = zc[tt];
    if (xq != nullptr)
      store_row_fp4(v, g_in, c, xq + static_cast<size_t>(s_pos[i]) * nc * 4, xsf + static_cast<size_t>(s_pos[i]) * (nc / 8));
    else
      x_perm[static_cast<size_t>(s_pos[i]) * nc + c] = v;
  }
  __syncthreads();
  if (c == 0) {
    red_release(sync + 2, 1);
    *ticket = 0;
  }
}

}  // namespace

int route_decode_blocks(int E, int num_sms) {
  return num_sms < E / 2 ? E / 2 : (num_sms > E ? E : num_sms);
}

bool route_decode_supported(int T, int H, int E, int G, int K) {
  return T >= 1 && T <= kMaxT && E == kE && G == 8 && K <= kMaxK && T * K <= kMaxPairs && H % 256 == 0 &&
         H / 8 >= kE && H / 8 <= kMaxThreads;
}

cudaError_t launch_route_decode(const uint16_t* h, const uint16_t* x, const uint16_t* w_post, const uint16_t* w_pre,
                                const float* W, const float* bias, int T, int H, int E, int G, int TG, int K,
                                float scale, float eps, int n, uint16_t* h_out, uint16_t* z_out, float* logits,
                                int32_t* ids, float* w, int32_t* offsets, int32_t* perm_token, int32_t* inv_perm,
                                uint16_t* x_perm, int* sync, void* clear, size_t clear_bytes, int num_sms,
                                cudaStream_t stream, bool pdl, bool sync_zeroed, uint8_t* xq, uint8_t* xsf,
                                float g_in) {
  cudaError_t err = cudaSuccess;
  if (!sync_zeroed && (err = cudaMemsetAsync(sync, 0, kRouteSyncInts * sizeof(int), stream)) != cudaSuccess)
    return err;
  const ResidualCoef coef = norm::residual_coef(n);
  const F2 inv_h = norm::inv_hidden(H);
  auto kernel = T <= 1 ? route_decode_kernel<1> : T <= 2 ? route_decode_kernel<2>
              : T <= 4 ? route_decode_kernel<4> : route_decode_kernel<8>;
  err = launch_kernel(kernel, dim3(route_decode_blocks(E, num_sms)), dim3(H / 8), 0, stream, pdl,
                      reinterpret_cast<const uint4*>(h),
                      reinterpret_cast<const uint4*>(x), reinterpret_cast<const uint4*>(w_post),
                      reinterpret_cast<const uint4*>(w_pre), W, bias, T, E, G, TG, K, scale, inv_h, eps, coef, reinterpret_cast<uint4*>(h_out), reinterpret_cast<uint4*>(z_out),
                      logits, ids, w, offsets, perm_token, inv_perm, reinterpret_cast<uint4*>(x_perm), xq,
                      reinterpret_cast<uint4*>(xsf), g_in, sync, static_cast<int*>(clear),
                      static_cast<int>(clear_bytes / sizeof(int)));
  ++launch_counter();
  return err;
}

}  // namespace beam
