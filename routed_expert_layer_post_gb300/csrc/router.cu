// FP32 router and group-limited top-k.
//
// TokenSpeed blog, "Fused FP32 routing": the router multiplies BF16
// activations by FP32 weights and returns FP32 scores; up to 16 tokens, one
// thread block per expert reads that expert's weights once for all tokens;
// larger batches run on FP32 CUDA cores; a single kernel then computes the
// sigmoid, bias addition, group top-k and the routing weights including the
// routed scale 2.5, all in FP32. vLLM Beam summary, "MoE and residual
// stream": the 5120 x 256 router keeps FP32 weights, accumulation and logits.
// Gaudi cookbook port, "Model code": the correction bias is about 28 for
// every expert, so lower precision erases the differences that pick experts.
//
// Arithmetic is plain fp32 FMA everywhere (no TF32, no bf16).
#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "topk.cuh"

namespace beam {

namespace {

// ------------------------------------------------------------------ small T
// One block per expert; each thread keeps its slice of the expert's weight
// row in registers and walks the tokens in groups of kTT.
constexpr int kSmallThreads = 256;
constexpr int kTT = 8;
constexpr int kSmallMaxT = 128;  // one block per expert up to here
constexpr int kFusedMaxT = 32;   // router + top-k in one launch up to here

// ------------------------------------------------------------------ large T
// Classic shared-memory SGEMM: block tile 64 tokens x 64 experts, k-slab 16,
// 256 threads with 4 x 4 outputs each, register-staged double buffering.
constexpr int kBM = 64, kBN = 64, kBK = 16;

__global__ void __launch_bounds__(256)
    router_sgemm_kernel(const uint16_t* __restrict__ z, const float* __restrict__ W, int T, int H, int E,
                        float* __restrict__ logits) {
  __shared__ __align__(16) float As[2][kBK][kBM + 4];
  __shared__ __align__(16) float Bs[2][kBK][kBN + 4];
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int tid = threadIdx.x;
  const int m0 = blockIdx.x * kBM;
  const int n0 = blockIdx.y * kBN;
  const int ty = tid >> 4, tx = tid & 15;
  // loader coordinates: row r = tid / 4, k quad kq = (tid % 4) * 4
  const int lr = tid >> 2, lk = (tid & 3) * 4;
  const int arow = min(m0 + lr, T - 1);  // clamp; rows >= T are never stored
  const uint16_t* aptr = z + static_cast<size_t>(arow) * H + lk;
  const float* bptr = W + static_cast<size_t>(min(n0 + lr, E - 1)) * H + lk;

  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  uint2 ra = *reinterpret_cast<const uint2*>(aptr);
  float4 rb = *reinterpret_cast<const float4*>(bptr);
  const int nk = H / kBK;
  for (int kt = 0; kt < nk; ++kt) {
    const int buf = kt & 1;
    As[buf][lk + 0][lr] = bf16_lo(ra.x);
    As[buf][lk + 1][lr] = bf16_hi(ra.x);
    As[buf][lk + 2][lr] = bf16_lo(ra.y);
    As[buf][lk + 3][lr] = bf16_hi(ra.y);
    Bs[buf][lk + 0][lr] = rb.x;
    Bs[buf][lk + 1][lr] = rb.y;
    Bs[buf][lk + 2][lr] = rb.z;
    Bs[buf][lk + 3][lr] = rb.w;
    __syncthreads();
    if (kt + 1 < nk) {
      ra = *reinterpret_cast<const uint2*>(aptr + (kt + 1) * kBK);
      rb = *reinterpret_cast<const float4*>(bptr + (kt + 1) * kBK);
    }
#pragma unroll
    for (int kk = 0; kk < kBK; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&As[buf][kk][ty * 4]);
      const float4 b = *reinterpret_cast<const float4*>(&Bs[buf][kk][tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w};
      const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    // the next iteration writes the other buffer; the barrier above already
    // separates it from the reads two iterations back
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m < T) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int n = n0 + tx * 4 + j;
        if (n < E) logits[static_cast<size_t>(m) * E + n] = acc[i][j];
      }
    }
  }
}

// ------------------------------------------------------------------ top-k
// One warp per token. Scores live in shared memory; groups and experts are
// selected by rank (the number of competitors that beat a candidate, with
// ties going to the lower index), which also yields the slot order.
constexpr int kTopkWarps = 4;
constexpr int kMaxE = 256;
constexpr int kMaxK = 16;

__global__ void __launch_bounds__(kTopkWarps * 32)
    topk_kernel(const float* __restrict__ logits, const float* __restrict__ bias, int T, int E, int G, int TG, int K,
                float scale, int32_t* __restrict__ ids, float* __restrict__ wout) {
  __shared__ float s_sb[kTopkWarps][kMaxE];
  __shared__ float s_s[kTopkWarps][kMaxE];
  __shared__ float s_gs[kTopkWarps][32];
  __shared__ float s_cs[kTopkWarps][kMaxK];
  __shared__ int s_ci[kTopkWarps][kMaxK];
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int wi = threadIdx.x >> 5;
  const int t = blockIdx.x * kTopkWarps + wi;
  if (t >= T) return;
  float* sb = s_sb[wi];
  float* sc = s_s[wi];
  for (int e = lane; e < E; e += 32) {
    const float l = logits[static_cast<size_t>(t) * E + e];
    const float s = 1.0f / (1.0f + expf(-l));
    sc[e] = s;
    sb[e] = s + bias[e];
  }
  __syncwarp();
  const int per = E / G;
  float gs = -INFINITY;
  if (lane < G) {
    float top1 = -INFINITY, top2 = -INFINITY;
    for (int i = 0; i < per; ++i) {
      const float v = sb[lane * per + i];
      if (v > top1) {
        top2 = top1;
        top1 = v;
      } else if (v > top2) {
        top2 = v;
      }
    }
    gs = per >= 2 ? top1 + top2 : top1;
    s_gs[wi][lane] = gs;
  }
  __syncwarp();
  bool chosen = false;
  if (lane < G) {
    int rank = 0;
    for (int g = 0; g < G; ++g) {
      const float o = s_gs[wi][g];
      rank += (o > gs) || (o == gs && g < lane);
    }
    chosen = rank < TG;
  }
  const unsigned gmask = __ballot_sync(kFullMask, chosen);
  for (int e = lane; e < E; e += 32) {
    if ((gmask >> (e / per)) & 1u) {
      const float v = sb[e];
      int rank = 0;
      for (unsigned m = gmask; m; m &= m - 1) {
        const int g = __ffs(m) - 1;
        for (int i = 0; i < per; ++i) {
          const int o = g * per + i;
          const float u = sb[o];
          rank += (u > v) || (u == v && o < e);
        }
      }
      if (rank < K) {
        s_ci[wi][rank] = e;
        s_cs[wi][rank] = sc[e];
      }
    }
  }
  __syncwarp();
  float total = 0.f;
  for (int k = 0; k < K; ++k) total += s_cs[wi][k];
  if (lane < K) {
    ids[static_cast<size_t>(t) * K + lane] = s_ci[wi][lane];
    wout[static_cast<size_t>(t) * K + lane] = scale * s_cs[wi][lane] / total;
  }
}

template <int EPL, int LPG>
__global__ void __launch_bounds__(kTopkWarps * 32)
    topk_lanes_kernel(const float* __restrict__ logits, const float* __restrict__ bias, int T, int G, int TG,
                      int K, float scale, int32_t* __restrict__ ids, float* __restrict__ wout) {
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int t = blockIdx.x * kTopkWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  topk_lanes_token<EPL, LPG>(logits, bias, t, G, TG, K, scale, ids, wout);
}

constexpr int kMaxQ = 8192 / 4 / kSmallThreads;  // float4 slices of a row per thread (H <= 8192)

// With `ticket` set (Beam's 256 experts in 8 groups only), the last block to
// finish also runs the register top-k for every token: the logits of all
// experts are in L2 by then, and one launch is saved. The ticket must be zero
// on entry (the layer's boundary kernel clears it); the last block leaves it
// at zero.
__global__ void __launch_bounds__(kSmallThreads)
    router_small_kernel(const uint16_t* __restrict__ z, const float* __restrict__ W, int T, int H, int E,
                        float* __restrict__ logits, const float* __restrict__ bias, int G, int TG, int K,
                        float scale, int32_t* __restrict__ ids, float* __restrict__ wout, int* ticket) {
  const int e = blockIdx.x;
  const int tid = threadIdx.x;
  const int nq = H / 4;  // float4 chunks per row
  const float4* wrow = reinterpret_cast<const float4*>(W + static_cast<size_t>(e) * H);
  __shared__ float red[kSmallThreads / 32][kTT];

  // the expert's weight row, read once for all tokens; every load is issued before any use
  float4 w[kMaxQ];
#pragma unroll
  for (int i = 0; i < kMaxQ; ++i) {
    const int q = tid + i * kSmallThreads;
    w[i] = q < nq ? __ldg(wrow + q) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // the weights do not depend on the previous kernel; z does
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  for (int t0 = 0; t0 < T; t0 += kTT) {
    uint2 zz[kTT][kMaxQ];
#pragma unroll
    for (int t = 0; t < kTT; ++t)
#pragma unroll
      for (int i = 0; i < kMaxQ; ++i) {
        const int q = tid + i * kSmallThreads;
        zz[t][i] = (t0 + t < T && q < nq)
                       ? *reinterpret_cast<const uint2*>(z + static_cast<size_t>(t0 + t) * H + 4 * q)
                       : make_uint2(0u, 0u);
      }
#pragma unroll
    for (int t = 0; t < kTT; ++t) {
      float a = 0.f;
#pragma unroll
      for (int i = 0; i < kMaxQ; ++i) {
        a = fmaf(bf16_lo(zz[t][i].x), w[i].x, a);
        a = fmaf(bf16_hi(zz[t][i].x), w[i].y, a);
        a = fmaf(bf16_lo(zz[t][i].y), w[i].z, a);
        a = fmaf(bf16_hi(zz[t][i].y), w[i].w, a);
      }
      const float sum = warp_sum(a);
      if ((tid & 31) == 0) red[tid >> 5][t] = sum;
    }
    __syncthreads();
    if (tid < kTT && t0 + tid < T) {
      float sum = 0.f;
#pragma unroll
      for (int w8 = 0; w8 < kSmallThreads / 32; ++w8) sum += red[w8][tid];
      logits[static_cast<size_t>(t0 + tid) * E + e] = sum;
    }
    __syncthreads();
  }
  if (ticket == nullptr) return;
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(ticket, 1) == static_cast<int>(gridDim.x) - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int t = tid >> 5; t < T; t += kSmallThreads / 32) topk_lanes_token<8, 4>(logits, bias, t, G, TG, K, scale, ids, wout);
  if (tid == 0) *ticket = 0;
}

}  // namespace

cudaError_t launch_router_logits(const uint16_t* z, const float* W, int T, int H, int E, float* logits,
                                 cudaStream_t stream, bool pdl) {
  cudaError_t err;
  if (T <= kSmallMaxT) {
    err = launch_kernel(router_small_kernel, dim3(E), dim3(kSmallThreads), 0, stream, pdl, z, W, T, H, E, logits,
                        static_cast<const float*>(nullptr), 0, 0, 0, 0.0f, static_cast<int32_t*>(nullptr),
                        static_cast<float*>(nullptr), static_cast<int*>(nullptr));
  } else {
    dim3 grid((T + kBM - 1) / kBM, (E + kBN - 1) / kBN);
    err = launch_kernel(router_sgemm_kernel, grid, dim3(256), 0, stream, pdl, z, W, T, H, E, logits);
  }
  ++launch_counter();
  return err;
}

bool router_topk_fusable(int T, int E, int G) { return T <= kFusedMaxT && E == 256 && G == 8; }

cudaError_t launch_router_topk_fused(const uint16_t* z, const float* W, const float* bias, int T, int H, int E,
                                     int G, int TG, int K, float scale, float* logits, int32_t* ids, float* w,
                                     int* ticket, cudaStream_t stream, bool pdl) {
  const cudaError_t err = launch_kernel(router_small_kernel, dim3(E), dim3(kSmallThreads), 0, stream, pdl, z, W, T,
                                        H, E, logits, bias, G, TG, K, scale, ids, w, ticket);
  ++launch_counter();
  return err;
}

cudaError_t launch_topk(const float* logits, const float* bias, int T, int E, int G, int TG, int K, float scale,
                        int32_t* ids, float* w, cudaStream_t stream, bool pdl) {
  const int blocks = (T + kTopkWarps - 1) / kTopkWarps;
  cudaError_t err;
  if (E == 256 && G == 8) {  // Beam's layout: 8 experts per lane, a group is 4 lanes
    err = launch_kernel(topk_lanes_kernel<8, 4>, dim3(blocks), dim3(kTopkWarps * 32), 0, stream, pdl, logits, bias,
                        T, G, TG, K, scale, ids, w);
  } else {
    err = launch_kernel(topk_kernel, dim3(blocks), dim3(kTopkWarps * 32), 0, stream, pdl, logits, bias, T, E, G, TG,
                        K, scale, ids, w);
  }
  ++launch_counter();
  return err;
}

}  // namespace beam
