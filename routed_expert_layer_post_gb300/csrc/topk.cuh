// Group-limited top-k for one token in one warp, for layouts where every
// group covers whole lanes (the router kernels).
#pragma once

#include "common.cuh"

namespace beam {

// Register top-k, for layouts where every group covers whole lanes: E = 32 *
// EPL experts with lane l holding experts l*EPL .. l*EPL + EPL - 1, and a
// group of E/G experts covering LPG = E/(G*EPL) consecutive lanes (Beam: EPL 8,
// LPG 4). Group top-2 sums come from lane-local top-2 pairs merged across the
// group's lanes; the TG groups are chosen by rank; the K experts by K rounds
// of a warp argmax (ties to the lower index), which also yields the slot
// order. The weights sum in slot order exactly as the generic kernel does.
template <int EPL, int LPG>
__device__ __forceinline__ void topk_lanes_token(const float* logits, const float* __restrict__ bias, int t, int G,
                                                 int TG, int K, float scale, int32_t* __restrict__ ids,
                                                 float* __restrict__ wout) {
  const int lane = threadIdx.x & 31;
  constexpr int E = 32 * EPL;
  float s[EPL], sb[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane * EPL + i;
    // L2 loads: the logits may have been written by other blocks of the same kernel
    s[i] = 1.0f / (1.0f + expf(-__ldcg(logits + static_cast<size_t>(t) * E + e)));
    sb[i] = s[i] + bias[e];
  }
  // group score: sum of the two largest biased scores of the group
  float top1 = -INFINITY, top2 = -INFINITY;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    if (sb[i] > top1) {
      top2 = top1;
      top1 = sb[i];
    } else if (sb[i] > top2) {
      top2 = sb[i];
    }
  }
#pragma unroll
  for (int o = 1; o < LPG; o <<= 1) {
    const float b1 = __shfl_xor_sync(kFullMask, top1, o);
    const float b2 = __shfl_xor_sync(kFullMask, top2, o);
    const float n1 = fmaxf(top1, b1);
    top2 = fmaxf(fminf(top1, b1), fmaxf(top2, b2));
    top1 = n1;
  }
  const float gs = (EPL * LPG >= 2) ? top1 + top2 : top1;
  const int my_group = lane / LPG;
  int rank = 0;
  for (int g = 0; g < G; ++g) {
    const float o = __shfl_sync(kFullMask, gs, g * LPG);
    rank += (o > gs) || (o == gs && g < my_group);
  }
  const bool chosen = rank < TG;  // same for every lane of a group
  // K rounds of argmax over the chosen groups' experts
  unsigned taken = 0;
  float s_sel = 0.f;
  int id_sel = 0;
  float total = 0.f;
  for (int k = 0; k < K; ++k) {
    float best = -INFINITY;
    int bi = 0x7fffffff;
    if (chosen) {
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        if (!((taken >> i) & 1u) && sb[i] > best) {  // strict: keeps the lower index on ties
          best = sb[i];
          bi = lane * EPL + i;
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(kFullMask, best, o);
      const int oi = __shfl_xor_sync(kFullMask, bi, o);
      if (ov > best || (ov == best && oi < bi)) {
        best = ov;
        bi = oi;
      }
    }
    const int owner = bi / EPL;
    float sv = 0.f;
    if (lane == owner) {
      const int i = bi - owner * EPL;
#pragma unroll
      for (int j = 0; j < EPL; ++j)
        if (j == i) sv = s[j];
      taken |= 1u << i;
    }
    sv = __shfl_sync(kFullMask, sv, owner);
    total += sv;
    if (lane == k) {
      s_sel = sv;
      id_sel = bi;
    }
  }
  if (lane < K) {
    ids[static_cast<size_t>(t) * K + lane] = id_sel;
    wout[static_cast<size_t>(t) * K + lane] = scale * s_sel / total;
  }
}

}  // namespace beam
