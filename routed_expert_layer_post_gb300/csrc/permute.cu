// Permutation of (token, slot) pairs by expert: histogram, exclusive prefix
// scan and a stable scatter, plus the row gather that lays the grouped GEMM's
// input out expert by expert.
//
// The vLLM Beam summary ("The fused decoding graph runs one MoE layer in 13
// kernels") feeds two grouped GEMMs from the routing kernels; a grouped GEMM
// needs each expert's rows contiguous. Pairs i = t*K + k are ordered by
// (expert, i), i.e. by (expert, token): a counting sort. Counts are summed
// with shared-memory atomics (order-free); every position is computed from
// counts and in-warp ranks (__match_any_sync), so no atomic decides an order
// and the result is deterministic.
//
// Kernels (one chunk = kChunk pairs per block):
//   count:   per-chunk histograms; the last block to finish (a ticket
//            counter, no waiting) scans them into expert offsets and per-chunk
//            bases, then resets the ticket;
//   scatter: per-warp counts, a block-level prefix over warps, then stable
//            positions -> perm_token, inv_perm;
//   gather:  x_perm[inv_perm[i]] = z[i / K], one warp per pair in pair order
//            so the K copies of a token row hit L2.
#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace beam {

namespace {

constexpr int kChunk = 2048;
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kPerWarp = kChunk / kWarps;  // 256 pairs, 8 batches of 32
constexpr int kMaxE = 256;

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__global__ void __launch_bounds__(kThreads)
    permute_count_kernel(const int32_t* __restrict__ ids, int total, int E, int nb, int* block_counts,
                         int* block_base, int* ticket, int32_t* __restrict__ offsets) {
  __shared__ int hist[kMaxE];
  __shared__ int s_last;
  __shared__ int s_tot[kMaxE];
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int tid = threadIdx.x;
  const int b = blockIdx.x;
  for (int e = tid; e < E; e += kThreads) hist[e] = 0;
  __syncthreads();
  const int beg = b * kChunk, end = min(total, beg + kChunk);
  for (int i = beg + tid; i < end; i += kThreads) {
    const int e = ids[i];
    if (e >= 0 && e < E) atomicAdd(&hist[e], 1);  // ids outside [0, E) are dropped
  }
  __syncthreads();
  for (int e = tid; e < E; e += kThreads) block_counts[static_cast<size_t>(b) * E + e] = hist[e];
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(ticket, 1) == nb - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // last block: per-expert running sums over chunks, then a scan over experts
  for (int e = tid; e < E; e += kThreads) {
    int run = 0;
    for (int c = 0; c < nb; ++c) {
      const int v = __ldcg(block_counts + static_cast<size_t>(c) * E + e);
      block_base[static_cast<size_t>(c) * E + e] = run;
      run += v;
    }
    s_tot[e] = run;
  }
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int e = 0; e < E; ++e) {
      const int v = s_tot[e];
      s_tot[e] = acc;
      offsets[e] = acc;
      acc += v;
    }
    offsets[E] = acc;
    *ticket = 0;
  }
  __syncthreads();
  for (int e = tid; e < E; e += kThreads) {
    const int off = s_tot[e];
    for (int c = 0; c < nb; ++c) block_base[static_cast<size_t>(c) * E + e] += off;
  }
}

__global__ void __launch_bounds__(kThreads)
    permute_scatter_kernel(const int32_t* __restrict__ ids, int total, int K, int E, const int* block_base,
                           int32_t* __restrict__ perm_token, int32_t* __restrict__ inv_perm) {
  __shared__ int wcnt[kWarps][kMaxE];
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int b = blockIdx.x;
  for (int i = tid; i < kWarps * kMaxE; i += kThreads) (&wcnt[0][0])[i] = 0;
  __syncthreads();
  const int wbeg = b * kChunk + w * kPerWarp;
  // pass A: per-warp counts
  for (int j = 0; j < kPerWarp; j += 32) {
    const int i = wbeg + j + lane;
    int e = i < total ? ids[i] : -1;
    if (e >= E) e = -1;
    const unsigned peers = __match_any_sync(kFullMask, e);
    if (e >= 0 && lane == __ffs(peers) - 1) wcnt[w][e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  // exclusive prefix over warps, starting from this chunk's base
  for (int e = tid; e < E; e += kThreads) {
    int acc = block_base[static_cast<size_t>(b) * E + e];
#pragma unroll
    for (int ww = 0; ww < kWarps; ++ww) {
      const int v = wcnt[ww][e];
      wcnt[ww][e] = acc;
      acc += v;
    }
  }
  __syncthreads();
  // pass B: stable positions
  for (int j = 0; j < kPerWarp; j += 32) {
    const int i = wbeg + j + lane;
    int e = i < total ? ids[i] : -1;
    if (e >= E || e < 0) {
      e = -1;
      if (i < total) inv_perm[i] = -1;  // dropped pair
    }
    const unsigned peers = __match_any_sync(kFullMask, e);
    int pos = 0;
    if (e >= 0) pos = wcnt[w][e] + __popc(peers & lanemask_lt());
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) wcnt[w][e] += __popc(peers);
    __syncwarp();
    if (e >= 0) {
      perm_token[pos] = i / K;
      inv_perm[i] = pos;
    }
  }
}

__global__ void __launch_bounds__(kThreads)
    gather_rows_kernel(const uint4* __restrict__ z, const int32_t* __restrict__ inv_perm, int total, int K,
                       int row_chunks, uint4* __restrict__ x_perm) {
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int i = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (i >= total) return;
  const int p = inv_perm[i];
  if (p < 0) return;
  const size_t src = static_cast<size_t>(i / K) * row_chunks;
  const size_t dst = static_cast<size_t>(p) * row_chunks;
  for (int c = lane; c < row_chunks; c += 32) x_perm[dst + c] = z[src + c];
}

// Small batches (T*K <= kChunk): one kernel. Every block recomputes the
// histogram, the scan and the stable positions of all pairs from the ids
// (at most 2048 of them, cheap), block 0 writes offsets / perm_token /
// inv_perm, and each block copies its share of rows into x_perm. No scratch,
// no ticket, no memset: it replaces the three-kernel path at decode sizes.
__global__ void __launch_bounds__(kThreads)
    permute_small_kernel(const int32_t* __restrict__ ids, int total, int K, int E, const uint4* __restrict__ z,
                         int row_chunks, int rows_per_block, int32_t* __restrict__ offsets,
                         int32_t* __restrict__ perm_token, int32_t* __restrict__ inv_perm, uint4* __restrict__ x_perm,
                         int* __restrict__ clear, int clear_ints) {
  __shared__ int s_ids[kChunk];
  __shared__ int s_pos[kChunk];
  __shared__ int wcnt[kWarps][kMaxE];
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  if (blockIdx.x == 0)  // zero what the next kernels expect zeroed (the experts' counters and tickets)
    for (int i = tid; i < clear_ints; i += kThreads) clear[i] = 0;
  const int padded = ((total + kWarps * 32 - 1) / (kWarps * 32)) * kWarps * 32;
  for (int i = tid; i < padded; i += kThreads) {
    int e = i < total ? ids[i] : -1;
    if (e >= E) e = -1;
    s_ids[i] = e < 0 ? -1 : e;
  }
  for (int i = tid; i < kWarps * kMaxE; i += kThreads) (&wcnt[0][0])[i] = 0;
  __syncthreads();
  // the pairs are split evenly over the warps (in order), 32 at a time
  const int per_warp = ((total + kWarps * 32 - 1) / (kWarps * 32)) * 32;
  const int wbeg = w * per_warp;
  for (int j = 0; j < per_warp; j += 32) {  // per-warp counts
    const int e = s_ids[wbeg + j + lane];
    const unsigned peers = __match_any_sync(kFullMask, e);
    if (e >= 0 && lane == __ffs(peers) - 1) wcnt[w][e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  if (w == 0) {  // exclusive scan over experts of the per-expert totals (warp 0, E <= 256)
    const int per_lane = (E + 31) / 32;
    int local = 0;
    for (int j = 0; j < per_lane; ++j) {
      const int e = lane * per_lane + j;
      if (e < E) {
        int t = 0;
#pragma unroll
        for (int ww = 0; ww < kWarps; ++ww) t += wcnt[ww][e];
        local += t;
      }
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(kFullMask, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - local;
    for (int j = 0; j < per_lane; ++j) {
      const int e = lane * per_lane + j;
      if (e < E) {
        if (blockIdx.x == 0) offsets[e] = run;
#pragma unroll
        for (int ww = 0; ww < kWarps; ++ww) {  // counts -> exclusive prefix over warps
          const int v = wcnt[ww][e];
          wcnt[ww][e] = run;
          run += v;
        }
      }
    }
    if (blockIdx.x == 0 && lane == 31) offsets[E] = incl;
  }
  __syncthreads();
  for (int j = 0; j < per_warp; j += 32) {  // stable positions
    const int i = wbeg + j + lane;
    const int e = s_ids[i];
    const unsigned peers = __match_any_sync(kFullMask, e);
    int pos = -1;
    if (e >= 0) pos = wcnt[w][e] + __popc(peers & lanemask_lt());
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) wcnt[w][e] += __popc(peers);
    __syncwarp();
    s_pos[i] = pos;
    if (blockIdx.x == 0 && i < total) {
      inv_perm[i] = pos;
      if (pos >= 0) perm_token[pos] = i / K;
    }
  }
  __syncthreads();
  if (x_perm == nullptr) return;
  // the block's rows as one flat range of 16-byte chunks over all threads,
  // four loads in flight per thread before their stores
  const int beg = blockIdx.x * rows_per_block, end = min(total, beg + rows_per_block);
  const int n = (end - beg) * row_chunks;
  for (int j0 = tid; j0 < n; j0 += 4 * kThreads) {
    uint4 v[4];
    int dst[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int j = j0 + u * kThreads;
      dst[u] = -1;
      if (j < n) {
        const int i = beg + j / row_chunks, c = j % row_chunks;
        const int pos = s_pos[i];
        if (pos >= 0) {
          v[u] = z[static_cast<size_t>(i / K) * row_chunks + c];
          dst[u] = pos * row_chunks + c;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (dst[u] >= 0) x_perm[dst[u]] = v[u];
  }
}

}  // namespace

size_t permute_scratch_bytes(int T, int K, int E) {
  const size_t total = static_cast<size_t>(T) * K;
  const size_t nb = (total + kChunk - 1) / kChunk;
  return (2 * nb * E + 64) * sizeof(int);
}

cudaError_t launch_permute(const int32_t* ids, const uint16_t* z, int T, int K, int E, int H, int32_t* offsets,
                           int32_t* perm_token, int32_t* inv_perm, uint16_t* x_perm, void* scratch,
                           cudaStream_t stream, bool pdl, void* clear, size_t clear_bytes) {
  const int total = T * K;
  if (total <= kChunk) {
    // the gather is latency-bound: spread the rows over up to 128 blocks
    const int rows_per_block = (total + 127) / 128;
    const int blocks = x_perm != nullptr ? (total + rows_per_block - 1) / rows_per_block : 1;
    const cudaError_t err = launch_kernel(
        permute_small_kernel, dim3(blocks), dim3(kThreads), 0, stream, pdl, ids, total, K, E,
        reinterpret_cast<const uint4*>(z), H / 8, rows_per_block, offsets, perm_token, inv_perm,
        reinterpret_cast<uint4*>(x_perm), static_cast<int*>(clear), static_cast<int>(clear_bytes / sizeof(int)));
    ++launch_counter();
    return err;
  }
  if (clear != nullptr && clear_bytes > 0) {
    const cudaError_t err = cudaMemsetAsync(clear, 0, clear_bytes, stream);
    if (err != cudaSuccess) return err;
  }
  const int nb = (total + kChunk - 1) / kChunk;
  int* base = static_cast<int*>(scratch);
  int* ticket = base;                       // 64 ints reserved at the front
  int* counts = base + 64;
  int* bbase = counts + static_cast<size_t>(nb) * E;
  cudaError_t err = cudaMemsetAsync(ticket, 0, sizeof(int), stream);
  if (err != cudaSuccess) return err;
  permute_count_kernel<<<nb, kThreads, 0, stream>>>(ids, total, E, nb, counts, bbase, ticket, offsets);
  ++launch_counter();
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  permute_scatter_kernel<<<nb, kThreads, 0, stream>>>(ids, total, K, E, bbase, perm_token, inv_perm);
  ++launch_counter();
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  if (x_perm != nullptr) {
    const int blocks = (total + kWarps - 1) / kWarps;
    gather_rows_kernel<<<blocks, kThreads, 0, stream>>>(reinterpret_cast<const uint4*>(z), inv_perm, total, K,
                                                         H / 8, reinterpret_cast<uint4*>(x_perm));
    ++launch_counter();
    err = cudaGetLastError();
  }
  return err;
}

}  // namespace beam
