// Routed SwiGLU experts: two grouped GEMMs on tcgen05 tensor cores fed by
// TMA, and the deterministic weighted combine.
//
// TokenSpeed blog, "TensorRT-LLM NVFP4 MoE": the MoE kernel runs both expert
// GEMMs, fuses SwiGLU into the first, and computes each token's weighted sum
// of expert outputs from the FP32 routing weights. vLLM Beam summary, "MoE
// and residual stream": 256 routed experts, d_ff 2560, no shared expert.
//
// Grouped GEMM (one kernel template, two modes):
//   mode 0 (gate/up): for expert e and a block of 128 intermediate columns f,
//     D_g = W_g[f-block] . X_e^T and D_u = W_u[f-block] . X_e^T, then
//     act[row][f] = bf16(silu(D_g) * D_u);
//   mode 1 (down):    for a block of 128 hidden columns,
//     D = W_d[h-block] . act_e^T, y_perm[row][h] = bf16(D).
// The weight block is the MMA's M = 128 operand and the expert's token rows
// the N operand (16..128): decode batches put 1-3 tokens on an expert, and
// this orientation keeps the tensor-core tile full of weights instead of
// padding M with absent tokens. Accumulators live in tensor memory (TMEM),
// double-buffered so the epilogue of one tile overlaps the MMAs of the next.
//
// A persistent CTA per SM takes work units from a global counter. A unit is
// (expert, row block, token tile, k-split). Experts' row counts are
// read from expert_offsets on the device; the host never synchronises. When
// there are too few tiles to fill the GPU (decode), the reduction dimension
// is split; partial sums go to the workspace and the last unit of a tile to
// finish (a ticket counter, no waiting) adds them in fixed split order, so
// the result does not depend on timing.
//
// Warp roles: warp 0 issues TMA loads into a shared-memory ring, warp 1
// issues tcgen05.mma from one thread, warps 2-5 read TMEM (each warp its
// 32-lane quarter) and write outputs. Every mbarrier wait is bounded in time;
// on timeout the CTA records a site code in g_device_error and unwinds.
#include "common.cuh"
#include "kernels.h"
#include "nvfp4.cuh"
#include "ptx.cuh"

#include <cuda.h>
#include <algorithm>
#include <cstring>
#include <mutex>

namespace beam {

__device__ int g_device_error = 0;

namespace {

// warp 0: scheduler + TMA producer; warp 1: MMA issuer; warps 2-5 and 6-9:
// two epilogue groups taking alternate units (each group covers the four
// TMEM lane quarters), so one group's split-K round trips overlap the other's
constexpr int kThreads = 320;
// The single-CTA GEMM adds a watcher warp (warp 10): in the fused launch it
// polls the token tiles' gate/up completion counters and mirrors them in
// shared memory, so the producer never waits on a global round trip (under
// full HBM load one takes several microseconds) to learn that a down unit's
// rows are complete.
constexpr int kWatchWarp = kThreads / 32;
// ... and a claim warp (warp 11), which takes unit ids from the launch's
// counter two units ahead of the producer and hands them over in shared
// memory: the atomic's round trip then overlaps two units' loads without the
// producer ever waiting on it (an NVFP4 unit's loads take about as long as
// that round trip under full HBM load).
constexpr int kClaimWarp = kWatchWarp + 1;
constexpr int kClaimDepth = 2;
constexpr int kGemmThreads = kThreads + 64;
constexpr int kMaxWatchTiles = 2048;  // token tiles the shared-memory mirror holds (one bit each)
constexpr int kEpiGroups = 2;
constexpr int kBM = 128;                     // weight rows per tile (MMA M)
constexpr int kBK = 64;                      // reduction elements per stage: 128 bytes of bf16
constexpr int kTileABytes = kBM * kBK * 2;   // 16 KB
constexpr int kMaxE = 256;
constexpr int kCtrlBytes = 4096;
constexpr int kSmemLimit = 227 * 1024;
constexpr uint64_t kTimeoutNs = 2000000000ull;  // 2 s per wait
constexpr uint64_t kDrainNs = 50000000ull;      // 50 ms while unwinding
constexpr int kQueue = 8;                       // depth of the work-unit queue in shared memory
constexpr int kMaxSplit = 20;                   // largest split-K factor (partials summed from registers)

// One GEMM phase: gate/up (kind 0: two accumulators, SwiGLU epilogue) or
// down (kind 1: one accumulator).
struct PhaseParams {
  CUtensorMap tmap_w;   // weights, 3-D: (k, row, plane); expert e owns planes e*planes .. +planes-1
  CUtensorMap tmap_x;   // activations, 2-D: (k, permuted row)
  CUtensorMap tmap_sfx; // NVFP4: activation scale slots, 2-D: (16-byte slot, permuted row)
  uint16_t* out;        // bf16 output (down; gate/up of the bf16 path)
  uint8_t* out_q;       // NVFP4 gate/up: codes of the SwiGLU output [rows][F/2]
  uint8_t* out_sf;      // NVFP4 gate/up: its scale slots [rows][F/64][16]
  const uint8_t* sfw;   // NVFP4: weight scales, 512-byte atoms [plane][row/128][k-step][4][512]
  const float* wscale;  // NVFP4: per-expert FP32 weight scales
  float xscale;         // NVFP4: FP32 scale of the activation operand
  float out_scale;      // NVFP4 gate/up: FP32 scale of the SwiGLU output it quantizes
  float* partials;      // split-K partial sums of this phase
  int* tickets;         // split-K tickets of this phase (zero before the launch)
  int n_mb;             // 128-row weight blocks per expert
  int ksteps;           // reduction length / 64
  int split;            // split-K factor
  int out_ld;           // output row length (F for gate/up, H for down)
  int planes;           // weight planes per expert: 2 for gate/up (gate rows, up rows), 1 for down
  int max_tiles;        // tiles the workspace was sized for
};

// MODE 0: gate/up only; MODE 1: down only; MODE 2: both phases in one launch
// (phase 0 = gate/up, phase 1 = down), the down units of a token tile waiting
// for the gate/up tiles that produce its rows.
struct GemmParams {
  PhaseParams ph[2];
  const int32_t* offsets;
  int* counter;          // dynamic unit counter (zero before the launch)
  int* done;             // MODE 2: gate/up row blocks finished per token tile (zero before the launch)
  int E;
  int rows;              // permuted rows (T * K)
  int max_token_tiles;   // MODE 2: size of `done`
  // MODE 2 (optional): flags of the routing kernel before this launch; [0]
  // set once offsets and scratch are valid, [1] once the activation rows are
  // (polled instead of waiting for that kernel to end)
  const int* ready;
};

constexpr int pow2_at_least(int v) {
  int p = 32;
  while (p < v) p <<= 1;
  return p;
}

// FP4 (NVFP4 operands, block-scaled MMAs): a k-step is 256 values, 128 bytes
// per row as for bf16's 64, so the tile geometry is the same; each stage also
// holds the weight scales (two 2 KB atom sets) and the activation scales
// (four 512-byte slot boxes per k-step), copied to tensor memory by the MMA
// thread (64 columns per stage).
template <int MODE, int BN, bool FP4 = false>
struct Cfg {
  static constexpr int kNAcc = MODE == 1 ? 1 : 2;   // accumulators of the widest phase
  static constexpr int kTileBBytes = BN * kBK * 2;
  // MODE 2 keeps a second activation slot so that a down unit can fill a
  // stage with two k-steps (two weight tiles, two activation tiles)
  static constexpr int kBSlots = MODE == 2 ? 2 : 1;
  static constexpr int kSfABytes = FP4 ? 2 * 2048 : 0;
  static constexpr int kSfBBytes = FP4 ? kBSlots * 2048 : 0;
  static constexpr int kSfAOff = kNAcc * kTileABytes + kBSlots * kTileBBytes;
  static constexpr int kSfBOff = kSfAOff + kSfABytes;
  static constexpr int kStageBytes = kSfBOff + kSfBBytes;
  static constexpr int kAccCols = kNAcc * BN;
  // two accumulator buffers in TMEM: the epilogue of one tile overlaps the
  // MMAs of the next (four were measured slower at decode)
  static constexpr int kAccBufs = 2;  // one per epilogue group
  static constexpr int kSfCols = FP4 ? 64 : 0;  // scale columns per stage: A at +0, B at +32
  static constexpr int kStagesSmem = (kSmemLimit - 1024 - kCtrlBytes) / kStageBytes;
  static constexpr int kStagesTmem = FP4 ? (512 - kAccBufs * kAccCols) / 64 : 12;
  static constexpr int kStagesRaw = kStagesSmem < kStagesTmem ? kStagesSmem : kStagesTmem;
  static constexpr int kStages = kStagesRaw > 12 ? 12 : kStagesRaw;
  static constexpr int kTmemCols = pow2_at_least(kAccBufs * kAccCols + kStages * kSfCols);
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kCtrlBytes;
  static constexpr int kXStep = FP4 ? 128 : kBK;   // TMA x coordinate of one k-step (bytes or elements)
  static_assert(kStageBytes % 1024 == 0, "stage must keep 1024-byte alignment");
  static_assert(kTmemCols <= 512, "TMEM holds 512 columns");
  static_assert(!FP4 || (MODE == 2 && BN <= 32), "NVFP4 runs the fused launch with token tiles of at most 32");
};

// Wait until phase `parity` of `bar` has completed. Gives up after `limit_ns`
// (or as soon as another role raised the abort flag, if `abort_flag` is set),
// recording `site` in g_device_error on timeout.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int site,
                                         uint64_t limit_ns) {
  const uint32_t addr = ptx::smem_u32(bar);
  if (ptx::mbar_try_wait(addr, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait(addr, parity)) return true;
    if ((it & 63u) == 0) {
      if (abort_flag != nullptr && *abort_flag) return false;
      if (ptx::globaltimer() - t0 > limit_ns) {
        if (abort_flag != nullptr) *abort_flag = 1;
        atomicCAS(&g_device_error, 0, site);
        return false;
      }
    }
  }
}

// Split-K ticket: one atomic with acquire-release semantics at GPU scope (the
// caller's partial stores, ordered before it by a CTA barrier, are released
// with it; the last arriver acquires the other CTAs' partials).
__device__ __forceinline__ int atom_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ void red_add_release(int* p, int v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Shared-memory bits with release/acquire semantics at CTA scope: the watcher
// warp sets a token tile's bit after its GPU-scope acquire of the tile's
// completion counter; the producer's acquire of the bit then orders the rows
// the counter published before its own loads.
__device__ __forceinline__ void smem_or_release(uint32_t* w, uint32_t bits) {
  asm volatile("red.release.cta.shared::cta.or.b32 [%0], %1;" ::"r"(ptx::smem_u32(w)), "r"(bits) : "memory");
}

__device__ __forceinline__ uint32_t smem_ld_acquire(const uint32_t* w) {
  uint32_t v;
  asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(ptx::smem_u32(w)) : "memory");
  return v;
}

// Wait (bounded) until *counter >= target; other CTAs of this launch raise it.
__device__ __forceinline__ bool wait_counter(const int* counter, int target, volatile int* abort_flag, int site,
                                             uint64_t limit_ns = kTimeoutNs) {
  if (ld_acquire(counter) >= target) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(64);
    if (ld_acquire(counter) >= target) return true;
    if ((it & 15u) == 0) {
      if (*abort_flag) return false;
      if (ptx::globaltimer() - t0 > limit_ns) {
        *abort_flag = 1;
        atomicCAS(&g_device_error, 0, site);
        return false;
      }
    }
  }
}

// A work unit: phase, expert e, weight row block mb, token tile tt (and its
// global index gtt), split s, and the phase-local tile index.
struct Unit {
  int phase, e, mb, tt, gtt, s, tile;
};

// Expert owning global token tile j: the largest e with s_ttstart[e] <= j
// (experts without rows start where the next one does).
__device__ __forceinline__ int tile_owner(int j, int E, const int* s_ttstart) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_ttstart[mid] <= j) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Tiles of a phase are laid out expert by expert, row block by row block,
// token tile fastest; expert e's tiles start at n_mb * s_ttstart[e].
// `rot0` (fused launch): phase-0 tiles are taken starting at tile rot0 (an
// expert boundary), wrapping around at n_tiles0; with `rot_down` the phase-1
// tiles are rotated to the same expert.
__device__ __forceinline__ Unit decode_unit(int u, int n_units0, const GemmParams& p, const int* s_ttstart,
                                            const int* s_ntt, int rot0 = 0, int n_tiles0 = 0,
                                            bool rot_down = false) {
  Unit r;
  r.phase = (u < n_units0) ? 0 : 1;
  const PhaseParams& ph = p.ph[r.phase];
  const int v = r.phase == 0 ? u : u - n_units0;
  r.tile = v / ph.split;
  r.s = v - r.tile * ph.split;
  if (rot0 != 0 && (r.phase == 0 || rot_down)) {
    const int rt = (rot0 / p.ph[0].n_mb) * ph.n_mb;      // the same first token tile
    const int nt = (n_tiles0 / p.ph[0].n_mb) * ph.n_mb;  // this phase's tiles
    r.tile += rt;
    if (r.tile >= nt) r.tile -= nt;
  }
  const int q = r.tile / ph.n_mb;
  r.e = tile_owner(q, p.E, s_ttstart);
  const int local = r.tile - ph.n_mb * s_ttstart[r.e];
  const int ntt = s_ntt[r.e];
  r.mb = local / ntt;
  r.tt = local - r.mb * ntt;
  r.gtt = s_ttstart[r.e] + r.tt;
  return r;
}

template <int MODE>
__device__ __forceinline__ int unit_kind(int phase) {
  return MODE == 2 ? phase : MODE;
}

template <int BN>
__device__ __forceinline__ void store_outputs(const PhaseParams& ph, int rows, int kind, const float (&v)[2][16],
                                              int c0, int valid, int row0, int col) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (c0 + j < valid) {
      const int row = row0 + c0 + j;
      if (row >= 0 && row < rows && col < ph.out_ld) {
        float val;
        if (kind == 0) {
          const float g = v[0][j];
          val = g / (1.0f + __expf(-g)) * v[1][j];
        } else {
          val = v[0][j];
        }
        ph.out[static_cast<size_t>(row) * ph.out_ld + col] = static_cast<uint16_t>(f2bf(val));
      }
    }
  }
}

// NVFP4 gate/up epilogue for one token column: `val` is this lane's SwiGLU
// output (column f, the tile's weight row). The 16 lanes of a 16-value group
// agree on its scale (largest |val| by shuffles) and lane pairs pack two
// codes per byte. Every lane of the warp calls it, with the same `ok`.
__device__ __forceinline__ void store_act_fp4(const PhaseParams& ph, float val, bool ok, int row, int f) {
  float a = ok ? fabsf(val) : 0.f;
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(kFullMask, a, o));
  float d;
  const uint32_t s = block_scale(a, ph.out_scale, &d);
  const uint32_t q = ok ? e2m1_code(val, d) : 0u;
  const uint32_t hi = __shfl_down_sync(kFullMask, q, 1);
  if (ok) {
    const size_t F = static_cast<size_t>(ph.out_ld);
    if ((f & 1) == 0) ph.out_q[static_cast<size_t>(row) * (F / 2) + (f >> 1)] = static_cast<uint8_t>(q | (hi << 4));
    if ((f & 15) == 0)
      ph.out_sf[static_cast<size_t>(row) * (F / 4) + (f >> 6) * 16 + ((f & 63) >> 4)] = static_cast<uint8_t>(s);
  }
}

// Index of the 2 KB scale-atom set of (plane, 128-row block, k-step).
__device__ __forceinline__ size_t sf_atoms(const PhaseParams& ph, int plane, int mb, int k) {
  return ((static_cast<size_t>(plane) * ph.n_mb + mb) * ph.ksteps + k) * 2048;
}

template <int MODE, int BN, bool FP4>
__global__ void __launch_bounds__(kGemmThreads, 1) moe_gemm_kernel(const __grid_constant__ GemmParams p) {
  using C = Cfg<MODE, BN, FP4>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tiles =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* ctrl = tiles + C::kStages * C::kStageBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);
  uint64_t* empty = full + C::kStages;
  uint64_t* tfull = empty + C::kStages;
  uint64_t* tempty = tfull + 4;
  uint64_t* qfull = tempty + 4;
  uint64_t* qempty = qfull + kQueue;
  uint64_t* drain = qempty + kQueue;
  uint64_t* cfull = drain + 1;          // a claimed unit id is in the slot
  uint64_t* cfree = cfull + kClaimDepth;  // the producer has taken it
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(cfree + kClaimDepth);
  // [0] abort; [2] routing flags never came; [4] the producer has finished;
  // [6] the routing rows flag was seen; per epilogue group g: [4g+1] last
  // arriver, [4g+3] current unit
  int* s_flags = reinterpret_cast<int*>(tmem_slot + 1);
  int* s_queue = s_flags + 8;
  int* s_off = s_queue + kQueue;
  int* s_ntt = s_off + kMaxE + 1;
  int* s_ttstart = s_ntt + kMaxE;
  uint32_t* s_tile_done = reinterpret_cast<uint32_t*>(s_ttstart + kMaxE + 1);  // MODE 2: watcher bits
  uint32_t* s_rows = reinterpret_cast<uint32_t*>(s_flags + 6);  // MODE 2: the routing rows flag was seen
  int* s_claim = reinterpret_cast<int*>(s_tile_done + kMaxWatchTiles / 32);  // claimed unit ids
  volatile int* abort_flag = s_flags;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      ptx::mbar_init(&full[i], 1);
      ptx::mbar_init(&empty[i], 1);
    }
    for (int a = 0; a < C::kAccBufs; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], 128);
    }
    for (int q = 0; q < kQueue; ++q) {
      ptx::mbar_init(&qfull[q], 1);
      ptx::mbar_init(&qempty[q], 2);  // released by the MMA thread and the epilogue leader
    }
    ptx::mbar_init(drain, 1);
    for (int c = 0; c < kClaimDepth; ++c) {
      ptx::mbar_init(&cfull[c], 1);
      ptx::mbar_init(&cfree[c], 1);
    }
    for (int i = 0; i < 8; ++i) s_flags[i] = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tensormap(&p.ph[0].tmap_w);
    ptx::prefetch_tensormap(&p.ph[0].tmap_x);
    if (MODE == 2) {
      ptx::prefetch_tensormap(&p.ph[1].tmap_w);
      ptx::prefetch_tensormap(&p.ph[1].tmap_x);
    }
    if (FP4) {
      ptx::prefetch_tensormap(&p.ph[0].tmap_sfx);
      ptx::prefetch_tensormap(&p.ph[1].tmap_sfx);
    }
  }
  if (warp == kWatchWarp && lane == 0) {
    // Touch the launch's scalar parameters now, while the previous kernel
    // runs: every role reads them right after the dependency resolves, and a
    // constant-cache miss then costs a global round trip on the path to the
    // first weight load.
    uint32_t sink = static_cast<uint32_t>(p.E + p.rows + p.max_token_tiles) ^
                    static_cast<uint32_t>(reinterpret_cast<uintptr_t>(p.offsets) ^
                                          reinterpret_cast<uintptr_t>(p.counter) ^ reinterpret_cast<uintptr_t>(p.done) ^
                                          reinterpret_cast<uintptr_t>(p.ready));
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const PhaseParams& q = p.ph[i];
      sink += static_cast<uint32_t>(q.n_mb + q.ksteps + q.split + q.out_ld + q.planes + q.max_tiles) ^
              static_cast<uint32_t>(reinterpret_cast<uintptr_t>(q.out) ^ reinterpret_cast<uintptr_t>(q.out_q) ^
                                    reinterpret_cast<uintptr_t>(q.out_sf) ^ reinterpret_cast<uintptr_t>(q.sfw) ^
                                    reinterpret_cast<uintptr_t>(q.wscale) ^ reinterpret_cast<uintptr_t>(q.partials) ^
                                    reinterpret_cast<uintptr_t>(q.tickets)) ^
              __float_as_uint(q.xscale) ^ __float_as_uint(q.out_scale);
    }
    asm volatile("" ::"r"(sink));
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, C::kTmemCols);
    ptx::tmem_relinquish();
  }
  // Programmatic dependent launch: everything above overlaps the previous
  // kernel. MODES 0 and 2 read that kernel's outputs (offsets, x_perm) and
  // wait here. The separate down GEMM (MODE 1) reads offsets and weights
  // written before its predecessor started, so it builds its tile table and
  // streams weight tiles now; only its activation loads and its epilogue wait
  // for the gate/up GEMM.
  // Every unit, the first included, comes from the launch's unit counter, so
  // unit ids are handed out in increasing order to CTAs that are running.
  // A down unit waits only on gate/up units (lower ids), which running CTAs
  // hold and complete without waiting on later units: the launch progresses
  // however many of its CTAs are resident (another kernel may hold SMs).
  // Thread 0 (the producer) requests its first id as soon as the counter is
  // known to be zeroed; the round trip overlaps the tile-table set-up.
  int u_first = 0;
  if (MODE != 1) {
    if (MODE == 2 && p.ready != nullptr) {
      if (tid == 0) {
        if (!wait_counter(p.ready, 1, abort_flag, 9)) s_flags[2] = 1;
        else u_first = atomicAdd(p.counter, 1);
      }
      __syncthreads();  // thread 0's acquire orders the offset and counter reads below
    } else {
      ptx::griddep_wait();
      if (tid == 0) u_first = atomicAdd(p.counter, 1);
    }
    ptx::griddep_launch_dependents();
  } else if (tid == 0) {
    // the down GEMM's counter was zeroed two kernels back (the permutation),
    // which completed before the gate/up GEMM let this launch start
    u_first = atomicAdd(p.counter, 1);
  }
  for (int i = tid; i <= p.E; i += kGemmThreads) s_off[i] = p.offsets[i];
  if (MODE == 2)
    for (int i = tid; i < kMaxWatchTiles / 32; i += kGemmThreads) s_tile_done[i] = 0u;
  __syncthreads();
  if (warp == 0) {
    // token tiles per expert and their exclusive prefix (lane l owns a contiguous block of experts)
    const int per_lane = (p.E + 31) / 32;
    int local = 0;
    for (int j = 0; j < per_lane; ++j) {
      const int e = lane * per_lane + j;
      if (e < p.E) {
        const int cnt = max(0, s_off[e + 1] - s_off[e]);
        const int ntt = (cnt + BN - 1) / BN;
        s_ntt[e] = ntt;
        local += ntt;
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
      if (e < p.E) {
        s_ttstart[e] = run;
        run += s_ntt[e];
      }
    }
    if (lane == 31) s_ttstart[p.E] = incl;
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int n_tt = s_ttstart[p.E];
  int n_tiles0 = n_tt * p.ph[0].n_mb;
  if (n_tiles0 > p.ph[0].max_tiles || (MODE == 2 && n_tt > p.max_token_tiles)) {
    if (tid == 0) atomicCAS(&g_device_error, 0, 100);
    n_tiles0 = 0;  // workspace too small for this routing: do nothing rather than overrun it
  }
  if (MODE == 2 && s_flags[2]) n_tiles0 = 0;  // the routing flags never came: do nothing
  const int n_units0 = n_tiles0 * p.ph[0].split;
  const bool watch = MODE == 2 && n_tt <= kMaxWatchTiles;  // the watcher warp mirrors the tiles' completion
  // Fused launch: the first wave of gate/up units goes to the last experts.
  // Their epilogues run first on every SM, with cold instructions under full
  // HBM load, and finish late; the down units of those experts come last, so
  // nothing waits on them. rot0 is the start of the earliest expert such that
  // the experts from it to the end hold at least one wave of units. With
  // NVFP4 experts (a quarter of the bytes per unit, so the first wave's
  // epilogues are not late) the down units follow the gate/up order instead:
  // one token 83.4 -> 81.3 us per layer; in bf16 that order measured 1 %
  // slower at one token. (Handing each token tile's down units out a few
  // tiles after its gate/up units, interleaved with the later gate/up units,
  // measured slower: 1.28 against 1.01 ms at 64 tokens with NVFP4 experts,
  // 128 against 122 us at one token in bf16.)
  int rot0 = 0;
  if (MODE == 2 && n_tiles0 > 0) {
    const int wave_tiles = (static_cast<int>(gridDim.x) + p.ph[0].split - 1) / p.ph[0].split;
    const int limit = n_tiles0 - wave_tiles;
    if (limit > 0) rot0 = p.ph[0].n_mb * s_ttstart[tile_owner(limit / p.ph[0].n_mb, p.E, s_ttstart)];
  }
  int n_units = n_units0;
  if (MODE == 2 && n_tiles0 > 0) {
    const int n_tiles1 = n_tt * p.ph[1].n_mb;
    if (n_tiles1 <= p.ph[1].max_tiles) n_units += n_tiles1 * p.ph[1].split;
  }
  auto decode = [&](int u) -> Unit { return decode_unit(u, n_units0, p, s_ttstart, s_ntt, rot0, n_tiles0, FP4); };

  if (warp == 0) {
    // ------------------------------------------------------------ scheduler + TMA producer
    // Units are handed out dynamically from a global counter (the next id
    // is requested while the current unit's loads are issued), so SMs that
    // stream faster take more units and all SMs finish together. Each unit
    // id is published to the MMA and epilogue warps through a small queue in
    // shared memory.
    if (lane == 0) {
      const uint64_t pol_w = ptx::policy_evict_first();  // weights stream through once
      const uint64_t pol_x = ptx::policy_evict_last();   // activation tiles are re-read per row block
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      bool ok = true;
      // MODE 1: activation (B) loads wait for the previous kernel; MODE 2 with
      // routing flags: they wait for the flag of the permuted rows. Until then
      // stages get their weight tile only and are remembered here.
      bool dep_ready = (MODE == 0) || (MODE == 2 && p.ready == nullptr);
      int npend = 0;
      int pend_stage[C::kStages], pend_k[C::kStages], pend_row[C::kStages];
      // the activation tile(s) of one stage (one k-step, or two for `two`),
      // with NVFP4 also their four 512-byte scale-slot boxes per k-step
      auto load_b = [&](const PhaseParams& phb, int sidx, int k, int row, bool two) {
        uint8_t* st = tiles + sidx * C::kStageBytes;
        ptx::tma_load_2d(st + C::kNAcc * kTileABytes, &phb.tmap_x, &full[sidx], k * C::kXStep, row, pol_x);
        if (two)
          ptx::tma_load_2d(st + C::kNAcc * kTileABytes + C::kTileBBytes, &phb.tmap_x, &full[sidx],
                           (k + 1) * C::kXStep, row, pol_x);
        if constexpr (FP4) {
          for (int h = 0; h < (two ? 2 : 1); ++h)
#pragma unroll
            for (int c = 0; c < 4; ++c)
              ptx::tma_load_2d(st + C::kSfBOff + h * 2048 + c * 512, &phb.tmap_sfx, &full[sidx],
                               (4 * (k + h) + c) * 16, row, pol_x);
        }
      };
      // MODE 2: the routing kernel's second flag (permuted rows valid), as
      // mirrored in shared memory by the watcher warp
      auto rows_seen = [&]() -> bool { return smem_ld_acquire(s_rows) != 0u; };
      auto release_pending = [&]() {
        if (MODE == 1) {
          ptx::griddep_wait();
          ptx::griddep_launch_dependents();
        } else {
          if (!rows_seen()) {
            const uint64_t t0 = ptx::globaltimer();
            for (uint32_t it = 1;; ++it) {
              __nanosleep(32);
              if (rows_seen()) break;
              if ((it & 15u) == 0 && (*abort_flag || ptx::globaltimer() - t0 > kTimeoutNs)) {
                if (!*abort_flag) {
                  *abort_flag = 1;
                  atomicCAS(&g_device_error, 0, 10);
                }
                ok = false;
                break;
              }
            }
          }
          asm volatile("fence.proxy.async.global;" ::: "memory");  // the TMA reads what generic stores wrote
        }
        for (int i = 0; i < npend; ++i) load_b(p.ph[0], pend_stage[i], pend_k[i], pend_row[i], false);
        npend = 0;
        dep_ready = true;
      };
      int ready_gtt = -1;  // MODE 2: the last token tile whose gate/up rows were seen complete
      // MODE 2: a down unit whose activation rows are not complete yet still
      // streams its weight tiles; its activation loads wait here (token tile
      // pend_gtt, first deferred unit pend_seq0) until the gate/up units of
      // that tile are done, the ring is full, or the unit queue would block
      int pend_gtt = -1, pend_seq0 = 0;
      bool pend_two[C::kStages];
      // MODE 2: has token tile j's gate/up output been seen complete? From
      // the watcher warp's shared-memory bits (no global round trip), or, for
      // more tiles than the bits hold, from the counter itself.
      auto tile_done = [&](int j) -> bool {
        if (watch) return (smem_ld_acquire(&s_tile_done[j >> 5]) >> (j & 31)) & 1u;
        return ld_acquire(p.done + j) >= p.ph[0].n_mb;
      };
      auto wait_tile = [&](int j) -> bool {
        if (!watch) return wait_counter(p.done + j, p.ph[0].n_mb, abort_flag, 8);
        if (tile_done(j)) return true;
        const uint64_t t0 = ptx::globaltimer();
        for (uint32_t it = 1;; ++it) {
          __nanosleep(32);
          if (tile_done(j)) return true;
          if ((it & 15u) == 0) {
            if (*abort_flag) return false;
            if (ptx::globaltimer() - t0 > kTimeoutNs) {
              *abort_flag = 1;
              atomicCAS(&g_device_error, 0, 8);
              return false;
            }
          }
        }
      };
      auto release_down = [&]() -> bool {
        if (!wait_tile(pend_gtt)) return false;
        asm volatile("fence.proxy.async.global;" ::: "memory");  // the TMA reads what generic stores wrote
        for (int i = 0; i < npend; ++i) load_b(p.ph[1], pend_stage[i], pend_k[i], pend_row[i], pend_two[i]);
        npend = 0;
        ready_gtt = pend_gtt;
        return true;
      };
      for (int seq = 0;; ++seq) {
        // unit ids: the first from the set-up, then from the claim warp
        int u = u_first;
        if (seq > 0) {
          const int c = (seq - 1) % kClaimDepth;
          u = -1;
          if (ok && wait_bar(&cfull[c], ((seq - 1) / kClaimDepth) & 1, abort_flag, 14, kTimeoutNs)) {
            u = *reinterpret_cast<volatile int*>(&s_claim[c]);
            ptx::mbar_arrive(&cfree[c]);
          }
        }
        if (u >= n_units || !ok) u = -1;
        if (u < 0 && !dep_ready) release_pending();
        if (MODE == 2 && npend > 0 && ok && (u < 0 || seq - pend_seq0 >= kQueue - 1)) {
          // the MMA warp may be waiting on a deferred stage: it frees no queue slot until it gets it
          if (!release_down()) {
            ok = false;
            u = -1;
          }
        }
        const int slot = seq % kQueue;
        if (!wait_bar(&qempty[slot], ((seq / kQueue) & 1) ^ 1u, abort_flag, 5, kTimeoutNs)) {
          ok = false;
          u = -1;
        }
        s_queue[slot] = u;
        ptx::mbar_arrive(&qfull[slot]);
        if (u < 0) {
          // the epilogue group that would take the next unit also needs the stop mark
          const int s2 = (seq + 1) % kQueue;
          wait_bar(&qempty[s2], (((seq + 1) / kQueue) & 1) ^ 1u, abort_flag, 5, kTimeoutNs);
          s_queue[s2] = -1;
          ptx::mbar_arrive(&qfull[s2]);
          break;
        }
        const Unit w = decode(u);
        const PhaseParams& ph = p.ph[w.phase];
        const int kind = unit_kind<MODE>(w.phase);
        const int nacc = kind == 0 ? 2 : 1;
        const uint32_t stage_bytes = nacc * kTileABytes + C::kTileBBytes + (FP4 ? nacc * 2048 + 2048 : 0);
        const int k0 = w.s * ph.ksteps / ph.split, k1 = (w.s + 1) * ph.ksteps / ph.split;
        const int row0 = s_off[w.e] + w.tt * BN;
        bool defer = false;
        if (MODE == 2 && w.phase == 1 && !dep_ready) release_pending();  // pending rows first: one list at a time
        if (MODE == 2 && w.phase == 1) {
          // this token tile's rows of `act` come from gate/up units held by
          // running CTAs (all gate/up units are handed out before any down
          // unit). Deferred stages are always the newest in the ring: a unit
          // of another token tile first releases them.
          if (npend > 0 && (pend_gtt != w.gtt || tile_done(pend_gtt))) {
            if (!release_down()) {
              ok = false;
              continue;
            }
          }
          if (w.gtt != ready_gtt) {
            if (npend == 0 && tile_done(w.gtt)) {
              asm volatile("fence.proxy.async.global;" ::: "memory");
              ready_gtt = w.gtt;
            } else {
              if (npend == 0) pend_seq0 = seq;
              pend_gtt = w.gtt;
              defer = true;
            }
          }
        }
        // k-steps per stage: 1, or 2 for down units of the fused launch
        const int kps = (MODE == 2 && kind == 1) ? 2 : 1;
        for (int k = k0; k < k1; k += kps) {
          if (MODE == 2 && npend == C::kStages) {
            // every stage holds a deferred tile: the MMA needs the activations now
            if (!release_down()) {
              ok = false;
              break;
            }
            defer = false;
          }
          if (!wait_bar(&empty[stage], phase ^ 1u, abort_flag, 1, kTimeoutNs)) {
            ok = false;
            break;
          }
          uint8_t* st = tiles + stage * C::kStageBytes;
          if (kps == 2) {
            const bool two = k + 1 < k1;
            ptx::mbar_arrive_expect_tx(&full[stage],
                                       (two ? 2u : 1u) * (kTileABytes + C::kTileBBytes + (FP4 ? 4096u : 0u)));
            ptx::tma_load_3d(st, &ph.tmap_w, &full[stage], k * C::kXStep, w.mb * kBM, w.e * ph.planes, pol_w);
            if (two)
              ptx::tma_load_3d(st + kTileABytes, &ph.tmap_w, &full[stage], (k + 1) * C::kXStep, w.mb * kBM,
                               w.e * ph.planes, pol_w);
            if constexpr (FP4) {
              for (int h = 0; h < (two ? 2 : 1); ++h)
                ptx::bulk_load(st + C::kSfAOff + h * 2048, ph.sfw + sf_atoms(ph, w.e * ph.planes, w.mb, k + h), 2048,
                               &full[stage], pol_w);
            }
            if (defer) {
              pend_stage[npend] = stage;
              pend_k[npend] = k;
              pend_row[npend] = row0;
              pend_two[npend] = two;
              ++npend;
            } else {
              load_b(ph, stage, k, row0, two);
            }
            ++issued;
            if (++stage == C::kStages) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          ptx::mbar_arrive_expect_tx(&full[stage], stage_bytes);
          ptx::tma_load_3d(st, &ph.tmap_w, &full[stage], k * C::kXStep, w.mb * kBM, w.e * ph.planes, pol_w);
          if (kind == 0)  // the up rows: the expert's second plane
            ptx::tma_load_3d(st + kTileABytes, &ph.tmap_w, &full[stage], k * C::kXStep, w.mb * kBM,
                             w.e * ph.planes + 1, pol_w);
          if constexpr (FP4) {
            for (int a = 0; a < nacc; ++a)
              ptx::bulk_load(st + C::kSfAOff + a * 2048, ph.sfw + sf_atoms(ph, w.e * ph.planes + a, w.mb, k), 2048,
                             &full[stage], pol_w);
          }
          if (MODE == 2 && !dep_ready && rows_seen()) release_pending();  // the rows just became valid
          if (dep_ready) {
            load_b(ph, stage, k, row0, false);
          } else {
            pend_stage[npend] = stage;
            pend_k[npend] = k;
            pend_row[npend] = row0;
            if (++npend == C::kStages) release_pending();  // the ring is full: the MMA needs these tiles
          }
          ++issued;
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      reinterpret_cast<volatile int*>(s_flags)[4] = 1;  // every unit issued: the watcher may stop
      if (!ok) {
        // unwinding: let the copies already in flight land before the CTA exits
        for (int i = 0; i < C::kStages && i < issued; ++i) {
          const uint32_t par = (i < stage) ? phase : (phase ^ 1u);
          wait_bar(&full[i], par, nullptr, 11, kDrainNs);
        }
      }
    }
  } else if (warp == kClaimWarp) {
    // ------------------------------------------------------------ unit claims
    // The producer took the first id in the set-up; every further id comes
    // from here, at most kClaimDepth ahead of the producer. Stops after
    // handing over an id past the end, or once the producer has finished or
    // the launch aborts.
    if (lane == 0) {
      const volatile int* producer_done = s_flags + 4;
      for (int i = 0;; ++i) {
        const int c = i % kClaimDepth;
        const uint32_t addr = ptx::smem_u32(&cfree[c]);
        const uint32_t par = ((i / kClaimDepth) & 1) ^ 1u;
        bool free_slot = ptx::mbar_try_wait(addr, par);
        const uint64_t t0 = free_slot ? 0 : ptx::globaltimer();
        while (!free_slot) {
          if (*producer_done || *abort_flag || ptx::globaltimer() - t0 > kTimeoutNs) break;
          __nanosleep(32);
          free_slot = ptx::mbar_try_wait(addr, par);
        }
        if (!free_slot) break;
        const int u = atomicAdd(p.counter, 1);
        *reinterpret_cast<volatile int*>(&s_claim[c]) = u;
        ptx::mbar_arrive(&cfull[c]);
        if (u >= n_units) break;
      }
    }
  } else if (warp == kWatchWarp) {
    // ------------------------------------------------------------ token-tile watcher (fused launch)
    // First the routing kernel's rows flag (when the launch polls flags), then
    // lane l polls the completion counters of token tiles l, l + 32, ...: up
    // to four not yet seen complete per round, their loads in flight together,
    // and sets the bit of each tile whose gate/up row blocks are all done.
    // Stops once the rows and every tile are seen complete, the producer has
    // finished, or the launch aborts; anything it never sees ends in the
    // producer's own bounded wait.
    if (MODE == 2) {
      const int target = p.ph[0].n_mb;
      const volatile int* producer_done = s_flags + 4;
      bool rows = p.ready == nullptr;  // without routing flags the rows were valid at launch
      if (rows && lane == 0) smem_or_release(s_rows, 1u);
      const uint64_t t0 = ptx::globaltimer();
      for (uint32_t it = 0;; ++it) {
        int tj[4], tv[4], cnt = 0;
        bool more = false;
        if (!rows) {
          if (lane == 0 && ld_acquire(p.ready + 1) >= 1) smem_or_release(s_rows, 1u);
          rows = __shfl_sync(kFullMask, static_cast<int>(smem_ld_acquire(s_rows)), 0) != 0;
          more = !rows;
        }
        for (int j = lane; watch && j < n_tt; j += 32) {
          if ((s_tile_done[j >> 5] >> (j & 31)) & 1u) continue;  // only this lane sets tile j's bit
          if (cnt == 4) {
            more = true;
            break;
          }
          tj[cnt++] = j;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (i < cnt) tv[i] = ld_acquire(p.done + tj[i]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (i < cnt) {
            if (tv[i] >= target) smem_or_release(&s_tile_done[tj[i] >> 5], 1u << (tj[i] & 31));
            else more = true;
          }
        }
        if (!__any_sync(kFullMask, more)) break;  // the rows and every tile seen complete
        if (*producer_done || *abort_flag) break;
        if (ptx::globaltimer() - t0 > kTimeoutNs) break;
        __nanosleep(128);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = FP4 ? ptx::idesc_nvf4(kBM, BN) : ptx::idesc_bf16_f32(kBM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int seq = 0;; ++seq) {
        const int slot = seq % kQueue;
        int u = -1;
        if (wait_bar(&qfull[slot], (seq / kQueue) & 1, abort_flag, 6, kTimeoutNs)) u = s_queue[slot];
        ptx::mbar_arrive(&qempty[slot]);
        if (u < 0) break;
        const Unit w = decode(u);
        const PhaseParams& ph = p.ph[w.phase];
        const int kind = unit_kind<MODE>(w.phase);
        const int nacc = kind == 0 ? 2 : 1;
        const int k0 = w.s * ph.ksteps / ph.split, k1 = (w.s + 1) * ph.ksteps / ph.split;
        const int kps = (MODE == 2 && kind == 1) ? 2 : 1;
        if (!wait_bar(&tempty[acc], acc_phase ^ 1u, abort_flag, 2, kTimeoutNs)) break;
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc * C::kAccCols);
        bool ok = true;
        for (int k = k0; k < k1; k += kps) {
          if (!wait_bar(&full[stage], phase, abort_flag, 3, kTimeoutNs)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = ptx::smem_u32(tiles + stage * C::kStageBytes);
          const uint32_t sb = sa + C::kNAcc * kTileABytes;
          const int nk = (kps == 2 && k + 1 < k1) ? 2 : 1;  // k-steps in this stage
          // NVFP4: the stage's scales into its tensor-memory columns (A sets at
          // +0: per plane, or per k-step for down; B sets at +32: per k-step),
          // 4 columns per 64-value chunk, before the MMAs that read them
          const uint32_t sf = tmem_base + static_cast<uint32_t>(C::kAccBufs * C::kAccCols + stage * C::kSfCols);
          if constexpr (FP4) {
            const int na = kps == 2 ? nk : nacc;
            for (int i = 0; i < na; ++i)
#pragma unroll
              for (int c = 0; c < 4; ++c) ptx::tmem_cp_32x128_x4(sf + (i * 4 + c) * 4, sa + C::kSfAOff + i * 2048 + c * 512);
            for (int h = 0; h < nk; ++h)
#pragma unroll
              for (int c = 0; c < 4; ++c)
                ptx::tmem_cp_32x128_x4(sf + 32 + (h * 4 + c) * 4, sa + C::kSfBOff + h * 2048 + c * 512);
          }
          if (kps == 2) {
            // two k-steps of one accumulator: (A0, B0) then (A1, B1)
            for (int h = 0; h < nk; ++h) {
#pragma unroll
              for (int j = 0; j < kBK / 16; ++j) {
                const uint64_t bdesc = ptx::smem_desc_k128(sb + h * C::kTileBBytes + j * 32);
                const uint64_t adesc = ptx::smem_desc_k128(sa + h * kTileABytes + j * 32);
                const uint32_t accum = (k > k0 || h > 0 || j > 0) ? 1u : 0u;
                if constexpr (FP4)
                  ptx::mma_nvf4(d, adesc, bdesc, idesc, sf + (h * 4 + j) * 4, sf + 32 + (h * 4 + j) * 4, accum);
                else
                  ptx::mma_bf16(d, adesc, bdesc, idesc, accum);
              }
            }
          } else {
#pragma unroll
            for (int j = 0; j < kBK / 16; ++j) {
              const uint64_t bdesc = ptx::smem_desc_k128(sb + j * 32);
#pragma unroll
              for (int a = 0; a < C::kNAcc; ++a) {
                if (a < nacc) {
                  const uint64_t adesc = ptx::smem_desc_k128(sa + a * kTileABytes + j * 32);
                  const uint32_t accum = (k > k0 || j > 0) ? 1u : 0u;
                  if constexpr (FP4)
                    ptx::mma_nvf4(d + a * BN, adesc, bdesc, idesc, sf + (a * 4 + j) * 4, sf + 32 + j * 4, accum);
                  else
                    ptx::mma_bf16(d + a * BN, adesc, bdesc, idesc, accum);
                }
              }
            }
          }
          ptx::mma_commit(&empty[stage]);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit(&tfull[acc]);
        if (++acc == C::kAccBufs) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // every MMA issued by this thread has completed once `drain` flips
      ptx::mma_commit(drain);
      wait_bar(drain, 0, nullptr, 12, kTimeoutNs);
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2-5)
    static_assert(C::kAccBufs == kEpiGroups, "epilogue group g owns accumulator buffer g");
    const int eg = (warp - 2) >> 2;  // epilogue group: units eg, eg + 2, ...
    const int sub = warp & 3;        // TMEM lane quarter this warp may access
    const int m = sub * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(sub * 32) << 16;
    const bool leader = (warp == 2 + 4 * eg && lane == 0);
    const uint32_t bar_id = 1 + eg;
    int* g_flags = s_flags + 4 * eg;
    if (MODE == 1) ptx::griddep_wait();  // tickets and partial sums were last used by the previous kernel
    const int acc = eg;
    uint32_t acc_phase = 0;
    for (int seq = eg;; seq += kEpiGroups) {
      if (leader) {
        const int slot = seq % kQueue;
        int u = -1;
        if (wait_bar(&qfull[slot], (seq / kQueue) & 1, abort_flag, 7, kTimeoutNs)) u = s_queue[slot];
        ptx::mbar_arrive(&qempty[slot]);
        int ready = 0;
        if (u >= 0) ready = wait_bar(&tfull[acc], acc_phase, abort_flag, 4, kTimeoutNs) ? 1 : 0;
        g_flags[3] = ready ? u : -1;
      }
      ptx::named_bar_sync(bar_id, 128);
      const int u = *reinterpret_cast<volatile int*>(&g_flags[3]);
      ptx::named_bar_sync(bar_id, 128);
      if (u < 0) break;
      ptx::tc_fence_after();
      const Unit w = decode(u);
      const PhaseParams& ph = p.ph[w.phase];
      const int kind = unit_kind<MODE>(w.phase);
      const int nacc = kind == 0 ? 2 : 1;
      const int row0 = s_off[w.e] + w.tt * BN;
      const int valid = min(BN, s_off[w.e + 1] - row0);
      const int col = w.mb * kBM + m;
      const uint32_t tb = tmem_base + lane_off + static_cast<uint32_t>(acc * C::kAccCols);
      // NVFP4: the MMA sums products of block-scaled values; the two FP32
      // scales (the expert's and the activation's) multiply the sum
      const float gs = FP4 ? __fmul_rn(ph.wscale[w.e], ph.xscale) : 1.0f;
      bool tile_done = false;  // this unit completed its tile's outputs
      bool released = false;   // the accumulator was already handed back
      if (ph.split == 1) {
        for (int c0 = 0; c0 < valid; c0 += 16) {
          uint32_t r[2][16];
#pragma unroll
          for (int a = 0; a < C::kNAcc; ++a)
            if (a < nacc) ptx::tmem_ld16(tb + a * BN + c0, r[a]);
          ptx::tmem_ld_wait();
          float v[2][16];
#pragma unroll
          for (int a = 0; a < 2; ++a)
#pragma unroll
            for (int j = 0; j < 16; ++j) v[a][j] = (a < C::kNAcc && a < nacc) ? __uint_as_float(r[a][j]) : 0.f;
          if constexpr (FP4) {
#pragma unroll
            for (int a = 0; a < 2; ++a)
#pragma unroll
              for (int j = 0; j < 16; ++j) v[a][j] = __fmul_rn(v[a][j], gs);
            if (kind == 0) {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float g = v[0][j];
                store_act_fp4(ph, g / (1.0f + __expf(-g)) * v[1][j], c0 + j < valid, row0 + c0 + j, col);
              }
              continue;
            }
          }
          store_outputs<BN>(ph, p.rows, kind, v, c0, valid, row0, col);
        }
        tile_done = true;
      } else {
        // The accumulator is read once, stored as this split's partial, and
        // handed back to the MMA warp at once: the ticket round trip and the
        // final sum (which reads every split's partial, this one included,
        // from global memory) no longer hold the tensor memory.
        const size_t slot_elems = static_cast<size_t>(nacc * BN) * kBM;
        float* mine = ph.partials + (static_cast<size_t>(w.tile) * ph.split + w.s) * slot_elems;
        for (int c0 = 0; c0 < valid; c0 += 16) {
          uint32_t r[2][16];
#pragma unroll
          for (int a = 0; a < C::kNAcc; ++a)
            if (a < nacc) ptx::tmem_ld16(tb + a * BN + c0, r[a]);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int a = 0; a < C::kNAcc; ++a)
            if (a < nacc)
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (c0 + j < valid) mine[static_cast<size_t>(a * BN + c0 + j) * kBM + m] = __uint_as_float(r[a][j]);
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(&tempty[acc]);
        released = true;
        // the barrier orders every thread's partial stores before the
        // leader's release; the leader's acquire and the second barrier order
        // the ticket before the partial loads of the last arriver
        ptx::named_bar_sync(bar_id, 128);
        if (leader) g_flags[1] = (atom_add_acq_rel(&ph.tickets[w.tile], 1) == ph.split - 1) ? 1 : 0;
        ptx::named_bar_sync(bar_id, 128);
        const int last = *reinterpret_cast<volatile int*>(&g_flags[1]);
        if (last) {
          // One output column at a time: partials requested eight splits at a
          // time and summed in split order (the result does not depend on
          // timing), then SwiGLU or the plain value, one store. The loops stay
          // rolled: this path runs once per tile at decode sizes (a handful of
          // columns), and its first run on an SM fetches its instructions
          // while HBM is saturated, so its size is its cost.
          const float* tile_parts = ph.partials + static_cast<size_t>(w.tile) * ph.split * slot_elems;
#pragma unroll 1
          for (int j = 0; j < valid; ++j) {
            float g = 0.f, u2 = 0.f;
            const size_t off0 = static_cast<size_t>(j) * kBM + m;
            const size_t off1 = static_cast<size_t>(BN + j) * kBM + m;
#pragma unroll 1
            for (int s0 = 0; s0 < ph.split; s0 += 8) {
              float x0[8], x1[8];
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const bool in = s0 + i < ph.split;
                x0[i] = in ? __ldcg(tile_parts + (s0 + i) * slot_elems + off0) : 0.f;
                x1[i] = (in && nacc > 1) ? __ldcg(tile_parts + (s0 + i) * slot_elems + off1) : 0.f;
              }
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                if (s0 + i < ph.split) {
                  g = (s0 + i == 0) ? x0[i] : g + x0[i];
                  u2 = (s0 + i == 0) ? x1[i] : u2 + x1[i];
                }
              }
            }
            const int row = row0 + j;
            if constexpr (FP4) {
              g = __fmul_rn(g, gs);
              u2 = __fmul_rn(u2, gs);
              if (kind == 0) {  // every lane of the group runs this column: the scale is shared
                store_act_fp4(ph, g / (1.0f + __expf(-g)) * u2, true, row, col);
                continue;
              }
            }
            if (row >= 0 && row < p.rows && col < ph.out_ld) {
              const float val = kind == 0 ? g / (1.0f + __expf(-g)) * u2 : g;
              ph.out[static_cast<size_t>(row) * ph.out_ld + col] = static_cast<uint16_t>(f2bf(val));
            }
          }
          if (leader) ph.tickets[w.tile] = 0;
          tile_done = true;
        }
        ptx::named_bar_sync(bar_id, 128);
      }
      if (MODE == 2 && w.phase == 0 && tile_done) {
        // publish this row block of the token tile to the down units waiting on it
        ptx::named_bar_sync(bar_id, 128);
        if (leader) red_add_release(p.done + w.gtt, 1);
      }
      if (!released) {
        ptx::tc_fence_before();
        ptx::mbar_arrive(&tempty[acc]);
      }
      acc_phase ^= 1u;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, C::kTmemCols);
  }
  // with routing flags the routing kernel may still be running: end after it,
  // so that kernels waiting on this one also see everything it wrote
  if (MODE == 2 && p.ready != nullptr) ptx::griddep_wait();
}

// ------------------------------------------------------------------ paired-SM GEMMs (prefill)
// At prefill sizes the expert GEMMs are tensor-core bound, and what holds the
// tensor pipe below its peak is how much MMA work the shared-memory ring
// covers while its loads are in flight (four 48 KB stages per SM above). A
// pair of CTAs on two SMs (a cluster of two) issues tcgen05.mma with
// cta_group::2: one M = 256, N = 256 MMA per 16-value slice, each CTA holding
// 128 rows of the weight operand and 128 of the 256 token rows, each CTA's
// tensor memory receiving its own 128 weight rows of the product (all 256
// tokens). A stage is then 32 KB per SM (16 KB of weights, 16 KB of tokens)
// for the same MMA work per SM, so six stages fit. Both CTAs' loads of a stage
// complete on the leader's barrier (TMA with .cta_group::2), which expects the
// pair's bytes, so the leader issues a stage's MMAs with no extra hop.
//
// Gate/up: a CTA's 128 weight rows are 64 gate rows and the up rows of the
// same 64 d_ff columns (one TMA box of 64 rows in both planes), so its
// accumulator holds gate in tensor-memory lanes 0-63 and up in lanes 64-127;
// the epilogue pairs them through shared memory for SwiGLU. A pair covers 128 d_ff columns. Down: 128
// rows of W_d per CTA, 256 per pair.
//
// Tile widths: an expert's rows rarely fill whole 256-token tiles (at 16384
// tokens and 256 experts, 256-wide tiles would compute 19 % empty columns).
// Its rows are cut into ceil(rows / 256) tiles of one width, a multiple of 32
// (pair_tile_width), and each runs as an MMA of width N = its rows rounded up
// to 32; each CTA then supplies N/2 token rows (CTA 0 the first half, CTA 1
// the second, so accumulator column c is still the tile's token c), from one
// 128-row box.
//
// Work: tiles (expert, weight row block, token tile) from the launch's
// unit counter, taken by the leader and published to both CTAs' queues (no
// tile waits on another). Roles (320 threads): warp 0 loads this CTA's
// halves; warp 1 of the leader CTA (cluster rank 0) issues the MMAs of a stage
// once both halves have landed and commits to both CTAs' barriers; warps 2-9
// are two epilogue groups taking alternate tiles, each CTA reading its own
// rows (the peer's groups release the accumulator with a remote arrive).
constexpr int kPairN = 256;                                        // tokens per tile
constexpr int kPairRows = 128;                                     // token rows per CTA
constexpr int kPairStageBytes = kTileABytes + kPairRows * kBK * 2;  // 32 KB
constexpr int kPairXchBytes = 2 * 64 * 16 * 4;                     // SwiGLU exchange, both groups
constexpr int kPairStages = (kSmemLimit - 1024 - kCtrlBytes - kPairXchBytes) / kPairStageBytes;
constexpr int kPairSmem = 1024 + kPairStages * kPairStageBytes + kPairXchBytes + kCtrlBytes;
constexpr int kPairTmemCols = 2 * kPairN;                          // two accumulator buffers

// MMA width (tokens) of a tile holding `valid` rows: the rows rounded up to
// 32, at most 256, so that the tensor cores skip empty columns; each CTA
// supplies half of the width.
__device__ __forceinline__ int pair_width(int valid) { return valid >= kPairN ? kPairN : (valid + 31) & ~31; }

// Token tiles of an expert with R rows: ceil(R / 256) tiles of one width, R
// over the tile count rounded up to 32 (the last tile takes the rest), e.g.
// 600 rows as 224 + 224 + 152 rather than 256 + 256 + 88. Every tile streams
// a whole weight tile, so balanced widths spread the MMA work evenly over
// them. The width is at most 256 and every tile holds at least one row (a
// width below 256 means at most seven tiles, and seven 32-row roundings fit
// in the rows past the first tile).
__device__ __forceinline__ int pair_tile_width(const int* s_off, const int* s_ntt, int e) {
  const int nt = s_ntt[e];
  return ((s_off[e + 1] - s_off[e] + nt - 1) / nt + 31) & ~31;
}
static_assert(kPairStages >= 6, "six 32 KB stages per SM");

// Bounded wait at cluster scope (for barriers the other CTA arrives on).
__device__ __forceinline__ bool wait_bar_cluster(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int site) {
  const uint32_t addr = ptx::smem_u32(bar);
  if (ptx::mbar_try_wait_cluster(addr, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait_cluster(addr, parity)) return true;
    if ((it & 63u) == 0) {
      if (abort_flag != nullptr && *abort_flag) return false;
      if (ptx::globaltimer() - t0 > kTimeoutNs) {
        if (abort_flag != nullptr) *abort_flag = 1;
        atomicCAS(&g_device_error, 0, site);
        return false;
      }
    }
  }
}

// MODE 0: gate/up + SwiGLU (ph[0], planes of F rows, tensor map box 64 rows);
// MODE 1: down (ph[0], one plane of H rows, box 128 rows).
template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    moe_gemm_pair_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tiles =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  float* xch = reinterpret_cast<float*>(tiles + kPairStages * kPairStageBytes);  // [group][16 columns][64 lanes]
  uint8_t* ctrl = tiles + kPairStages * kPairStageBytes + kPairXchBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(ctrl);  // leader: both halves of a stage landed
  uint64_t* empty = full + kPairStages;
  uint64_t* tfull = empty + kPairStages;
  uint64_t* tempty = tfull + 2;    // leader: both CTAs' epilogues released the accumulator
  uint64_t* qfull = tempty + 2;    // a unit id is in the queue slot (both CTAs)
  uint64_t* qempty = qfull + kQueue;  // leader: the slot's four readers are done with it
  uint64_t* drain = qempty + kQueue;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  int* s_flags = reinterpret_cast<int*>(tmem_slot + 1);  // [0] abort; [4g+3] group g's current unit
  int* s_queue = s_flags + 8;
  int* s_off = s_queue + kQueue;
  int* s_ntt = s_off + kMaxE + 1;
  int* s_ttstart = s_ntt + kMaxE;
  volatile int* abort_flag = s_flags;
  const PhaseParams& ph = p.ph[0];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = ptx::cluster_rank();
  const bool leader = rank == 0;
  if (tid == 0) {
    for (int i = 0; i < kPairStages; ++i) {
      ptx::mbar_init(&full[i], 1);
      ptx::mbar_init(&empty[i], 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(&tfull[a], 1);
      ptx::mbar_init(&tempty[a], 2);
    }
    for (int q = 0; q < kQueue; ++q) {
      ptx::mbar_init(&qfull[q], 1);
      ptx::mbar_init(&qempty[q], 4);  // leader: MMA thread and an epilogue group; peer: producer and a group
    }
    ptx::mbar_init(drain, 1);
    for (int i = 0; i < 8; ++i) s_flags[i] = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tensormap(&ph.tmap_w);
    ptx::prefetch_tensormap(&ph.tmap_x);
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(tmem_slot, kPairTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::griddep_wait();  // offsets, activation rows and the zeroed unit counter come from earlier kernels
  ptx::griddep_launch_dependents();
  int u_first = 0;
  if (leader && tid == 0) u_first = atomicAdd(p.counter, 1);  // the round trip overlaps the set-up below
  for (int i = tid; i <= p.E; i += kThreads) s_off[i] = p.offsets[i];
  __syncthreads();
  if (warp == 0) {
    const int per_lane = (p.E + 31) / 32;
    int local = 0;
    for (int j = 0; j < per_lane; ++j) {
      const int e = lane * per_lane + j;
      if (e < p.E) {
        const int ntt = (max(0, s_off[e + 1] - s_off[e]) + kPairN - 1) / kPairN;
        s_ntt[e] = ntt;
        local += ntt;
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
      if (e < p.E) {
        s_ttstart[e] = run;
        run += s_ntt[e];
      }
    }
    if (lane == 31) s_ttstart[p.E] = incl;
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // both CTAs' barriers exist before any remote arrive
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int n_units = s_ttstart[p.E] * ph.n_mb;
  const uint32_t qempty0 = ptx::cluster_addr(qempty, 0);  // the leader's
  const uint32_t qfull1 = ptx::cluster_addr(qfull, 1);    // the peer's
  const uint32_t queue1 = ptx::cluster_addr(s_queue, 1);

  if (warp == 0) {
    // ------------------------------------------------------------ unit queue + TMA producer (this CTA's halves)
    // The leader takes unit ids from the launch's counter in increasing
    // order (tiles sharing weights run at the same time on neighbouring
    // pairs, so the second reads them from L2) and publishes each id to both
    // CTAs' queues; the peer's producer and both CTAs' MMA and epilogue
    // roles read it from their own copy.
    if (lane == 0) {
      // a weight tile is read by the pairs running the expert's two or three
      // token tiles at about the same time: normal priority keeps it in L2
      // between them (evict-first measured 2 % slower at 16384 tokens)
      const uint64_t pol_w = ptx::policy_evict_normal();
      const uint64_t pol_x = ptx::policy_evict_last();
      const uint32_t full0 = ptx::cluster_addr(full, 0);
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      int u_next = u_first;
      for (int seq = 0;; ++seq) {
        const int slot = seq % kQueue;
        const uint32_t qpar = (seq / kQueue) & 1;
        int u;
        if (leader) {
          u = (u_next < n_units && ok) ? u_next : -1;
          const int nslots = u < 0 ? 2 : 1;  // the epilogue group of the next slot also needs the stop mark
          for (int i = 0; i < nslots; ++i) {
            const int sl = (seq + i) % kQueue;
            if (!wait_bar_cluster(&qempty[sl], (((seq + i) / kQueue) & 1) ^ 1u, abort_flag, 39)) u = -1;
            s_queue[sl] = u;
            asm volatile("st.shared::cluster.b32 [%0], %1;" ::"r"(queue1 + static_cast<uint32_t>(sl * 4)), "r"(u)
                         : "memory");
            ptx::mbar_arrive(&qfull[sl]);
            ptx::mbar_arrive_remote(qfull1 + static_cast<uint32_t>(sl * sizeof(uint64_t)));
          }
          if (u < 0) break;
          u_next = atomicAdd(p.counter, 1);  // the next id, while this unit's loads are issued
        } else {
          u = -1;
          if (wait_bar_cluster(&qfull[slot], qpar, abort_flag, 40)) u = s_queue[slot];
          ptx::mbar_arrive_remote(qempty0 + static_cast<uint32_t>(slot * sizeof(uint64_t)));
          if (u < 0 || !ok) break;
        }
        const Unit w = decode_unit(u, n_units, p, s_ttstart, s_ntt);
        const int tw = pair_tile_width(s_off, s_ntt, w.e);
        const int base_row = s_off[w.e] + w.tt * tw;
        const int half = pair_width(min(tw, s_off[w.e + 1] - base_row)) / 2;  // token rows this CTA supplies
        const int row0 = base_row + static_cast<int>(rank) * half;
        // one 128-row box per CTA whatever the width: the MMA reads the first
        // `half` rows. A box per 16 rows cost the producer one TMA
        // instruction per 16 rows (16384 tokens: both GEMMs 3-4 % slower).
        constexpr uint32_t stage_tx = 2u * static_cast<uint32_t>(kPairStageBytes);
        for (int k = 0; k < ph.ksteps; ++k) {
          if (!wait_bar(&empty[stage], phase ^ 1u, abort_flag, 31, kTimeoutNs)) {
            ok = false;
            break;
          }
          uint8_t* st = tiles + stage * kPairStageBytes;
          // both CTAs' loads complete on the leader's full barrier, which expects the pair's bytes
          const uint32_t fb = full0 + static_cast<uint32_t>(stage * sizeof(uint64_t));
          if (leader) ptx::mbar_arrive_expect_tx(&full[stage], stage_tx);
          if (MODE == 0) {
            const int f0 = w.mb * kBM + static_cast<int>(rank) * 64;
            // one box of both planes: the 64 gate rows, then the same 64 d_ff columns' up rows
            ptx::tma_load_3d_pair(st, &ph.tmap_w, fb, k * kBK, f0, 2 * w.e, pol_w);
          } else {
            ptx::tma_load_3d_pair(st, &ph.tmap_w, fb, k * kBK, w.mb * 2 * kBM + static_cast<int>(rank) * kBM, w.e,
                                  pol_w);
          }
          ptx::tma_load_2d_pair(st + kTileABytes, &ph.tmap_x, fb, k * kBK, row0, pol_x);
          ++issued;
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && leader) {
        // unwinding: let the copies already in flight land (the peer's land on these barriers too)
        for (int i = 0; i < kPairStages && i < issued; ++i) {
          const uint32_t par = (i < stage) ? phase : (phase ^ 1u);
          wait_bar(&full[i], par, nullptr, 32, kDrainNs);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader CTA only)
    if (lane == 0 && leader) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      for (int seq = 0;; ++seq) {
        const int slot = seq % kQueue;
        int u = -1;
        if (wait_bar(&qfull[slot], (seq / kQueue) & 1, abort_flag, 41, kTimeoutNs)) u = s_queue[slot];
        ptx::mbar_arrive(&qempty[slot]);
        if (u < 0) break;
        const Unit w = decode_unit(u, n_units, p, s_ttstart, s_ntt);
        const int tw = pair_tile_width(s_off, s_ntt, w.e);
        const int base_row = s_off[w.e] + w.tt * tw;
        const uint32_t idesc = ptx::idesc_bf16_f32(2 * kBM, pair_width(min(tw, s_off[w.e + 1] - base_row)));
        if (!wait_bar_cluster(&tempty[acc], acc_phase ^ 1u, abort_flag, 33)) break;
        ptx::tc_fence_after();
        const uint32_t d = tmem_base + static_cast<uint32_t>(acc * kPairN);
        bool ok = true;
        for (int k = 0; k < ph.ksteps; ++k) {
          if (!wait_bar_cluster(&full[stage], phase, abort_flag, 34)) {  // both halves landed
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = ptx::smem_u32(tiles + stage * kPairStageBytes);
          const uint32_t sb = sa + kTileABytes;
#pragma unroll
          for (int j = 0; j < kBK / 16; ++j)
            ptx::mma_bf16_pair(d, ptx::smem_desc_k128(sa + j * 32), ptx::smem_desc_k128(sb + j * 32), idesc,
                               (k > 0 || j > 0) ? 1u : 0u);
          ptx::mma_commit_pair(&empty[stage]);
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit_pair(&tfull[acc]);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      ptx::mma_commit_pair(drain);  // every MMA of the pair issued here has completed once `drain` flips
      wait_bar(drain, 0, nullptr, 36, kTimeoutNs);
    }
  } else {
    // ------------------------------------------------------------ epilogue groups (warps 2-5, 6-9)
    const int eg = (warp - 2) >> 2;
    const int sub = warp & 3;  // TMEM lane quarter
    const int m = sub * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(sub * 32) << 16;
    const uint32_t bar_id = 1 + eg;
    const bool group_leader = (warp == 2 + 4 * eg && lane == 0);
    int* g_unit = s_flags + 4 * eg + 3;
    float* x = xch + eg * 64 * 16;
    const uint32_t tempty_leader = ptx::cluster_addr(&tempty[eg], 0);
    uint32_t acc_phase = 0;
    for (int seq = eg;; seq += 2) {
      if (group_leader) {
        const int slot = seq % kQueue;
        int u = -1;
        if (wait_bar_cluster(&qfull[slot], (seq / kQueue) & 1, abort_flag, 42)) u = s_queue[slot];
        if (leader) ptx::mbar_arrive(&qempty[slot]);
        else ptx::mbar_arrive_remote(qempty0 + static_cast<uint32_t>(slot * sizeof(uint64_t)));
        if (u >= 0 && !wait_bar(&tfull[eg], acc_phase, abort_flag, 38, kTimeoutNs)) u = -1;
        *g_unit = u;
      }
      ptx::named_bar_sync(bar_id, 128);
      const int u = *reinterpret_cast<volatile int*>(g_unit);
      ptx::named_bar_sync(bar_id, 128);
      if (u < 0) break;
      ptx::tc_fence_after();
      const Unit w = decode_unit(u, n_units, p, s_ttstart, s_ntt);
      const int tw = pair_tile_width(s_off, s_ntt, w.e);
      const int row0 = s_off[w.e] + w.tt * tw;
      const int valid = min(tw, s_off[w.e + 1] - row0);
      const uint32_t tb = tmem_base + lane_off + static_cast<uint32_t>(eg * kPairN);
      for (int c0 = 0; c0 < valid; c0 += 16) {
        uint32_t r[16];
        ptx::tmem_ld16(tb + c0, r);
        ptx::tmem_ld_wait();
        if (MODE == 1) {
          const int col = w.mb * 2 * kBM + static_cast<int>(rank) * kBM + m;  // row of W_d = output column
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c0 + j < valid)
              ph.out[static_cast<size_t>(row0 + c0 + j) * ph.out_ld + col] =
                  static_cast<uint16_t>(f2bf(__uint_as_float(r[j])));
        } else {
          if (m >= 64) {
#pragma unroll
            for (int j = 0; j < 16; ++j) x[j * 64 + (m - 64)] = __uint_as_float(r[j]);
          }
          ptx::named_bar_sync(bar_id, 128);
          if (m < 64) {
            const int col = w.mb * kBM + static_cast<int>(rank) * 64 + m;  // d_ff column
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              if (c0 + j < valid) {
                const float g = __uint_as_float(r[j]);
                const float val = g / (1.0f + __expf(-g)) * x[j * 64 + m];
                ph.out[static_cast<size_t>(row0 + c0 + j) * ph.out_ld + col] = static_cast<uint16_t>(f2bf(val));
              }
            }
          }
          ptx::named_bar_sync(bar_id, 128);  // the exchange buffer is free again
        }
      }
      ptx::tc_fence_before();
      ptx::named_bar_sync(bar_id, 128);
      if (group_leader) {
        if (leader) ptx::mbar_arrive(&tempty[eg]);
        else ptx::mbar_arrive_remote(tempty_leader);
      }
      acc_phase ^= 1u;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // the leader's MMAs into the peer's tensor memory are done before either frees it
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, kPairTmemCols);
  }
}

// ------------------------------------------------------------------ combine
// y[t] = bf16(sum_k w[t][k] * y_perm[inv_perm[t*K+k]]), k in slot order, one
// thread per 8 hidden columns of a token; no atomics. KMAX bounds K: the
// register arrays hold KMAX rows, so K <= 8 (Beam) keeps registers low enough
// for four blocks per SM (the kernel is latency-bound on the row loads).
constexpr int kMaxTopK = 16;

// `err_out` (optional): one thread copies the device error word there once
// the expert launch before it has completed, so a host caller can read it
// from page-locked memory without a separate copy.
template <int KMAX>
__global__ void __launch_bounds__(256)
    combine_kernel(const uint4* __restrict__ y_perm, const float* __restrict__ w, const int32_t* __restrict__ inv,
                   int T, int K, int chunks, uint4* __restrict__ y, int* err_out) {
  ptx::griddep_wait();
  ptx::griddep_launch_dependents();
  if (err_out != nullptr && blockIdx.x == 0 && threadIdx.x == 0)
    *reinterpret_cast<volatile int*>(err_out) = *reinterpret_cast<volatile int*>(&g_device_error);
  const size_t idx = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<size_t>(T) * chunks) return;
  const int t = static_cast<int>(idx / chunks);
  const int c = static_cast<int>(idx - static_cast<size_t>(t) * chunks);
  // all K rows are requested before the first one is used
  uint4 rows[KMAX];
  float wk[KMAX];
#pragma unroll
  for (int k = 0; k < KMAX; ++k) {
    rows[k] = make_uint4(0u, 0u, 0u, 0u);
    wk[k] = 0.f;
    if (k < K) {
      const int p = inv[static_cast<size_t>(t) * K + k];
      if (p >= 0) {
        wk[k] = w[static_cast<size_t>(t) * K + k];
        rows[k] = y_perm[static_cast<size_t>(p) * chunks + c];
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
  y[idx] = pack8(acc);
}

// ------------------------------------------------------------------ bounded-wait check
// One thread waits, through the same bounded wait the fused launch uses for
// its cross-CTA counters and routing flags, on a flag that nothing sets: it
// must give up after `limit_ns`, record `site` and return.
__global__ void bounded_wait_probe_kernel(const int* flag, uint64_t limit_ns, int site) {
  __shared__ int abort_s;
  abort_s = 0;
  wait_counter(flag, 1, &abort_s, site, limit_ns);
}

// ------------------------------------------------------------------ tensor-core FP32 router
// logits[t][e] = sum_k z[t][k] * W[e][k] for prefill sizes. Each fp32 weight
// is split exactly into three bf16 terms, W = hi + mid + lo (hi = bf16(W),
// mid = bf16(W - hi), lo = W - hi - mid, which fits bf16 because W has 24
// significand bits). z is bf16, so every product is exact in fp32. The tensor
// core adds them in fp32 but does not round each addition like an IEEE adder,
// and over the whole reduction that measured 2.3e-5 of the row's largest
// logit, above the router's 1e-5 bar. So each 64-wide k-step (its three terms,
// 192 products) accumulates in a fresh TMEM buffer, and the epilogue adds the
// 80 k-step sums in fp32 registers in k order.
__global__ void __launch_bounds__(256)
    split_router_weights_kernel(const float* __restrict__ W, uint16_t* __restrict__ w3, size_t n) {
  ptx::griddep_wait();  // w3 may still be read by an earlier router launch
  ptx::griddep_launch_dependents();
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float w = W[i];
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const float r1 = __fsub_rn(w, __bfloat162float(hi));  // exact
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = __fsub_rn(r1, __bfloat162float(mid));  // exact, at most 8 significant bits
    w3[i] = __bfloat16_as_ushort(hi);
    w3[n + i] = __bfloat16_as_ushort(mid);
    w3[2 * n + i] = __bfloat16_as_ushort(__float2bfloat16_rn(r2));
  }
}

constexpr int kRtStages = 3;
constexpr int kRtThreads = 192;

// One CTA per (128 experts, BN tokens) tile. Warp 0 issues TMA: the three
// weight terms of a 64-wide k-step as one 3-D box, and the token tile. Warp 1
// issues 12 MMAs per k-step into one accumulator. Warps 2-5 read TMEM (lane =
// expert, column = token) and store fp32 logits.
template <int BN>
__global__ void __launch_bounds__(kRtThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmap_w3, const __grid_constant__ CUtensorMap tmap_z, int T,
                     int E, int ksteps, float* __restrict__ logits) {
  constexpr uint32_t kA = 3 * kTileABytes;
  constexpr uint32_t kStage = kA + BN * kBK * 2;
  static_assert(kStage % 1024 == 0, "stage must keep 1024-byte alignment");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* tiles =
      reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t full[kRtStages], empty[kRtStages], tfull[2], tempty[2];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN, m0 = blockIdx.y * kBM;
  constexpr uint32_t kCols = 2 * BN;  // two k-step buffers
  if (threadIdx.x == 0) {
    for (int i = 0; i < kRtStages; ++i) {
      ptx::mbar_init(&full[i], 1);
      ptx::mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&tfull[i], 1);
      ptx::mbar_init(&tempty[i], 128);
    }
    abort_s = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tensormap(&tmap_w3);
    ptx::prefetch_tensormap(&tmap_z);
  }
  if (warp == 1) {
    ptx::tmem_alloc(&tmem_slot, kCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abort_flag = &abort_s;
  ptx::griddep_wait();  // z and the split weights come from the previous kernels
  ptx::griddep_launch_dependents();

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = ptx::policy_evict_last();  // both operands are re-read by other CTAs
      int issued = 0;
      for (int k = 0; k < ksteps; ++k) {
        const int st = k % kRtStages;
        const uint32_t ph = (k / kRtStages) & 1;
        if (!wait_bar(&empty[st], ph ^ 1u, abort_flag, 20, kTimeoutNs)) break;
        uint8_t* s = tiles + st * kStage;
        ptx::mbar_arrive_expect_tx(&full[st], kStage);
        ptx::tma_load_3d(s, &tmap_w3, &full[st], k * kBK, m0, 0, pol);
        ptx::tma_load_2d(s + kA, &tmap_z, &full[st], k * kBK, n0, pol);
        ++issued;
      }
      if (issued < ksteps) {
        // unwinding: let the copies already in flight land before the CTA exits
        for (int i = issued > kRtStages ? issued - kRtStages : 0; i < issued; ++i)
          wait_bar(&full[i % kRtStages], (i / kRtStages) & 1, nullptr, 23, kDrainNs);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(kBM, BN);
      for (int k = 0; k < ksteps; ++k) {
        const int st = k % kRtStages;
        const int b = k & 1;
        if (!wait_bar(&tempty[b], ((k >> 1) & 1) ^ 1u, abort_flag, 24, kTimeoutNs)) break;
        if (!wait_bar(&full[st], (k / kRtStages) & 1, abort_flag, 21, kTimeoutNs)) break;
        ptx::tc_fence_after();
        const uint32_t a = ptx::smem_u32(tiles + st * kStage);
        const uint32_t bt = a + kA;
        const uint32_t d = tmem + static_cast<uint32_t>(b * BN);
#pragma unroll
        for (int s = 0; s < 3; ++s)
#pragma unroll
          for (int j = 0; j < kBK / 16; ++j)
            ptx::mma_bf16(d, ptx::smem_desc_k128(a + s * kTileABytes + j * 32), ptx::smem_desc_k128(bt + j * 32),
                          idesc, (s > 0 || j > 0) ? 1u : 0u);
        ptx::mma_commit(&empty[st]);
        ptx::mma_commit(&tfull[b]);
      }
    }
  } else {
    const int sub = warp & 3;
    const int e = m0 + sub * 32 + lane;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(sub * 32) << 16);
    float acc[BN];
#pragma unroll
    for (int i = 0; i < BN; ++i) acc[i] = 0.f;
    bool ok = true;
    for (int k = 0; k < ksteps && ok; ++k) {
      const int b = k & 1;
      if (!wait_bar(&tfull[b], (k >> 1) & 1, abort_flag, 22, kTimeoutNs)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
#pragma unroll
      for (int c0 = 0; c0 < BN; c0 += 16) {
        uint32_t r[16];
        ptx::tmem_ld16(lane_base + static_cast<uint32_t>(b * BN + c0), r);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[c0 + j] = __fadd_rn(acc[c0 + j], __uint_as_float(r[j]));
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&tempty[b]);
    }
    if (ok) {
#pragma unroll
      for (int i = 0; i < BN; ++i) {
        const int t = n0 + i;
        if (t < T && e < E) logits[static_cast<size_t>(t) * E + e] = acc[i];
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kCols);
  }
}

// ------------------------------------------------------------------ host side
using EncodeFn = decltype(&cuTensorMapEncodeTiled);

EncodeFn get_encode_fn() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(ptr);
  });
  return fn;
}

bool encode_map(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                const cuuint32_t* box, CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeFn fn = get_encode_fn();
  if (fn == nullptr) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, dtype, rank, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE, int BN, bool FP4 = false>
cudaError_t launch_mode_bn(const GemmParams& prm, int grid, cudaStream_t stream, bool pdl) {
  using C = Cfg<MODE, BN, FP4>;
  static std::once_flag once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  cudaError_t attr_err = cudaSuccess;
  std::call_once(once[dev & 63], [&] {
    attr_err = cudaFuncSetAttribute(moe_gemm_kernel<MODE, BN, FP4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    C::kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const cudaError_t err =
      launch_kernel(moe_gemm_kernel<MODE, BN, FP4>, dim3(grid), dim3(kGemmThreads), C::kSmemBytes, stream, pdl, prm);
  ++launch_counter();
  return err;
}

template <int MODE>
cudaError_t launch_mode(int bn, const GemmParams& prm, int grid, cudaStream_t stream, bool pdl) {
  switch (bn) {
    case 16: return launch_mode_bn<MODE, 16>(prm, grid, stream, pdl);
    case 32: return launch_mode_bn<MODE, 32>(prm, grid, stream, pdl);
    case 64: return launch_mode_bn<MODE, 64>(prm, grid, stream, pdl);
    default: return launch_mode_bn<MODE, 128>(prm, grid, stream, pdl);
  }
}

// the down GEMM also has a 256-token tile (its single accumulator fits TMEM twice)
template <>
cudaError_t launch_mode<1>(int bn, const GemmParams& prm, int grid, cudaStream_t stream, bool pdl) {
  switch (bn) {
    case 16: return launch_mode_bn<1, 16>(prm, grid, stream, pdl);
    case 32: return launch_mode_bn<1, 32>(prm, grid, stream, pdl);
    case 64: return launch_mode_bn<1, 64>(prm, grid, stream, pdl);
    case 128: return launch_mode_bn<1, 128>(prm, grid, stream, pdl);
    default: return launch_mode_bn<1, 256>(prm, grid, stream, pdl);
  }
}

int accum_cols(int mode, int bn) { return (mode == 0 ? 2 : 1) * bn; }

}  // namespace

GemmPlan plan_gemm(int mode, int T, int K, int E, int H, int F, int num_sms, int units_per_sm, bool fp4) {
  GemmPlan plan{};
  const long long entries = static_cast<long long>(T) * K;
  const long long touched = entries < E ? entries : E;
  const double r = touched > 0 ? static_cast<double>(entries) / static_cast<double>(touched) : 1.0;
  // token tile: the smallest width holding the mean rows per expert with some
  // slack; up to 128 for gate/up (two accumulators) and 256 for down, where
  // the wider tile halves the operand bytes per MMA at prefill sizes (NVFP4:
  // up to 32, the rows one lane quarter holds the activation scales of)
  const int bn_max = fp4 ? 32 : (mode == 0 ? 128 : 256);
  int bn = 16;
  while (bn < bn_max && 1.25 * r > bn) bn <<= 1;
  const int n_mb = mode == 0 ? (F + kBM - 1) / kBM : H / kBM;
  // a k-step is 128 bytes of each weight row: 64 bf16 or 256 NVFP4 values
  const int kstep = fp4 ? 256 : kBK;
  const int ksteps = mode == 0 ? H / kstep : F / kstep;
  plan.bn = bn;
  plan.max_token_tiles = static_cast<int>(touched + entries / bn);
  plan.max_tiles = plan.max_token_tiles * n_mb;
  const long long per_expert = static_cast<long long>((r + bn - 1) / bn);
  const long long est = touched * (per_expert > 0 ? per_expert : 1) * n_mb;
  // Units are handed out dynamically, so balance depends on how small the
  // last units are: when tiles are few (decode), split the reduction until
  // there are at least `units_per_sm` units per SM, keeping at least 128 KB
  // of weights per unit (4 k-steps of gate+up rows, 8 of down rows; NVFP4
  // down units 64 KB, below) so that
  // the per-unit epilogue stays hidden behind the next unit's loads. Only
  // narrow token tiles (<= 64) are split: the final sum of a split tile
  // walks its columns one at a time, which costs more than the balance gains
  // once a tile holds 128 or 256 columns (few experts with many rows each).
  // NVFP4 down units may hold 4 k-steps (64 KB of codes): at one token the
  // finer down units shorten the tail, 79.9 -> 78.2 us per layer
  const int min_ksteps = mode == 0 ? 4 : (fp4 ? 4 : 8);
  int split = 1;
  const long long target = static_cast<long long>(units_per_sm) * num_sms;
  if (est < target && bn <= 64) {
    for (int s = 2; s <= ksteps && s <= kMaxSplit; ++s) {
      if (ksteps % s != 0) continue;
      if (ksteps / s < min_ksteps) break;
      split = s;
      if (est * s >= target) break;
    }
  }
  plan.split = split;
  // prefill sizes: paired-SM tiles of 256 tokens once the mean rows per
  // expert fill them (the tensor-core-bound regime); no split then
  plan.pair = !fp4 && split == 1 && r >= 192.0 && H % (2 * kBM) == 0 && F % kBM == 0;
  if (plan.pair) {
    plan.max_token_tiles = static_cast<int>(touched + entries / kPairN);
    plan.max_tiles = plan.max_token_tiles * (mode == 0 ? F / kBM : H / (2 * kBM));
  }
  return plan;
}

namespace {

// Scratch shared by one gate/up + down pass:
//   [0, 256)      the dynamic unit counters (one per launch)
//   tickets0/1    split-K tickets of each phase
//   done          gate/up row blocks finished per token tile (fused launch)
//   partials0/1   split-K partial sums of each phase
// Everything before partials0 must be zero when the pass starts.
constexpr size_t kCounterBytes = 256;

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

size_t partial_bytes(int mode, const GemmPlan& plan) {
  if (plan.split <= 1) return 0;
  return static_cast<size_t>(plan.max_tiles) * plan.split * accum_cols(mode, plan.bn) * kBM * sizeof(float);
}

struct ScratchLayout {
  size_t tickets0, tickets1, done, partials0, partials1, total;
};

ScratchLayout scratch_layout(const GemmPlan& g, const GemmPlan& d) {
  ScratchLayout l{};
  const int max_tt = g.max_token_tiles > d.max_token_tiles ? g.max_token_tiles : d.max_token_tiles;
  l.tickets0 = kCounterBytes;
  l.tickets1 = l.tickets0 + align256(static_cast<size_t>(g.max_tiles) * sizeof(int));
  l.done = l.tickets1 + align256(static_cast<size_t>(d.max_tiles) * sizeof(int));
  l.partials0 = l.done + align256(static_cast<size_t>(max_tt) * sizeof(int));
  l.partials1 = l.partials0 + align256(partial_bytes(0, g));
  l.total = l.partials1 + align256(partial_bytes(1, d));
  return l;
}

bool fill_phase(PhaseParams& ph, int mode, const GemmPlan& plan, const uint16_t* weights, const uint16_t* act_in,
                int rows, int E, int H, int F, uint16_t* out, char* base, const ScratchLayout& l) {
  const int kdim = mode == 0 ? H : F;  // reduction length
  // [E][2F][H] gate/up weights are read as [2E][F][H] (gate rows, then up
  // rows, of each expert), so a last 128-row block that runs past F reads the
  // zero fill, not the next rows
  const int planes = mode == 0 ? 2 : 1;
  const int prows = mode == 0 ? F : H;  // rows per plane
  {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kdim), static_cast<cuuint64_t>(prows),
                                static_cast<cuuint64_t>(E) * planes};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kdim) * 2,
                                   static_cast<cuuint64_t>(kdim) * 2 * static_cast<cuuint64_t>(prows)};
    const cuuint32_t box[3] = {kBK, kBM, 1};
    if (!encode_map(&ph.tmap_w, weights, 3, dims, strides, box)) return false;
  }
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kdim), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kdim) * 2};
    const cuuint32_t box[2] = {kBK, static_cast<cuuint32_t>(plan.bn)};
    if (!encode_map(&ph.tmap_x, act_in, 2, dims, strides, box)) return false;
  }
  ph.out = out;
  ph.tickets = reinterpret_cast<int*>(base + (mode == 0 ? l.tickets0 : l.tickets1));
  ph.partials = plan.split > 1 ? reinterpret_cast<float*>(base + (mode == 0 ? l.partials0 : l.partials1)) : nullptr;
  ph.n_mb = (prows + kBM - 1) / kBM;
  ph.ksteps = kdim / kBK;
  ph.split = plan.split;
  ph.out_ld = mode == 0 ? F : H;
  ph.planes = planes;
  ph.max_tiles = plan.max_tiles;
  return true;
}

template <int BN>
cudaError_t launch_fused_bn(const GemmParams& prm, int grid, cudaStream_t stream, bool pdl) {
  return launch_mode_bn<2, BN>(prm, grid, stream, pdl);
}

// One NVFP4 phase: codes read as bytes (two values each), 128-byte k-steps
// (256 values) with the 128-byte swizzle; activation scale slots as 16-byte
// x 32-row boxes without swizzle.
bool fill_phase_fp4(PhaseParams& ph, int mode, const GemmPlan& plan, const uint8_t* wq, const uint8_t* wsf,
                    const float* wscale, const uint8_t* xq, const uint8_t* xsf, float xscale, int rows, int E, int H,
                    int F, char* base, const ScratchLayout& l) {
  const int kdim = mode == 0 ? H : F;
  const int planes = mode == 0 ? 2 : 1;
  const int prows = mode == 0 ? F : H;
  {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kdim / 2), static_cast<cuuint64_t>(prows),
                                static_cast<cuuint64_t>(E) * planes};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kdim / 2),
                                   static_cast<cuuint64_t>(kdim / 2) * static_cast<cuuint64_t>(prows)};
    const cuuint32_t box[3] = {128, kBM, 1};
    if (!encode_map(&ph.tmap_w, wq, 3, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_UINT8)) return false;
  }
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kdim / 2), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kdim / 2)};
    const cuuint32_t box[2] = {128, static_cast<cuuint32_t>(plan.bn)};
    if (!encode_map(&ph.tmap_x, xq, 2, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_UINT8)) return false;
  }
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kdim / 4), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kdim / 4)};
    const cuuint32_t box[2] = {16, 32};
    if (!encode_map(&ph.tmap_sfx, xsf, 2, dims, strides, box, CU_TENSOR_MAP_DATA_TYPE_UINT8,
                    CU_TENSOR_MAP_SWIZZLE_NONE))
      return false;
  }
  ph.sfw = wsf;
  ph.wscale = wscale;
  ph.xscale = xscale;
  ph.tickets = reinterpret_cast<int*>(base + (mode == 0 ? l.tickets0 : l.tickets1));
  ph.partials = plan.split > 1 ? reinterpret_cast<float*>(base + (mode == 0 ? l.partials0 : l.partials1)) : nullptr;
  ph.n_mb = prows / kBM;
  ph.ksteps = kdim / 256;
  ph.split = plan.split;
  ph.out_ld = mode == 0 ? F : H;
  ph.planes = planes;
  ph.max_tiles = plan.max_tiles;
  return true;
}

}  // namespace

namespace {

// The pairs launched: as many clusters of two as can be resident at once
// (GPCs with an odd number of free SMs leave one idle), so that no pair
// waits for a second wave; queried once per device.
template <int MODE>
cudaError_t launch_pair_mode(const GemmParams& prm, int num_sms, cudaStream_t stream, bool pdl) {
  static std::once_flag once[64];
  static int pairs[64];
  int dev = 0;
  cudaGetDevice(&dev);
  cudaError_t attr_err = cudaSuccess;
  std::call_once(once[dev & 63], [&] {
    attr_err = cudaFuncSetAttribute(moe_gemm_pair_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kPairSmem);
    int clusters = 0;
    if (attr_err == cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((num_sms / 2) * 2);
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = kPairSmem;
      if (cudaOccupancyMaxActiveClusters(&clusters, moe_gemm_pair_kernel<MODE>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        clusters = 0;
      }
    }
    pairs[dev & 63] = clusters > 0 ? std::min(clusters, num_sms / 2) : num_sms / 2;
  });
  if (attr_err != cudaSuccess) return attr_err;
  const cudaError_t err = launch_kernel(moe_gemm_pair_kernel<MODE>, dim3(2 * pairs[dev & 63]), dim3(kThreads),
                                        kPairSmem, stream, pdl, prm);
  ++launch_counter();
  return err;
}

}  // namespace

cudaError_t launch_gemm_pair(int mode, const uint16_t* weights, const uint16_t* act_in, const int32_t* offsets,
                             int rows, int E, int H, int F, uint16_t* out, int* counter, int num_sms,
                             cudaStream_t stream, bool pdl) {
  GemmParams prm;
  memset(&prm, 0, sizeof(prm));
  PhaseParams& ph = prm.ph[0];
  const int kdim = mode == 0 ? H : F;
  const int planes = mode == 0 ? 2 : 1;
  const int prows = mode == 0 ? F : H;
  {
    // gate/up: a box of 64 rows in both planes (a CTA's 64 gate rows and the
    // matching 64 up rows, one TMA instruction: the producer's issue rate is
    // part of what feeds the MMAs); down: 128 rows
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kdim), static_cast<cuuint64_t>(prows),
                                static_cast<cuuint64_t>(E) * planes};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kdim) * 2,
                                   static_cast<cuuint64_t>(kdim) * 2 * static_cast<cuuint64_t>(prows)};
    const cuuint32_t box[3] = {kBK, static_cast<cuuint32_t>(mode == 0 ? 64 : kBM),
                               static_cast<cuuint32_t>(mode == 0 ? 2 : 1)};
    if (!encode_map(&ph.tmap_w, weights, 3, dims, strides, box)) return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kdim), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kdim) * 2};
    const cuuint32_t box[2] = {kBK, static_cast<cuuint32_t>(kPairRows)};
    if (!encode_map(&ph.tmap_x, act_in, 2, dims, strides, box)) return cudaErrorInvalidValue;
  }
  ph.out = out;
  ph.n_mb = mode == 0 ? F / kBM : H / (2 * kBM);
  ph.ksteps = kdim / kBK;
  ph.split = 1;
  ph.out_ld = mode == 0 ? F : H;
  ph.planes = planes;
  prm.offsets = offsets;
  prm.counter = counter;
  prm.E = E;
  prm.rows = rows;
  return mode == 0 ? launch_pair_mode<0>(prm, num_sms, stream, pdl) : launch_pair_mode<1>(prm, num_sms, stream, pdl);
}

size_t gemm_scratch_bytes(const GemmPlan& gate_up, const GemmPlan& down) {
  return scratch_layout(gate_up, down).total;
}

size_t gemm_clear_bytes(const GemmPlan& gate_up, const GemmPlan& down) {
  return scratch_layout(gate_up, down).partials0;
}

cudaError_t clear_gemm_scratch(void* scratch, const GemmPlan& gate_up, const GemmPlan& down, cudaStream_t stream) {
  return cudaMemsetAsync(scratch, 0, gemm_clear_bytes(gate_up, down), stream);
}

cudaError_t launch_gemm(int mode, const GemmPlan& gate_up, const GemmPlan& down, const uint16_t* weights,
                        const uint16_t* act_in, const int32_t* offsets, int rows, int E, int H, int F, uint16_t* out,
                        void* scratch, int num_sms, cudaStream_t stream, bool pdl) {
  const GemmPlan& plan = mode == 0 ? gate_up : down;
  if (plan.pair)
    return launch_gemm_pair(mode, weights, act_in, offsets, rows, E, H, F, out, static_cast<int*>(scratch) + mode,
                            num_sms, stream, pdl);
  GemmParams prm;
  memset(&prm, 0, sizeof(prm));
  char* base = static_cast<char*>(scratch);
  const ScratchLayout l = scratch_layout(gate_up, down);
  if (!fill_phase(prm.ph[0], mode, plan, weights, act_in, rows, E, H, F, out, base, l)) return cudaErrorInvalidValue;
  prm.offsets = offsets;
  prm.counter = reinterpret_cast<int*>(base) + mode;
  prm.done = nullptr;
  prm.E = E;
  prm.rows = rows;
  prm.max_token_tiles = plan.max_token_tiles;
  return mode == 0 ? launch_mode<0>(plan.bn, prm, num_sms, stream, pdl)
                   : launch_mode<1>(plan.bn, prm, num_sms, stream, pdl);
}

void plan_experts(int T, int K, int E, int H, int F, int num_sms, GemmPlan* gate_up, GemmPlan* down, bool fp4) {
  *gate_up = plan_gemm(0, T, K, E, H, F, num_sms, 16, fp4);
  *down = plan_gemm(1, T, K, E, H, F, num_sms, 16, fp4);
  if (fused_experts_supported(*gate_up, *down)) {
    // One launch runs both phases from one unit list, so only the down units
    // at its end need to be small for balance; fewer, larger gate/up units
    // mean fewer split-K tickets, whose round trips the epilogue waits on.
    *gate_up = plan_gemm(0, T, K, E, H, F, num_sms, 4, fp4);
  }
}

bool fused_experts_supported(const GemmPlan& gate_up, const GemmPlan& down) {
  return gate_up.bn == down.bn && gate_up.bn <= 64;
}

cudaError_t launch_fused_experts(const GemmPlan& gate_up, const GemmPlan& down, const uint16_t* w_gate_up,
                                 const uint16_t* w_down, const uint16_t* x_perm, const int32_t* offsets, int rows,
                                 int E, int H, int F, uint16_t* act, uint16_t* y_perm, void* scratch, int num_sms,
                                 cudaStream_t stream, bool pdl, const int* ready) {
  GemmParams prm;
  memset(&prm, 0, sizeof(prm));
  char* base = static_cast<char*>(scratch);
  const ScratchLayout l = scratch_layout(gate_up, down);
  if (!fill_phase(prm.ph[0], 0, gate_up, w_gate_up, x_perm, rows, E, H, F, act, base, l) ||
      !fill_phase(prm.ph[1], 1, down, w_down, act, rows, E, H, F, y_perm, base, l))
    return cudaErrorInvalidValue;
  prm.offsets = offsets;
  prm.counter = reinterpret_cast<int*>(base) + 2;
  prm.done = reinterpret_cast<int*>(base + l.done);
  prm.E = E;
  prm.rows = rows;
  prm.max_token_tiles = gate_up.max_token_tiles;
  prm.ready = ready;
  switch (gate_up.bn) {
    case 16: return launch_fused_bn<16>(prm, num_sms, stream, pdl);
    case 32: return launch_fused_bn<32>(prm, num_sms, stream, pdl);
    default: return launch_fused_bn<64>(prm, num_sms, stream, pdl);
  }
}

cudaError_t launch_fused_experts_fp4(const GemmPlan& gate_up, const GemmPlan& down, const Nvfp4Experts& wt,
                                     const uint8_t* xq, const uint8_t* xsf, float x_scale, const int32_t* offsets,
                                     int rows, int E, int H, int F, uint8_t* act_q, uint8_t* act_sf, float act_scale,
                                     uint16_t* y_perm, void* scratch, int num_sms, cudaStream_t stream, bool pdl,
                                     const int* ready) {
  if (!fused_experts_supported(gate_up, down) || gate_up.bn > 32) return cudaErrorInvalidValue;
  GemmParams prm;
  memset(&prm, 0, sizeof(prm));
  char* base = static_cast<char*>(scratch);
  const ScratchLayout l = scratch_layout(gate_up, down);
  if (!fill_phase_fp4(prm.ph[0], 0, gate_up, wt.q_gate_up, wt.sf_gate_up, wt.scale, xq, xsf, x_scale, rows, E, H, F,
                      base, l) ||
      !fill_phase_fp4(prm.ph[1], 1, down, wt.q_down, wt.sf_down, wt.scale, act_q, act_sf, act_scale, rows, E, H, F,
                      base, l))
    return cudaErrorInvalidValue;
  prm.ph[0].out_q = act_q;
  prm.ph[0].out_sf = act_sf;
  prm.ph[0].out_scale = act_scale;
  prm.ph[1].out = y_perm;
  prm.offsets = offsets;
  prm.counter = reinterpret_cast<int*>(base) + 2;
  prm.done = reinterpret_cast<int*>(base + l.done);
  prm.E = E;
  prm.rows = rows;
  prm.max_token_tiles = gate_up.max_token_tiles;
  prm.ready = ready;
  return gate_up.bn == 16 ? launch_mode_bn<2, 16, true>(prm, num_sms, stream, pdl)
                          : launch_mode_bn<2, 32, true>(prm, num_sms, stream, pdl);
}

cudaError_t launch_combine(const uint16_t* y_perm, const float* w, const int32_t* inv_perm, int T, int K, int H,
                           uint16_t* y, cudaStream_t stream, bool pdl, int* err_out) {
  const int chunks = H / 8;
  const size_t n = static_cast<size_t>(T) * chunks;
  const int blocks = static_cast<int>((n + 255) / 256);
  const cudaError_t err = launch_kernel(K <= 8 ? combine_kernel<8> : combine_kernel<kMaxTopK>, dim3(blocks),
                                        dim3(256), 0, stream, pdl,
                                        reinterpret_cast<const uint4*>(y_perm), w, inv_perm, T, K, chunks,
                                        reinterpret_cast<uint4*>(y), err_out);
  ++launch_counter();
  return err;
}

namespace {

template <int BN>
cudaError_t launch_router_tc_bn(const CUtensorMap& mw, const CUtensorMap& mz, int T, int E, int H, float* logits,
                                cudaStream_t stream, bool pdl) {
  constexpr int kSmem = 1024 + kRtStages * (3 * kTileABytes + BN * kBK * 2);
  static std::once_flag once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  cudaError_t attr_err = cudaSuccess;
  std::call_once(once[dev & 63], [&] {
    attr_err = cudaFuncSetAttribute(router_tc_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  });
  if (attr_err != cudaSuccess) return attr_err;
  const dim3 grid((T + BN - 1) / BN, E / kBM);
  const cudaError_t err =
      launch_kernel(router_tc_kernel<BN>, grid, dim3(kRtThreads), kSmem, stream, pdl, mw, mz, T, E, H / kBK, logits);
  ++launch_counter();
  return err;
}

}  // namespace

bool router_tc_supported(int T, int E, int H) { return T > 128 && E % kBM == 0 && E <= 256 && H % kBK == 0; }

size_t router_tc_scratch_bytes(int E, int H) { return 3 * static_cast<size_t>(E) * H * sizeof(uint16_t); }

cudaError_t launch_router_tc(const uint16_t* z, const float* W, int T, int E, int H, float* logits, uint16_t* w3,
                             int num_sms, cudaStream_t stream, bool pdl) {
  const size_t n = static_cast<size_t>(E) * H;
  cudaError_t err = launch_kernel(split_router_weights_kernel, dim3(num_sms * 4), dim3(256), 0, stream, pdl, W, w3, n);
  ++launch_counter();
  if (err != cudaSuccess) return err;
  // the weight terms as a 3-D tensor (k, expert, term), the tokens as 2-D (k, token)
  CUtensorMap mw, mz;
  const cuuint64_t dw[3] = {static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(E), 3};
  const cuuint64_t sw[2] = {static_cast<cuuint64_t>(H) * 2, static_cast<cuuint64_t>(E) * H * 2};
  const cuuint32_t bw[3] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(kBM), 3};
  if (!encode_map(&mw, w3, 3, dw, sw, bw)) return cudaErrorInvalidValue;
  // token tile: the widest of 128/64/32 that still gives at least one CTA per SM
  int bn = 128;
  while (bn > 32 && ((T + bn - 1) / bn) * (E / kBM) < num_sms) bn >>= 1;
  const cuuint64_t dz[2] = {static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(T)};
  const cuuint64_t sz[1] = {static_cast<cuuint64_t>(H) * 2};
  const cuuint32_t bz[2] = {static_cast<cuuint32_t>(kBK), static_cast<cuuint32_t>(bn)};
  if (!encode_map(&mz, z, 2, dz, sz, bz)) return cudaErrorInvalidValue;
  switch (bn) {
    case 128: return launch_router_tc_bn<128>(mw, mz, T, E, H, logits, stream, pdl);
    case 64: return launch_router_tc_bn<64>(mw, mz, T, E, H, logits, stream, pdl);
    default: return launch_router_tc_bn<32>(mw, mz, T, E, H, logits, stream, pdl);
  }
}

cudaError_t launch_bounded_wait_probe(int* flag, uint64_t limit_ns, int site, cudaStream_t stream) {
  cudaError_t err = cudaMemsetAsync(flag, 0, sizeof(int), stream);
  if (err != cudaSuccess) return err;
  bounded_wait_probe_kernel<<<1, 1, 0, stream>>>(flag, limit_ns, site);
  ++launch_counter();
  return cudaGetLastError();
}

cudaError_t read_and_clear_device_error(int* code, cudaStream_t stream) {
  cudaError_t err = cudaStreamSynchronize(stream);
  if (err != cudaSuccess) return err;
  int v = 0;
  err = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int));
  if (err != cudaSuccess) return err;
  if (v != 0) {
    const int zero = 0;
    err = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
  }
  *code = v;
  return err;
}

}  // namespace beam
