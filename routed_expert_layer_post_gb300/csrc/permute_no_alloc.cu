// beam_moe_permute_no_alloc: the expert permutation for callers that cannot
// provide a workspace.
//
// Some callers of this library have no way to hand it scratch memory: for
// example an operator plugin inside an inference runtime that only receives
// the tensors the operator declares, or a latency-critical loop where a
// device allocation (which can synchronise the whole device) is not allowed.
// This entry point runs the same permutation kernels as beam_moe_permute but
// takes its scratch (per-chunk histograms, per-chunk bases and the ticket
// counter) from a fixed array in the library's own device memory, so it needs
// no workspace argument and allocates nothing.
//
// Limits and sharing:
// - the array holds the scratch of at most kMaxPairs = 131072 (token, slot)
//   pairs with at most 256 experts (131,328 bytes); larger calls are rejected
//   with BEAM_ERR_WORKSPACE_TOO_SMALL;
// - every GPU that loads the library holds its own copy until the process
//   exits;
// - all calls on a device share that copy and it keeps whatever the last call
//   left in it: the ticket counter is cleared at the start of every call, and
//   two calls whose kernels overlap on the GPU (for example on two streams
//   without ordering between them) race on it and give wrong results;
// - the first call on each device looks up the array's device address with
//   cudaGetSymbolAddress (with that device current); make that first call
//   before starting any stream capture on the device. Only a successful
//   lookup is kept: after a failed one (for example a call made before the
//   device's context could be created) the next call looks it up again;
// - the address is kept for the life of the process, so resetting the
//   device (cudaDeviceReset) after the first call is not supported: the
//   array may then sit at another address.
#include "../../include/beam.h"
#include "kernels.h"

#include <mutex>

namespace {

constexpr int kMaxPairs = BEAM_NO_ALLOC_MAX_PAIRS;
constexpr int kMaxExperts = 256;
constexpr int kChunk = 2048;  // pairs per block in the permutation kernels
constexpr size_t kScratchInts = 64 + 2 * static_cast<size_t>((kMaxPairs + kChunk - 1) / kChunk) * kMaxExperts;

// The scratch itself: file scope, in device memory, one copy per GPU.
static __device__ __align__(256) int g_permute_scratch[kScratchInts];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu[kMaxDevices];

// Device address of g_permute_scratch on the current device. A successful
// lookup is kept per device; a failed one is retried on the next call.
beam_status_t scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BEAM_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return BEAM_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_scratch_mu[dev]);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // leave no sticky error from the failed lookup
      return BEAM_ERR_CUDA;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return BEAM_OK;
}

}  // namespace

extern "C" beam_status_t beam_moe_permute_no_alloc(const int32_t* topk_ids, const uint16_t* z, int T,
                                                   const beam_moe_config_t* cfg, int32_t* expert_offsets,
                                                   int32_t* perm_token, int32_t* inv_perm, uint16_t* x_perm,
                                                   void* stream) {
  // same argument rules as beam_moe_permute, minus the workspace
  if (cfg == nullptr) return BEAM_ERR_INVALID_ARG;
  const size_t need = beam_moe_permute_workspace_size(cfg, T);
  if (need == 0)  // invalid config or T: let the regular entry point name the error
    return beam_moe_permute(topk_ids, z, T, cfg, expert_offsets, perm_token, inv_perm, x_perm, nullptr, 0, stream);
  if (T == 0) return BEAM_OK;
  if (static_cast<long long>(T) * cfg->topk > kMaxPairs || cfg->num_experts > kMaxExperts ||
      need > sizeof(int) * kScratchInts)
    return BEAM_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const beam_status_t st = scratch_for_current_device(&scratch);
  if (st != BEAM_OK) return st;
  return beam_moe_permute(topk_ids, z, T, cfg, expert_offsets, perm_token, inv_perm, x_perm, scratch,
                          sizeof(int) * kScratchInts, stream);
}
