// C ABI of libbeam.so (declared in include/beam.h): argument validation on
// the host, workspace carving and stream-ordered launch orchestration. No
// entry point allocates device memory or synchronises (except the host-buffer
// layer variant and the device-error query).
#include "../../include/beam.h"
#include "kernels.h"
#include "ptx.cuh"

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

namespace beam {

int& launch_counter() {
  static thread_local int n = 0;
  return n;
}

}  // namespace beam

namespace {

using beam::launch_counter;

constexpr size_t kAlign = 256;

size_t align_up(size_t v) { return (v + kAlign - 1) & ~(kAlign - 1); }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

beam_status_t check_config(const beam_moe_config_t* c) {
  if (c == nullptr) return BEAM_ERR_INVALID_ARG;
  if (c->hidden <= 0 || c->num_experts <= 0 || c->num_groups <= 0 || c->topk_groups <= 0 || c->topk <= 0 ||
      c->d_ff <= 0)
    return BEAM_ERR_INVALID_ARG;
  if (!(c->eps >= 0.0f) || !std::isfinite(c->eps) || !std::isfinite(c->routed_scale)) return BEAM_ERR_INVALID_ARG;
  if (c->num_experts % c->num_groups != 0) return BEAM_ERR_INVALID_ARG;
  if (c->topk_groups > c->num_groups) return BEAM_ERR_INVALID_ARG;
  if (c->topk > c->topk_groups * (c->num_experts / c->num_groups)) return BEAM_ERR_INVALID_ARG;
  if (!beam::boundary_supported(c->hidden)) return BEAM_ERR_UNSUPPORTED_SHAPE;
  if (c->d_ff % 64 != 0) return BEAM_ERR_UNSUPPORTED_SHAPE;
  if (c->num_experts > 256 || c->num_groups > 32 || c->num_experts / c->num_groups > 32) return BEAM_ERR_UNSUPPORTED_SHAPE;
  if (c->topk > 16) return BEAM_ERR_UNSUPPORTED_SHAPE;
  return BEAM_OK;
}

beam_status_t check_T(int T, const beam_moe_config_t* c) {
  if (T < 0) return BEAM_ERR_INVALID_ARG;
  if (static_cast<long long>(T) * c->topk >= (1LL << 31)) return BEAM_ERR_UNSUPPORTED_SHAPE;
  return BEAM_OK;
}

struct DeviceInfo {
  int sms = 0;
  bool ok = false;
};

beam_status_t device_info(DeviceInfo* out) {
  static DeviceInfo cache[64];
  static std::once_flag once[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BEAM_ERR_CUDA;
  if (dev < 0 || dev >= 64) return BEAM_ERR_UNSUPPORTED_DEVICE;
  std::call_once(once[dev], [dev] {
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cache[dev].sms = sms;
    cache[dev].ok = (major == 10 && minor == 3 && sms > 0);
  });
  *out = cache[dev];
  return out->ok ? BEAM_OK : BEAM_ERR_UNSUPPORTED_DEVICE;
}

beam_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? BEAM_OK : BEAM_ERR_CUDA; }

// ------------------------------------------------------------------ workspace layouts
struct ExpertsWs {
  size_t act, y_perm, gemm, total;
};

// the SM count enters the split-K plan; size for the largest GB300 part
constexpr int kPlanSms = 152;

ExpertsWs experts_ws(const beam_moe_config_t* c, int T, int sms) {
  ExpertsWs w{};
  const size_t rows = static_cast<size_t>(T) * c->topk;
  // scratch for the experts stage's plans and for the separate gate/up and
  // down entry points' plans (which may split differently)
  beam::GemmPlan p0, p1;
  beam::plan_experts(T, c->topk, c->num_experts, c->hidden, c->d_ff, sms, &p0, &p1);
  const beam::GemmPlan q0 = beam::plan_gemm(0, T, c->topk, c->num_experts, c->hidden, c->d_ff, sms);
  const beam::GemmPlan q1 = beam::plan_gemm(1, T, c->topk, c->num_experts, c->hidden, c->d_ff, sms);
  const size_t scratch = std::max(beam::gemm_scratch_bytes(p0, p1), beam::gemm_scratch_bytes(q0, q1));
  w.act = 0;
  w.y_perm = align_up(w.act + rows * c->d_ff * 2);
  w.gemm = align_up(w.y_perm + rows * c->hidden * 2);
  w.total = align_up(w.gemm + scratch);
  return w;
}

// NVFP4 experts stage: the quantized input rows, the quantized SwiGLU output,
// the bf16 down output and the GEMM scratch of the NVFP4 plans.
struct ExpertsWsFp4 {
  size_t xq, xsf, act_q, act_sf, y_perm, gemm, total;
};

ExpertsWsFp4 experts_ws_fp4(const beam_moe_config_t* c, int T, int sms) {
  ExpertsWsFp4 w{};
  const size_t rows = static_cast<size_t>(T) * c->topk;
  beam::GemmPlan p0, p1;
  beam::plan_experts(T, c->topk, c->num_experts, c->hidden, c->d_ff, sms, &p0, &p1, /*fp4=*/true);
  w.xq = 0;
  w.xsf = align_up(w.xq + rows * c->hidden / 2);
  w.act_q = align_up(w.xsf + rows * c->hidden / 4);
  w.act_sf = align_up(w.act_q + rows * c->d_ff / 2);
  w.y_perm = align_up(w.act_sf + rows * c->d_ff / 4);
  w.gemm = align_up(w.y_perm + rows * c->hidden * 2);
  w.total = align_up(w.gemm + beam::gemm_scratch_bytes(p0, p1));
  return w;
}

struct LayerWs {
  size_t z, logits, ids, w, offsets, perm, inv, perm_scratch, router_ticket, router_w3, x_perm, experts, total;
};

LayerWs layer_ws(const beam_moe_config_t* c, int T, int sms, bool fp4 = false) {
  LayerWs l{};
  const size_t rows = static_cast<size_t>(T) * c->topk;
  size_t o = 0;
  l.z = o;            o = align_up(o + static_cast<size_t>(T) * c->hidden * 2);
  l.logits = o;       o = align_up(o + static_cast<size_t>(T) * c->num_experts * 4);
  l.ids = o;          o = align_up(o + rows * 4);
  l.w = o;            o = align_up(o + rows * 4);
  l.offsets = o;      o = align_up(o + (c->num_experts + 1) * 4);
  l.perm = o;         o = align_up(o + rows * 4);
  l.inv = o;          o = align_up(o + rows * 4);
  l.perm_scratch = o; o = align_up(o + beam::permute_scratch_bytes(T, c->topk, c->num_experts));
  l.router_ticket = o; o = align_up(o + beam::kRouteSyncInts * sizeof(int));
  l.router_w3 = o;
  if (beam::router_tc_supported(T, c->num_experts, c->hidden))
    o = align_up(o + beam::router_tc_scratch_bytes(c->num_experts, c->hidden));
  l.x_perm = o;       o = align_up(o + rows * c->hidden * 2);
  l.experts = o;      o = align_up(o + (fp4 ? experts_ws_fp4(c, T, sms).total : experts_ws(c, T, sms).total));
  l.total = o;
  return l;
}

int plan_sms() {
  DeviceInfo d;
  if (device_info(&d) == BEAM_OK) return d.sms;
  return kPlanSms;
}

void record(const beam_moe_debug_t* dbg, int i, cudaStream_t s) {
  if (dbg != nullptr && dbg->stage_events[i] != nullptr) cudaEventRecord(static_cast<cudaEvent_t>(dbg->stage_events[i]), s);
}

// Gate/up GEMM -> down GEMM -> combine. `pdl`: launch with programmatic
// dependent launch; `cleared`: the GEMM counters and tickets were already
// zeroed by an earlier kernel (the layer's permutation does it).
beam_status_t run_experts(const uint16_t* x_perm, const int32_t* offsets, const uint16_t* w_gu, const uint16_t* w_d,
                          const float* topk_w, const int32_t* inv, int T, const beam_moe_config_t* c, uint16_t* y,
                          char* ws, int sms, cudaStream_t s, const beam_moe_debug_t* dbg = nullptr, bool pdl = false,
                          bool cleared = false, const int* ready = nullptr, int* err_out = nullptr) {
  const ExpertsWs w = experts_ws(c, T, sms);
  const int rows = T * c->topk;
  uint16_t* act = reinterpret_cast<uint16_t*>(ws + w.act);
  uint16_t* y_perm = reinterpret_cast<uint16_t*>(ws + w.y_perm);
  void* g = ws + w.gemm;
  beam::GemmPlan p0, p1;
  beam::plan_experts(T, c->topk, c->num_experts, c->hidden, c->d_ff, sms, &p0, &p1);
  // unit counters and split-K tickets start at zero (one memset for both GEMMs)
  cudaError_t e = cudaSuccess;
  if (!cleared && (e = beam::clear_gemm_scratch(g, p0, p1, s)) != cudaSuccess) return BEAM_ERR_CUDA;
  record(dbg, 3, s);
  if (beam::fused_experts_supported(p0, p1)) {
    // both GEMMs in one launch (the per-stage events bracket it as gate/up; down reads 0)
    e = beam::launch_fused_experts(p0, p1, w_gu, w_d, x_perm, offsets, rows, c->num_experts, c->hidden, c->d_ff,
                                   act, y_perm, g, sms, s, pdl, ready);
    if (e != cudaSuccess) return BEAM_ERR_CUDA;
    record(dbg, 4, s);
  } else {
    e = beam::launch_gemm(0, p0, p1, w_gu, x_perm, offsets, rows, c->num_experts, c->hidden, c->d_ff, act, g, sms,
                          s, pdl);
    if (e != cudaSuccess) return BEAM_ERR_CUDA;
    record(dbg, 4, s);
    e = beam::launch_gemm(1, p0, p1, w_d, act, offsets, rows, c->num_experts, c->hidden, c->d_ff, y_perm, g, sms, s,
                          pdl);
    if (e != cudaSuccess) return BEAM_ERR_CUDA;
  }
  record(dbg, 5, s);
  // the combine's predecessor is always the expert launch just above, so it
  // may start early (it waits for that launch before reading anything)
  if (y != nullptr)
    e = beam::launch_combine(y_perm, topk_w, inv, T, c->topk, c->hidden, y, s, /*pdl=*/true, err_out);
  record(dbg, 6, s);
  return cuda_status(e);
}

// The NVFP4 experts stage: the bf16 input rows quantized (FP32 scale g_in),
// both GEMMs in one launch (the SwiGLU output quantized with g_act), then
// the combine. `cleared`: the GEMM counters and tickets were zeroed by an
// earlier kernel. `inter` (optional) receives the workspace addresses of the
// intermediates. `ready` (decode routing): the routing kernel already wrote
// the quantized rows to the workspace and raises these flags; the experts
// launch polls them (x_perm is not read).
beam_status_t run_experts_fp4(const uint16_t* x_perm, const int32_t* offsets, const beam::Nvfp4Experts& wt,
                              float g_in, float g_act, const float* topk_w, const int32_t* inv, int T,
                              const beam_moe_config_t* c, uint16_t* y, char* ws, int sms, cudaStream_t s,
                              const beam_moe_debug_t* dbg, bool pdl, bool cleared, int* err_out,
                              beam_moe_nvfp4_intermediates_t* inter, const int* ready = nullptr) {
  const ExpertsWsFp4 w = experts_ws_fp4(c, T, sms);
  const int rows = T * c->topk;
  uint8_t* xq = reinterpret_cast<uint8_t*>(ws + w.xq);
  uint8_t* xsf = reinterpret_cast<uint8_t*>(ws + w.xsf);
  uint8_t* aq = reinterpret_cast<uint8_t*>(ws + w.act_q);
  uint8_t* asf = reinterpret_cast<uint8_t*>(ws + w.act_sf);
  uint16_t* y_perm = reinterpret_cast<uint16_t*>(ws + w.y_perm);
  void* g = ws + w.gemm;
  if (inter != nullptr) *inter = beam_moe_nvfp4_intermediates_t{xq, xsf, aq, asf, y_perm};
  beam::GemmPlan p0, p1;
  beam::plan_experts(T, c->topk, c->num_experts, c->hidden, c->d_ff, sms, &p0, &p1, /*fp4=*/true);
  cudaError_t e = cudaSuccess;
  if (!cleared && (e = beam::clear_gemm_scratch(g, p0, p1, s)) != cudaSuccess) return BEAM_ERR_CUDA;
  if (ready == nullptr && (e = beam::launch_quantize_rows(x_perm, rows, c->hidden, g_in, xq, xsf, s, pdl)) != cudaSuccess)
    return BEAM_ERR_CUDA;
  record(dbg, 3, s);
  e = beam::launch_fused_experts_fp4(p0, p1, wt, xq, xsf, g_in, offsets, rows, c->num_experts, c->hidden, c->d_ff,
                                     aq, asf, g_act, y_perm, g, sms, s, pdl, ready);
  if (e != cudaSuccess) return BEAM_ERR_CUDA;
  record(dbg, 4, s);
  record(dbg, 5, s);
  if (y != nullptr)
    e = beam::launch_combine(y_perm, topk_w, inv, T, c->topk, c->hidden, y, s, /*pdl=*/true, err_out);
  record(dbg, 6, s);
  return cuda_status(e);
}

beam_status_t check_nvfp4_weights(const beam_moe_nvfp4_weights_t* w, const beam_moe_config_t* c) {
  if (w == nullptr) return BEAM_ERR_INVALID_ARG;
  if (!beam::nvfp4_experts_supported(c->num_experts, c->hidden, c->d_ff)) return BEAM_ERR_UNSUPPORTED_SHAPE;
  if (!w->q_gate_up || !w->sf_gate_up || !w->q_down || !w->sf_down || !w->expert_scale) return BEAM_ERR_INVALID_ARG;
  if (!(w->input_scale > 0.0f) || !(w->act_scale > 0.0f) || !std::isfinite(w->input_scale) ||
      !std::isfinite(w->act_scale))
    return BEAM_ERR_INVALID_ARG;
  if (!aligned16(w->q_gate_up) || !aligned16(w->sf_gate_up) || !aligned16(w->q_down) || !aligned16(w->sf_down) ||
      !aligned4(w->expert_scale))
    return BEAM_ERR_MISALIGNED;
  return BEAM_OK;
}

beam::Nvfp4Experts nvfp4_of(const beam_moe_nvfp4_weights_t* w) {
  return beam::Nvfp4Experts{w->q_gate_up, w->sf_gate_up, w->q_down, w->sf_down, w->expert_scale};
}

}  // namespace

extern "C" {

const char* beam_status_string(beam_status_t s) {
  switch (s) {
    case BEAM_OK: return "ok";
    case BEAM_ERR_INVALID_ARG: return "invalid argument";
    case BEAM_ERR_MISALIGNED: return "misaligned pointer";
    case BEAM_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case BEAM_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case BEAM_ERR_CUDA: return "CUDA error";
    case BEAM_ERR_DEVICE_TIMEOUT: return "bounded wait timed out on the device";
    case BEAM_ERR_UNSUPPORTED_DEVICE: return "device is not compute capability 10.3 (GB300)";
  }
  return "unknown status";
}

const char* beam_version(void) { return "beam-moe-gb300 0.1 (sm_103a)"; }

int beam_last_launch_count(void) { return launch_counter(); }

beam_status_t beam_boundary_norm(const uint16_t* h, const uint16_t* x, const uint16_t* w_post, const uint16_t* w_pre,
                                 int T, int H, float eps, int n, uint16_t* h_out, uint16_t* z_out, void* stream) {
  if (T < 0 || n < 1 || !(eps >= 0.0f) || !std::isfinite(eps)) return BEAM_ERR_INVALID_ARG;
  if (!beam::boundary_supported(H)) return BEAM_ERR_UNSUPPORTED_SHAPE;
  launch_counter() = 0;
  if (T == 0) return BEAM_OK;
  if (!h || !x || !w_post || !w_pre || !h_out || !z_out) return BEAM_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(x) || !aligned16(w_post) || !aligned16(w_pre) || !aligned16(h_out) ||
      !aligned16(z_out))
    return BEAM_ERR_MISALIGNED;
  if (z_out == h_out || z_out == h || z_out == x || h_out == x) return BEAM_ERR_INVALID_ARG;
  DeviceInfo d;
  beam_status_t st = device_info(&d);
  if (st != BEAM_OK) return st;
  return cuda_status(
      beam::launch_boundary(h, x, w_post, w_pre, T, H, eps, n, h_out, z_out, static_cast<cudaStream_t>(stream)));
}

beam_status_t beam_router_topk(const uint16_t* z, const float* router_w, const float* bias, int T,
                               const beam_moe_config_t* cfg, float* logits_out, int32_t* topk_ids, float* topk_w,
                               void* stream) {
  beam_status_t st = check_config(cfg);
  if (st != BEAM_OK) return st;
  if ((st = check_T(T, cfg)) != BEAM_OK) return st;
  launch_counter() = 0;
  if (T == 0) return BEAM_OK;
  if (!z || !router_w || !bias || !logits_out || !topk_ids || !topk_w) return BEAM_ERR_INVALID_ARG;
  if (!aligned16(z) || !aligned16(router_w) || !aligned4(bias) || !aligned4(logits_out) || !aligned4(topk_ids) ||
      !aligned4(topk_w))
    return BEAM_ERR_MISALIGNED;
  DeviceInfo d;
  if ((st = device_info(&d)) != BEAM_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = beam::launch_router_logits(z, router_w, T, cfg->hidden, cfg->num_experts, logits_out, s);
  if (e != cudaSuccess) return BEAM_ERR_CUDA;
  return cuda_status(beam::launch_topk(logits_out, bias, T, cfg->num_experts, cfg->num_groups, cfg->topk_groups,
                                       cfg->topk, cfg->routed_scale, topk_ids, topk_w, s));
}

size_t beam_moe_permute_workspace_size(const beam_moe_config_t* cfg, int T) {
  if (check_config(cfg) != BEAM_OK || T < 0) return 0;
  return align_up(beam::permute_scratch_bytes(T, cfg->topk, cfg->num_experts));
}

beam_status_t beam_moe_permute(const int32_t* topk_ids, const uint16_t* z, int T, const beam_moe_config_t* cfg,
                               int32_t* expert_offsets, int32_t* perm_token, int32_t* inv_perm, uint16_t* x_perm,
                               void* ws, size_t ws_bytes, void* stream) {
  beam_status_t st = check_config(cfg);
  if (st != BEAM_OK) return st;
  if ((st = check_T(T, cfg)) != BEAM_OK) return st;
  launch_counter() = 0;
  if (T == 0) return BEAM_OK;
  if (!topk_ids || !expert_offsets || !perm_token || !inv_perm || !ws) return BEAM_ERR_INVALID_ARG;
  if (x_perm != nullptr && z == nullptr) return BEAM_ERR_INVALID_ARG;
  if (!aligned4(topk_ids) || !aligned4(expert_offsets) || !aligned4(perm_token) || !aligned4(inv_perm) ||
      (x_perm && (!aligned16(x_perm) || !aligned16(z))) || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)))
    return BEAM_ERR_MISALIGNED;
  if (ws_bytes < beam_moe_permute_workspace_size(cfg, T)) return BEAM_ERR_WORKSPACE_TOO_SMALL;
  DeviceInfo d;
  if ((st = device_info(&d)) != BEAM_OK) return st;
  return cuda_status(beam::launch_permute(topk_ids, z, T, cfg->topk, cfg->num_experts, cfg->hidden, expert_offsets,
                                          perm_token, inv_perm, x_perm, ws, static_cast<cudaStream_t>(stream)));
}

size_t beam_moe_experts_workspace_size(const beam_moe_config_t* cfg, int T) {
  if (check_config(cfg) != BEAM_OK || T < 0) return 0;
  return experts_ws(cfg, T, plan_sms()).total;
}

static beam_status_t check_experts_common(int T, const beam_moe_config_t* cfg, void* ws, size_t ws_bytes) {
  beam_status_t st = check_config(cfg);
  if (st != BEAM_OK) return st;
  if ((st = check_T(T, cfg)) != BEAM_OK) return st;
  if (T == 0) return BEAM_OK;
  if (!ws) return BEAM_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) return BEAM_ERR_MISALIGNED;
  if (ws_bytes < beam_moe_experts_workspace_size(cfg, T)) return BEAM_ERR_WORKSPACE_TOO_SMALL;
  return BEAM_OK;
}

beam_status_t beam_moe_experts(const uint16_t* x_perm, const int32_t* expert_offsets, const uint16_t* w_gate_up,
                               const uint16_t* w_down, const float* topk_w, const int32_t* inv_perm, int T,
                               const beam_moe_config_t* cfg, uint16_t* y_out, void* ws, size_t ws_bytes,
                               void* stream) {
  launch_counter() = 0;
  beam_status_t st = check_experts_common(T, cfg, ws, ws_bytes);
  if (st != BEAM_OK || T == 0) return st;
  if (!x_perm || !expert_offsets || !w_gate_up || !w_down || !topk_w || !inv_perm || !y_out)
    return BEAM_ERR_INVALID_ARG;
  if (!aligned16(x_perm) || !aligned16(w_gate_up) || !aligned16(w_down) || !aligned16(y_out) ||
      !aligned4(expert_offsets) || !aligned4(topk_w) || !aligned4(inv_perm))
    return BEAM_ERR_MISALIGNED;
  DeviceInfo d;
  if ((st = device_info(&d)) != BEAM_OK) return st;
  return run_experts(x_perm, expert_offsets, w_gate_up, w_down, topk_w, inv_perm, T, cfg, y_out,
                     static_cast<char*>(ws), d.sms, static_cast<cudaStream_t>(stream));
}

beam_status_t beam_moe_gate_up(const uint16_t* x_perm, const int32_t* expert_offsets, const uint16_t* w_gate_up,
                               int T, const beam_moe_config_t* cfg, uint16_t* act, void* ws, size_t ws_bytes,
                               void* stream) {
  launch_counter() = 0;
  beam_status_t st = check_experts_common(T, cfg, ws, ws_bytes);
  if (st != BEAM_OK || T == 0) return st;
  if (!x_perm || !expert_offsets || !w_gate_up || !act) return BEAM_ERR_INVALID_ARG;
  if (!aligned16(x_perm) || !aligned16(w_gate_up) || !aligned16(act) || !aligned4(expert_offsets))
    return BEAM_ERR_MISALIGNED;
  DeviceInfo d;
  if ((st = device_info(&d)) != BEAM_OK) return st;
  const ExpertsWs w = experts_ws(cfg, T, d.sms);
  const beam::GemmPlan p0 = beam::plan_gemm(0, T, cfg->topk, cfg->num_experts, cfg->hidden, cfg->d_ff, d.sms);
  const beam::GemmPlan p1 = beam::plan_gemm(1, T, cfg->topk, cfg->num_experts, cfg->hidden, cfg->d_ff, d.sms);
  if (beam::clear_gemm_scratch(static_cast<char*>(ws) + w.gemm, p0, p1, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return BEAM_ERR_CUDA;
  return cuda_status(beam::launch_gemm(0, p0, p1, w_gate_up, x_perm, expert_offsets, T * cfg->topk, cfg->num_experts,
                                       cfg->hidden, cfg->d_ff, act, static_cast<char*>(ws) + w.gemm, d.sms,
                                       static_cast<cudaStream_t>(stream)));
}

beam_status_t beam_moe_down(const uint16_t* act, const int32_t* expert_offsets, const uint16_t* w_down, int T,
                            const beam_moe_config_t* cfg, uint16_t* y_perm, void* ws, size_t ws_bytes, void* stream) {
  launch_counter() = 0;
  beam_status_t st = check_experts_common(T, cfg, ws, ws_bytes);
  if (st != BEAM_OK || T == 0) return st;
  if (!act || !expert_offsets || !w_down || !y_perm) return BEAM_ERR_INVALID_ARG;
  if (!aligned16(act) || !aligned16(w_down) || !aligned16(y_perm) || !aligned4(expert_offsets))
    return BEAM_ERR_MISALIGNED;
  DeviceInfo d;
  if ((st = device_info(&d)) != BEAM_OK) return st;
  const ExpertsWs w = experts_ws(cfg, T, d.sms);
  const beam::GemmPlan p0 = beam::plan_gemm(0, T, cfg->topk, cfg->num_experts, cfg->hidden, cfg->d_ff, d.sms);
  const beam::GemmPlan p1 = beam::plan_gemm(1, T, cfg->topk, cfg->num_experts, cfg->hidden, cfg->d_ff, d.sms);
  if (beam::clear_gemm_scratch(static_cast<char*>(ws) + w.gemm, p0, p1, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return BEAM_ERR_CUDA;
  return cuda_status(beam::launch_gemm(1, p0, p1, w_down, act, expert_offsets, T * cfg->topk, cfg->num_experts,
                                       cfg->hidden, cfg->d_ff, y_perm, static_cast<char*>(ws) + w.gemm, d.sms,
                                       static_cast<cudaStream_t>(stream)));
}

beam_status_t beam_moe_combine(const uint16_t* y_perm, const float* topk_w, const int32_t* inv_perm, int T,
                               const beam_moe_config_t* cfg, uint16_t* y_out, void* stream) {
  beam_status_t st = check_config(cfg);
  if (st != BEAM_OK) return st;
  if ((st = check_T(T, cfg)) != BEAM_OK) return st;
  launch_counter() = 0;
  if (T == 0) return BEAM_OK;
  if (!y_perm || !topk_w || !inv_perm || !y_out) return BEAM_ERR_INVALID_ARG;
  if (!aligned16(y_perm) || !aligned16(y_out) || !aligned4(topk_w) || !aligned4(inv_perm))
    return BEAM_ERR_MISALIGNED;
  DeviceInfo d;
  if ((st = device_info(&d)) != BEAM_OK) return st;
  return cuda_status(beam::launch_combine(y_perm, topk_w, inv_perm, T, cfg->topk, cfg->hidden, y_out,
                                          static_cast<cudaStream_t>(stream)));
}

size_t beam_moe_workspace_size(const beam_moe_config_t* cfg, int T) {
  if (check_config(cfg) != BEAM_OK || T < 0) return 0;
  return layer_ws(cfg, T, plan_sms()).total;
}

// beam_moe_layer; `route_sync_zeroed`: an earlier kernel on the stream zeroed
// the decode routing kernel's flags (no memset before it). With `uncombined`
// (and y_out null) the combine is left out and *uncombined receives the
// workspace addresses of its inputs. `err_out` (optional, device-visible):
// the combine copies the device error word there.
static beam_status_t layer_impl(const uint16_t* h, const uint16_t* x, int n, const beam_moe_weights_t* wt, int T,
                                const beam_moe_config_t* cfg, uint16_t* h_out, uint16_t* y_out,
                                const beam_moe_debug_t* dbg, void* ws, size_t ws_bytes, void* stream,
                                bool route_sync_zeroed, beam_moe_uncombined_t* uncombined = nullptr,
                                int* err_out = nullptr, const beam_moe_nvfp4_weights_t* fp4w = nullptr) {
  beam_status_t st = check_config(cfg);
  if (st != BEAM_OK) return st;
  if ((st = check_T(T, cfg)) != BEAM_OK) return st;
  if (n < 1 || wt == nullptr) return BEAM_ERR_INVALID_ARG;
  const bool fp4 = fp4w != nullptr;  // NVFP4 experts (the bf16 expert weights are then unused)
  if (fp4 && (st = check_nvfp4_weights(fp4w, cfg)) != BEAM_OK) return st;
  launch_counter() = 0;
  if (T == 0) return BEAM_OK;
  if (!h || !x || !h_out || (y_out == nullptr) == (uncombined == nullptr) || !ws || !wt->w_post || !wt->w_pre ||
      !wt->router_w || !wt->bias || (!fp4 && (!wt->w_gate_up || !wt->w_down)) || (fp4 && uncombined))
    return BEAM_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(x) || !aligned16(h_out) || !aligned16(y_out) || !aligned16(wt->w_post) ||
      !aligned16(wt->w_pre) || !aligned16(wt->router_w) || !aligned4(wt->bias) || !aligned16(wt->w_gate_up) ||
      !aligned16(wt->w_down) || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)))
    return BEAM_ERR_MISALIGNED;
  if (h_out == x || y_out == h || y_out == x || y_out == h_out) return BEAM_ERR_INVALID_ARG;
  if (dbg && ((dbg->z && !aligned16(dbg->z)) || (dbg->logits && !aligned4(dbg->logits)) ||
              (dbg->topk_ids && !aligned4(dbg->topk_ids)) || (dbg->topk_w && !aligned4(dbg->topk_w)) ||
              (dbg->expert_offsets && !aligned4(dbg->expert_offsets))))
    return BEAM_ERR_MISALIGNED;
  DeviceInfo d;
  if ((st = device_info(&d)) != BEAM_OK) return st;
  const LayerWs L = layer_ws(cfg, T, d.sms, fp4);
  if (ws_bytes < L.total) return BEAM_ERR_WORKSPACE_TOO_SMALL;
  char* base = static_cast<char*>(ws);
  uint16_t* z = (dbg && dbg->z) ? dbg->z : reinterpret_cast<uint16_t*>(base + L.z);
  float* logits = (dbg && dbg->logits) ? dbg->logits : reinterpret_cast<float*>(base + L.logits);
  int32_t* ids = (dbg && dbg->topk_ids) ? dbg->topk_ids : reinterpret_cast<int32_t*>(base + L.ids);
  float* w = (dbg && dbg->topk_w) ? dbg->topk_w : reinterpret_cast<float*>(base + L.w);
  int32_t* offsets = (dbg && dbg->expert_offsets) ? dbg->expert_offsets : reinterpret_cast<int32_t*>(base + L.offsets);
  int32_t* perm = reinterpret_cast<int32_t*>(base + L.perm);
  int32_t* inv = reinterpret_cast<int32_t*>(base + L.inv);
  uint16_t* x_perm = reinterpret_cast<uint16_t*>(base + L.x_perm);
  if (uncombined != nullptr) {
    uncombined->y_perm = reinterpret_cast<const uint16_t*>(base + L.experts + experts_ws(cfg, T, d.sms).y_perm);
    uncombined->topk_w = w;
    uncombined->inv_perm = inv;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int H = cfg->hidden;
  int launches = 0;
  record(dbg, 0, s);
  // every kernel of the layer is launched with programmatic dependent launch
  const bool pdl = true;
  int* router_ticket = reinterpret_cast<int*>(base + L.router_ticket);
  beam::GemmPlan p0, p1;
  beam::plan_experts(T, cfg->topk, cfg->num_experts, cfg->hidden, cfg->d_ff, d.sms, &p0, &p1, fp4);
  char* gemm_scratch =
      base + L.experts + (fp4 ? experts_ws_fp4(cfg, T, d.sms).gemm : experts_ws(cfg, T, d.sms).gemm);
  cudaError_t e;
  if (beam::route_decode_supported(T, H, cfg->num_experts, cfg->num_groups, cfg->topk)) {
    // decode sizes: boundary, router, top-k, permutation and the GEMM scratch
    // clear in one launch (the stage events of router and permutation are
    // empty); the fused experts launch starts on the routing kernel's flags
    // NVFP4 experts: the routing kernel writes the permuted rows quantized
    const ExpertsWsFp4 wq = fp4 ? experts_ws_fp4(cfg, T, d.sms) : ExpertsWsFp4{};
    const bool fp4_rows = fp4 && beam::fused_experts_supported(p0, p1);
    uint8_t* xq = fp4_rows ? reinterpret_cast<uint8_t*>(base + L.experts + wq.xq) : nullptr;
    uint8_t* xsf = fp4_rows ? reinterpret_cast<uint8_t*>(base + L.experts + wq.xsf) : nullptr;
    e = beam::launch_route_decode(h, x, wt->w_post, wt->w_pre, wt->router_w, wt->bias, T, H, cfg->num_experts,
                                  cfg->num_groups, cfg->topk_groups, cfg->topk, cfg->routed_scale, cfg->eps, n,
                                  h_out, z, logits, ids, w, offsets, perm, inv, x_perm, router_ticket, gemm_scratch,
                                  beam::gemm_clear_bytes(p0, p1), d.sms, s, pdl, route_sync_zeroed, xq, xsf,
                                  fp4 ? fp4w->input_scale : 0.f);
    if (e != cudaSuccess) return BEAM_ERR_CUDA;
    record(dbg, 1, s);
    record(dbg, 2, s);
    launches += launch_counter();
    launch_counter() = 0;
    if (fp4) {
      st = run_experts_fp4(x_perm, offsets, nvfp4_of(fp4w), fp4w->input_scale, fp4w->act_scale, w, inv, T, cfg,
                           y_out, base + L.experts, d.sms, s, dbg, pdl, /*cleared=*/true, err_out, nullptr,
                           fp4_rows ? router_ticket + 1 : nullptr);
    } else {
      const int* ready = beam::fused_experts_supported(p0, p1) ? router_ticket + 1 : nullptr;
      st = run_experts(x_perm, offsets, wt->w_gate_up, wt->w_down, w, inv, T, cfg, y_out, base + L.experts, d.sms,
                       s, dbg, pdl, /*cleared=*/true, ready, err_out);
    }
    launch_counter() += launches;
    return st;
  }
  // the boundary also zeroes the router's ticket (used when router and top-k share a launch)
  e = beam::launch_boundary(h, x, wt->w_post, wt->w_pre, T, H, cfg->eps, n, h_out, z, s, pdl, router_ticket);
  if (e != cudaSuccess) return BEAM_ERR_CUDA;
  record(dbg, 1, s);
  launches += launch_counter();
  launch_counter() = 0;
  if (beam::router_topk_fusable(T, cfg->num_experts, cfg->num_groups)) {
    e = beam::launch_router_topk_fused(z, wt->router_w, wt->bias, T, H, cfg->num_experts, cfg->num_groups,
                                       cfg->topk_groups, cfg->topk, cfg->routed_scale, logits, ids, w,
                                       router_ticket, s, pdl);
    if (e != cudaSuccess) return BEAM_ERR_CUDA;
  } else {
    if (beam::router_tc_supported(T, cfg->num_experts, H))
      e = beam::launch_router_tc(z, wt->router_w, T, cfg->num_experts, H, logits,
                                 reinterpret_cast<uint16_t*>(base + L.router_w3), d.sms, s, pdl);
    else
      e = beam::launch_router_logits(z, wt->router_w, T, H, cfg->num_experts, logits, s, pdl);
    if (e != cudaSuccess) return BEAM_ERR_CUDA;
    e = beam::launch_topk(logits, wt->bias, T, cfg->num_experts, cfg->num_groups, cfg->topk_groups, cfg->topk,
                          cfg->routed_scale, ids, w, s, pdl);
    if (e != cudaSuccess) return BEAM_ERR_CUDA;
  }
  record(dbg, 2, s);
  // the permutation also zeroes the experts' counters and tickets
  e = beam::launch_permute(ids, z, T, cfg->topk, cfg->num_experts, H, offsets, perm, inv, x_perm,
                           base + L.perm_scratch, s, pdl, gemm_scratch, beam::gemm_clear_bytes(p0, p1));
  if (e != cudaSuccess) return BEAM_ERR_CUDA;
  launches += launch_counter();
  launch_counter() = 0;
  if (fp4)
    st = run_experts_fp4(x_perm, offsets, nvfp4_of(fp4w), fp4w->input_scale, fp4w->act_scale, w, inv, T, cfg, y_out,
                         base + L.experts, d.sms, s, dbg, pdl, /*cleared=*/true, err_out, nullptr);
  else
    st = run_experts(x_perm, offsets, wt->w_gate_up, wt->w_down, w, inv, T, cfg, y_out, base + L.experts, d.sms, s,
                     dbg, pdl, /*cleared=*/true, nullptr, err_out);
  launch_counter() += launches;
  return st;
}

beam_status_t beam_moe_layer(const uint16_t* h, const uint16_t* x, int n, const beam_moe_weights_t* wt, int T,
                             const beam_moe_config_t* cfg, uint16_t* h_out, uint16_t* y_out,
                             const beam_moe_debug_t* dbg, void* ws, size_t ws_bytes, void* stream) {
  return layer_impl(h, x, n, wt, T, cfg, h_out, y_out, dbg, ws, ws_bytes, stream, false);
}

beam_status_t beam_moe_layer_uncombined(const uint16_t* h, const uint16_t* x, int n, const beam_moe_weights_t* wt,
                                        int T, const beam_moe_config_t* cfg, uint16_t* h_out,
                                        beam_moe_uncombined_t* out, void* ws, size_t ws_bytes, void* stream) {
  if (out == nullptr) return BEAM_ERR_INVALID_ARG;
  *out = beam_moe_uncombined_t{};
  return layer_impl(h, x, n, wt, T, cfg, h_out, nullptr, nullptr, ws, ws_bytes, stream, false, out);
}

beam_status_t beam_boundary_norm_combine(const uint16_t* h, const uint16_t* y_perm, const float* topk_w,
                                         const int32_t* inv_perm, int K, const uint16_t* w_post,
                                         const uint16_t* w_pre, int T, int H, float eps, int n, uint16_t* h_out,
                                         uint16_t* z_out, void* stream) {
  if (T < 0 || n < 1 || K < 1 || !(eps >= 0.0f) || !std::isfinite(eps)) return BEAM_ERR_INVALID_ARG;
  if (K > 16 || !beam::boundary_supported(H)) return BEAM_ERR_UNSUPPORTED_SHAPE;
  if (static_cast<long long>(T) * K >= (1LL << 31)) return BEAM_ERR_UNSUPPORTED_SHAPE;
  launch_counter() = 0;
  if (T == 0) return BEAM_OK;
  if (!h || !y_perm || !topk_w || !inv_perm || !w_post || !w_pre || !h_out || !z_out) return BEAM_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(y_perm) || !aligned16(w_post) || !aligned16(w_pre) || !aligned16(h_out) ||
      !aligned16(z_out) || !aligned4(topk_w) || !aligned4(inv_perm))
    return BEAM_ERR_MISALIGNED;
  if (z_out == h_out || z_out == h || z_out == y_perm || h_out == y_perm) return BEAM_ERR_INVALID_ARG;
  DeviceInfo d;
  beam_status_t st = device_info(&d);
  if (st != BEAM_OK) return st;
  return cuda_status(beam::launch_boundary_combine(h, y_perm, topk_w, inv_perm, K, w_post, w_pre, T, H, eps, n,
                                                   h_out, z_out, static_cast<cudaStream_t>(stream), true));
}

// ------------------------------------------------------------------ NVFP4 experts
size_t beam_nvfp4_expert_bytes(const beam_moe_config_t* cfg, size_t* q_gate_up, size_t* sf_gate_up, size_t* q_down,
                               size_t* sf_down) {
  if (check_config(cfg) != BEAM_OK || !beam::nvfp4_experts_supported(cfg->num_experts, cfg->hidden, cfg->d_ff))
    return 0;
  const size_t E = cfg->num_experts, H = cfg->hidden, F = cfg->d_ff;
  const size_t a = E * 2 * F * H / 2, b = E * 2 * F * H / 16, c = E * H * F / 2, dd = E * H * F / 16;
  if (q_gate_up) *q_gate_up = a;
  if (sf_gate_up) *sf_gate_up = b;
  if (q_down) *q_down = c;
  if (sf_down) *sf_down = dd;
  return a + b + c + dd + E * sizeof(float);
}

beam_status_t beam_nvfp4_quantize_experts(const uint16_t* w_gate_up, const uint16_t* w_down,
                                          const beam_moe_config_t* cfg, uint8_t* q_gate_up, uint8_t* sf_gate_up,
                                          uint8_t* q_down, uint8_t* sf_down, float* expert_scale, void* stream) {
  beam_status_t st = check_config(cfg);
  if (st != BEAM_OK) return st;
  if (!beam::nvfp4_experts_supported(cfg->num_experts, cfg->hidden, cfg->d_ff)) return BEAM_ERR_UNSUPPORTED_SHAPE;
  if (!w_gate_up || !w_down || !q_gate_up || !sf_gate_up || !q_down || !sf_down || !expert_scale)
    return BEAM_ERR_INVALID_ARG;
  if (!aligned16(w_gate_up) || !aligned16(w_down) || !aligned16(q_gate_up) || !aligned16(sf_gate_up) ||
      !aligned16(q_down) || !aligned16(sf_down) || !aligned4(expert_scale))
    return BEAM_ERR_MISALIGNED;
  DeviceInfo d;
  if ((st = device_info(&d)) != BEAM_OK) return st;
  launch_counter() = 0;
  return cuda_status(beam::launch_quantize_experts(w_gate_up, w_down, cfg->num_experts, cfg->hidden, cfg->d_ff,
                                                   q_gate_up, sf_gate_up, q_down, sf_down, expert_scale, d.sms,
                                                   static_cast<cudaStream_t>(stream)));
}

beam_status_t beam_nvfp4_quantize_rows(const uint16_t* x, int rows, int K, float scale, uint8_t* q, uint8_t* sf,
                                       void* stream) {
  if (rows < 0 || K <= 0 || !(scale > 0.0f) || !std::isfinite(scale)) return BEAM_ERR_INVALID_ARG;
  if (K % 64 != 0) return BEAM_ERR_UNSUPPORTED_SHAPE;
  launch_counter() = 0;
  if (rows == 0) return BEAM_OK;
  if (!x || !q || !sf) return BEAM_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(q) || !aligned16(sf)) return BEAM_ERR_MISALIGNED;
  DeviceInfo d;
  beam_status_t st = device_info(&d);
  if (st != BEAM_OK) return st;
  return cuda_status(beam::launch_quantize_rows(x, rows, K, scale, q, sf, static_cast<cudaStream_t>(stream)));
}

size_t beam_moe_experts_nvfp4_workspace_size(const beam_moe_config_t* cfg, int T) {
  if (check_config(cfg) != BEAM_OK || T < 0 ||
      !beam::nvfp4_experts_supported(cfg->num_experts, cfg->hidden, cfg->d_ff))
    return 0;
  return experts_ws_fp4(cfg, T, plan_sms()).total;
}

beam_status_t beam_moe_experts_nvfp4(const uint16_t* x_perm, const int32_t* expert_offsets,
                                     const beam_moe_nvfp4_weights_t* weights, const float* topk_w,
                                     const int32_t* inv_perm, int T, const beam_moe_config_t* cfg, uint16_t* y_out,
                                     beam_moe_nvfp4_intermediates_t* inter, void* ws, size_t ws_bytes,
                                     void* stream) {
  launch_counter() = 0;
  beam_status_t st = check_config(cfg);
  if (st != BEAM_OK) return st;
  if ((st = check_T(T, cfg)) != BEAM_OK) return st;
  if ((st = check_nvfp4_weights(weights, cfg)) != BEAM_OK) return st;
  if (inter != nullptr) *inter = beam_moe_nvfp4_intermediates_t{};
  if (T == 0) return BEAM_OK;
  if (!x_perm || !expert_offsets || !topk_w || !inv_perm || !y_out || !ws) return BEAM_ERR_INVALID_ARG;
  if (!aligned16(x_perm) || !aligned16(y_out) || !aligned4(expert_offsets) || !aligned4(topk_w) ||
      !aligned4(inv_perm) || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)))
    return BEAM_ERR_MISALIGNED;
  if (ws_bytes < beam_moe_experts_nvfp4_workspace_size(cfg, T)) return BEAM_ERR_WORKSPACE_TOO_SMALL;
  DeviceInfo d;
  if ((st = device_info(&d)) != BEAM_OK) return st;
  return run_experts_fp4(x_perm, expert_offsets, nvfp4_of(weights), weights->input_scale, weights->act_scale, topk_w,
                         inv_perm, T, cfg, y_out, static_cast<char*>(ws), d.sms, static_cast<cudaStream_t>(stream),
                         nullptr, /*pdl=*/false, /*cleared=*/false, nullptr, inter);
}

size_t beam_moe_nvfp4_workspace_size(const beam_moe_config_t* cfg, int T) {
  if (check_config(cfg) != BEAM_OK || T < 0 ||
      !beam::nvfp4_experts_supported(cfg->num_experts, cfg->hidden, cfg->d_ff))
    return 0;
  return layer_ws(cfg, T, plan_sms(), /*fp4=*/true).total;
}

beam_status_t beam_moe_layer_nvfp4(const uint16_t* h, const uint16_t* x, int n,
                                   const beam_moe_nvfp4_weights_t* weights, int T, const beam_moe_config_t* cfg,
                                   uint16_t* h_out, uint16_t* y_out, const beam_moe_debug_t* dbg, void* ws,
                                   size_t ws_bytes, void* stream) {
  if (weights == nullptr) return BEAM_ERR_INVALID_ARG;
  const beam_moe_weights_t shared = {weights->w_post, weights->w_pre, weights->router_w, weights->bias, nullptr,
                                     nullptr};
  return layer_impl(h, x, n, &shared, T, cfg, h_out, y_out, dbg, ws, ws_bytes, stream, false, nullptr, nullptr,
                    weights);
}

size_t beam_moe_layer_host_workspace_size(const beam_moe_config_t* cfg, int T) {
  const size_t base = beam_moe_workspace_size(cfg, T);
  if (base == 0 && T != 0) return 0;
  const size_t act = align_up(static_cast<size_t>(T) * cfg->hidden * 2);
  return base + 4 * act;
}

size_t beam_moe_layer_nvfp4_host_workspace_size(const beam_moe_config_t* cfg, int T) {
  const size_t base = beam_moe_nvfp4_workspace_size(cfg, T);
  if (base == 0 && T != 0) return 0;
  const size_t act = align_up(static_cast<size_t>(T) * cfg->hidden * 2);
  return base + 4 * act;
}

namespace {

// Device-visible address of a page-locked host buffer, or nullptr.
void* mapped_host(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// h and x from mapped host memory into the device workspace in one launch.
// It also zeroes the decode routing kernel's flags (`sync`, may be null), so
// that kernel needs no memset before it and starts at once: its loads of the
// router rows and norm weights overlap the reads of host memory here.
__global__ void stage_in_kernel(const uint4* __restrict__ h, const uint4* __restrict__ x, uint4* __restrict__ dh,
                                uint4* __restrict__ dx, int n16, int* __restrict__ sync, int sync_ints) {
  beam::ptx::griddep_launch_dependents();
  if (sync != nullptr && blockIdx.x == 0 && static_cast<int>(threadIdx.x) < sync_ints) sync[threadIdx.x] = 0;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += gridDim.x * blockDim.x) {
    dh[i] = h[i];
    dx[i] = x[i];
  }
}

// The device error word as seen by the host entry point. The layer's combine
// kernel copies the word into a page-locked host slot (one per device), so
// after its stream synchronise the call reads it with a plain load instead of
// a device-to-host copy. The slot is registered with the driver once per
// process; if that fails the call reads the word with a copy instead.
alignas(4096) int g_err_slots[64 * 16];  // one 64-byte slot per device
std::once_flag g_err_once;
int* g_err_slots_dev = nullptr;

int* host_error_slot_dev(int dev) {
  std::call_once(g_err_once, [] {
    void* d = nullptr;
    if (cudaHostRegister(g_err_slots, sizeof g_err_slots, cudaHostRegisterMapped | cudaHostRegisterPortable) ==
            cudaSuccess &&
        cudaHostGetDevicePointer(&d, g_err_slots, 0) == cudaSuccess)
      g_err_slots_dev = static_cast<int*>(d);
    else
      cudaGetLastError();
  });
  return g_err_slots_dev != nullptr ? g_err_slots_dev + 16 * dev : nullptr;
}

// After the call's stream synchronise: BEAM_ERR_DEVICE_TIMEOUT (and the
// device word cleared) if a bounded wait on the device gave up.
beam_status_t host_call_error(int dev, bool slot_used, cudaStream_t s) {
  if (slot_used && *reinterpret_cast<volatile int*>(&g_err_slots[16 * dev]) == 0) return BEAM_OK;
  int code = 0;
  if (beam::read_and_clear_device_error(&code, s) != cudaSuccess) return BEAM_ERR_CUDA;
  return code != 0 ? BEAM_ERR_DEVICE_TIMEOUT : BEAM_OK;
}

// One zero-copy host call: its device-visible buffers and every argument
// that enters a kernel. Zero-filled before use, so whole keys compare with
// memcmp (padding included).
struct HostCall {
  int device, n, T;
  const void* h;
  const void* x;
  void* h_out;
  void* y_out;
  beam_moe_weights_t wt;
  beam_moe_nvfp4_weights_t fp4w;  // with fp4: the NVFP4 experts (wt then holds the shared weights only)
  int fp4;
  beam_moe_config_t cfg;
  void* ws;
  size_t ws_bytes;
  int* err_out;
};

uint64_t hash_call(const HostCall& k) {  // FNV-1a over the key's bytes
  const unsigned char* b = reinterpret_cast<const unsigned char*>(&k);
  uint64_t v = 1469598103934665603ull;
  for (size_t i = 0; i < sizeof k; ++i) v = (v ^ b[i]) * 1099511628211ull;
  return v;
}

// The launches of a zero-copy call: stage-in, then the layer writing h' and y
// to the mapped output buffers. Sets the thread's launch count.
beam_status_t zero_copy_launches(const HostCall& k, cudaStream_t s) {
  const size_t bytes = static_cast<size_t>(k.T) * k.cfg.hidden * 2;
  const size_t act = align_up(bytes);
  char* base = static_cast<char*>(k.ws);
  uint16_t* d_h = reinterpret_cast<uint16_t*>(base);
  uint16_t* d_x = reinterpret_cast<uint16_t*>(base + act);
  char* lws = base + 4 * act;
  const size_t lws_bytes = k.ws_bytes - 4 * act;
  const bool route = beam::route_decode_supported(k.T, k.cfg.hidden, k.cfg.num_experts, k.cfg.num_groups,
                                                  k.cfg.topk);
  int* sync = route ? reinterpret_cast<int*>(lws + layer_ws(&k.cfg, k.T, plan_sms()).router_ticket) : nullptr;
  const int n16 = static_cast<int>(bytes / 16);
  stage_in_kernel<<<(n16 + 255) / 256, 256, 0, s>>>(static_cast<const uint4*>(k.h), static_cast<const uint4*>(k.x),
                                                  reinterpret_cast<uint4*>(d_h), reinterpret_cast<uint4*>(d_x), n16,
                                                  sync, beam::kRouteSyncInts);
  if (cudaGetLastError() != cudaSuccess) return BEAM_ERR_CUDA;
  const beam_status_t st = layer_impl(d_h, d_x, k.n, &k.wt, k.T, &k.cfg, static_cast<uint16_t*>(k.h_out),
                                      static_cast<uint16_t*>(k.y_out), nullptr, lws, lws_bytes, s, route, nullptr,
                                      k.err_out, k.fp4 ? &k.fp4w : nullptr);
  launch_counter() += 1;
  return st;
}

// Graphs of repeated zero-copy calls. A decode loop makes the same call (same
// buffers, weights and workspace) once per token, so the second call with a
// given key captures its launches into a CUDA graph and later calls replay it
// with one launch. Keys seen once run as direct launches: a loop over more
// keys than the table holds never pays for a capture it cannot reuse.
struct HostGraph {
  HostCall key;
  uint64_t hash = 0, last_use = 0;
  cudaGraphExec_t exec = nullptr;
  int launches = 0;
  bool used = false, failed = false;
};

constexpr int kHostGraphs = 256;
std::mutex g_graph_mu;
HostGraph g_graphs[kHostGraphs];
uint64_t g_graph_tick = 0;
cudaStream_t g_capture_stream[64] = {};

HostGraph* find_graph(const HostCall& k, uint64_t hash) {
  for (HostGraph& g : g_graphs)
    if (g.used && g.hash == hash && std::memcmp(&g.key, &k, sizeof k) == 0) return &g;
  return nullptr;
}

HostGraph* insert_graph(const HostCall& k, uint64_t hash) {
  HostGraph* v = &g_graphs[0];
  for (HostGraph& g : g_graphs) {
    if (!g.used) {
      v = &g;
      break;
    }
    if (g.last_use < v->last_use) v = &g;
  }
  if (v->exec != nullptr) cudaGraphExecDestroy(v->exec);  // freed once any replay in flight ends
  *v = HostGraph{};
  v->key = k;
  v->hash = hash;
  v->used = true;
  return v;
}

// Captures the call on a private stream; false (and the table entry marked
// failed) when any step of the capture fails.
bool capture_graph(HostGraph* g) {
  cudaStream_t& cs = g_capture_stream[g->key.device];
  if (cs == nullptr && cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) {
    cs = nullptr;
    cudaGetLastError();
    g->failed = true;
    return false;
  }
  cudaGraph_t graph = nullptr;
  bool ok = cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) == cudaSuccess;
  if (ok) {
    launch_counter() = 0;
    ok = zero_copy_launches(g->key, cs) == BEAM_OK;
    g->launches = launch_counter();
    ok = (cudaStreamEndCapture(cs, &graph) == cudaSuccess) && ok && graph != nullptr;
  }
  if (ok) ok = cudaGraphInstantiate(&g->exec, graph, 0) == cudaSuccess;
  if (graph != nullptr) cudaGraphDestroy(graph);
  if (!ok) {
    g->exec = nullptr;
    g->failed = true;
    cudaGetLastError();
  }
  return ok;
}

// The copy path's side streams and events, one set per device. From
// kOverlapTokens tokens up, h' (final once the boundary has run) is copied
// back on the side stream while the rest of the layer computes. From
// kPipeTokens tokens up the layer is pipelined with the copies in
// pipe_chunks(T) token chunks (layer_host_pipelined).
constexpr int kOverlapTokens = 64;
constexpr int kPipeTokens = 8192;  // measured: 16384 tokens e2e 10.70 -> 10.39 ms; 2048 tokens 3.58 -> 3.69 ms (not used there)
constexpr int kPipeMaxChunks = 8;
// chunks of at least 2048 tokens: four from 8192 tokens, eight from 16384,
// so that less of the routing waits for the last chunk's copy and less of
// the output's copy waits for the last combine
constexpr int pipe_chunks(int T) { return T >= 16384 ? 8 : 4; }

struct CopyAux {
  cudaStream_t side = nullptr, side_in = nullptr;
  cudaEvent_t after_boundary = nullptr, h_copied = nullptr;
  cudaEvent_t in_done[kPipeMaxChunks] = {}, bnd_done[kPipeMaxChunks] = {}, y_done[kPipeMaxChunks] = {};
  bool ok = false;
};

std::mutex g_aux_mu;  // held across a call's use of its device's set
CopyAux g_aux[64];

CopyAux* copy_aux(int dev) {
  CopyAux& a = g_aux[dev];
  if (!a.ok) {
    bool ok = cudaStreamCreateWithFlags(&a.side, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&a.side_in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&a.after_boundary, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&a.h_copied, cudaEventDisableTiming) == cudaSuccess;
    for (int c = 0; ok && c < kPipeMaxChunks; ++c)
      ok = cudaEventCreateWithFlags(&a.in_done[c], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&a.bnd_done[c], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&a.y_done[c], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
      cudaGetLastError();
      return nullptr;
    }
    a.ok = true;
  }
  return &a;
}

// Large batches through host buffers, pipelined with the copies: the
// tokens arrive in pipe_chunks(T) chunks on a copy-in stream, and each chunk's
// boundary, router and top-k run (on the call's stream) while the next chunk
// is still being copied; h' goes back on the side stream once the last
// chunk's boundary has run. The permutation and the expert GEMMs take the
// whole batch; the combine then runs chunk by chunk, each chunk's y copied
// back while the next chunk combines. Every kernel computes each token as in
// beam_moe_layer (the same kernels on the same per-token data; chunks hold
// more than 128 tokens, so the router is the same tensor-core kernel), so
// the outputs are bit-identical to it.
beam_status_t layer_host_pipelined(const uint16_t* h_host, const uint16_t* x_host, int n,
                                   const beam_moe_weights_t* wt, int T, const beam_moe_config_t* cfg,
                                   uint16_t* h_out_host, uint16_t* y_out_host, uint16_t* d_h, uint16_t* d_x,
                                   uint16_t* d_hn, uint16_t* d_y, char* base, int sms, cudaStream_t s, CopyAux* a,
                                   int* err_slot) {
  const int H = cfg->hidden, E = cfg->num_experts, K = cfg->topk;
  const LayerWs L = layer_ws(cfg, T, sms);
  uint16_t* z = reinterpret_cast<uint16_t*>(base + L.z);
  float* logits = reinterpret_cast<float*>(base + L.logits);
  int32_t* ids = reinterpret_cast<int32_t*>(base + L.ids);
  float* w = reinterpret_cast<float*>(base + L.w);
  int32_t* offsets = reinterpret_cast<int32_t*>(base + L.offsets);
  int32_t* perm = reinterpret_cast<int32_t*>(base + L.perm);
  int32_t* inv = reinterpret_cast<int32_t*>(base + L.inv);
  uint16_t* x_perm = reinterpret_cast<uint16_t*>(base + L.x_perm);
  int* router_ticket = reinterpret_cast<int*>(base + L.router_ticket);
  beam::GemmPlan p0, p1;
  beam::plan_experts(T, K, E, H, cfg->d_ff, sms, &p0, &p1, false);
  char* ews = base + L.experts;
  const ExpertsWs xw = experts_ws(cfg, T, sms);
  const uint16_t* y_perm = reinterpret_cast<const uint16_t*>(ews + xw.y_perm);
  const size_t row = static_cast<size_t>(H) * 2;
  const int nch = pipe_chunks(T);
  auto t0 = [&](int c) { return static_cast<int>(static_cast<long long>(T) * c / nch); };
  cudaError_t e = cudaSuccess;
  launch_counter() = 0;
  // the copy-in stream starts after everything queued on the call's stream before this call
  if ((e = cudaEventRecord(a->h_copied, s)) != cudaSuccess || (e = cudaStreamWaitEvent(a->side_in, a->h_copied, 0)) != cudaSuccess)
    return BEAM_ERR_CUDA;
  for (int c = 0; c < nch; ++c) {
    const size_t o = static_cast<size_t>(t0(c)) * H, bytes = static_cast<size_t>(t0(c + 1) - t0(c)) * row;
    if (cudaMemcpyAsync(d_h + o, h_host + o, bytes, cudaMemcpyHostToDevice, a->side_in) != cudaSuccess ||
        cudaMemcpyAsync(d_x + o, x_host + o, bytes, cudaMemcpyHostToDevice, a->side_in) != cudaSuccess ||
        cudaEventRecord(a->in_done[c], a->side_in) != cudaSuccess)
      return BEAM_ERR_CUDA;
  }
  for (int c = 0; c < nch; ++c) {
    const int tc = t0(c + 1) - t0(c);
    const size_t o = static_cast<size_t>(t0(c)) * H;
    if (cudaStreamWaitEvent(s, a->in_done[c], 0) != cudaSuccess) return BEAM_ERR_CUDA;
    e = beam::launch_boundary(d_h + o, d_x + o, wt->w_post, wt->w_pre, tc, H, cfg->eps, n, d_hn + o, z + o, s,
                              /*pdl=*/false, c == 0 ? router_ticket : nullptr);
    if (e != cudaSuccess) return BEAM_ERR_CUDA;
    if (c == nch - 1) {
      // h' goes back once the copies in are done: the link then carries it
      // alongside the expert GEMMs instead of slowing the incoming chunks
      if (cudaEventRecord(a->bnd_done[c], s) != cudaSuccess ||
          cudaStreamWaitEvent(a->side, a->bnd_done[c], 0) != cudaSuccess ||
          cudaMemcpyAsync(h_out_host, d_hn, static_cast<size_t>(T) * row, cudaMemcpyDeviceToHost, a->side) !=
              cudaSuccess)
        return BEAM_ERR_CUDA;
    }
    const size_t lo = static_cast<size_t>(t0(c)) * E, ko = static_cast<size_t>(t0(c)) * K;
    e = beam::launch_router_tc(z + o, wt->router_w, tc, E, H, logits + lo,
                               reinterpret_cast<uint16_t*>(base + L.router_w3), sms, s, true);
    if (e != cudaSuccess) return BEAM_ERR_CUDA;
    e = beam::launch_topk(logits + lo, wt->bias, tc, E, cfg->num_groups, cfg->topk_groups, K, cfg->routed_scale,
                          ids + ko, w + ko, s, true);
    if (e != cudaSuccess) return BEAM_ERR_CUDA;
  }
  // the permutation also zeroes the expert GEMMs' counters and tickets
  e = beam::launch_permute(ids, z, T, K, E, H, offsets, perm, inv, x_perm, base + L.perm_scratch, s, true,
                           ews + xw.gemm, beam::gemm_clear_bytes(p0, p1));
  if (e != cudaSuccess) return BEAM_ERR_CUDA;
  const int launches = launch_counter();
  launch_counter() = 0;
  beam_status_t st = run_experts(x_perm, offsets, wt->w_gate_up, wt->w_down, w, inv, T, cfg, nullptr, ews, sms, s,
                                 nullptr, true, /*cleared=*/true, nullptr, nullptr);
  if (st != BEAM_OK) return st;
  for (int c = 0; c < nch; ++c) {
    const int tc = t0(c + 1) - t0(c);
    const size_t o = static_cast<size_t>(t0(c)) * H, ko = static_cast<size_t>(t0(c)) * K;
    e = beam::launch_combine(y_perm, w + ko, inv + ko, tc, K, H, d_y + o, s, /*pdl=*/true,
                             c == 0 ? err_slot : nullptr);
    if (e != cudaSuccess || cudaEventRecord(a->y_done[c], s) != cudaSuccess ||
        cudaStreamWaitEvent(a->side_in, a->y_done[c], 0) != cudaSuccess ||
        cudaMemcpyAsync(y_out_host + o, d_y + o, static_cast<size_t>(tc) * row, cudaMemcpyDeviceToHost,
                        a->side_in) != cudaSuccess)
      return BEAM_ERR_CUDA;
  }
  launch_counter() += launches;
  // the call's stream ends after both side streams' copies
  if (cudaEventRecord(a->after_boundary, a->side) != cudaSuccess ||
      cudaStreamWaitEvent(s, a->after_boundary, 0) != cudaSuccess ||
      cudaEventRecord(a->h_copied, a->side_in) != cudaSuccess || cudaStreamWaitEvent(s, a->h_copied, 0) != cudaSuccess)
    return BEAM_ERR_CUDA;
  return BEAM_OK;
}

// beam_moe_layer_host and beam_moe_layer_nvfp4_host: `fp4w` set for NVFP4
// experts (then `wt` holds the shared weights only).
beam_status_t layer_host_impl(const uint16_t* h_host, const uint16_t* x_host, int n, const beam_moe_weights_t* wt,
                              const beam_moe_nvfp4_weights_t* fp4w, int T, const beam_moe_config_t* cfg,
                              uint16_t* h_out_host, uint16_t* y_out_host, void* ws, size_t ws_bytes, void* stream) {
  beam_status_t st = check_config(cfg);
  if (st != BEAM_OK) return st;
  if ((st = check_T(T, cfg)) != BEAM_OK) return st;
  if (n < 1 || wt == nullptr) return BEAM_ERR_INVALID_ARG;
  if (T == 0) return BEAM_OK;
  if (!h_host || !x_host || !h_out_host || !y_out_host || !ws) return BEAM_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) return BEAM_ERR_MISALIGNED;
  const size_t need = fp4w != nullptr ? beam_moe_layer_nvfp4_host_workspace_size(cfg, T)
                                      : beam_moe_layer_host_workspace_size(cfg, T);
  if (need == 0 || ws_bytes < need) return need == 0 ? BEAM_ERR_UNSUPPORTED_SHAPE : BEAM_ERR_WORKSPACE_TOO_SMALL;
  const size_t bytes = static_cast<size_t>(T) * cfg->hidden * 2;
  const size_t act = align_up(bytes);
  char* base = static_cast<char*>(ws);
  uint16_t* d_h = reinterpret_cast<uint16_t*>(base);
  uint16_t* d_x = reinterpret_cast<uint16_t*>(base + act);
  uint16_t* d_hn = reinterpret_cast<uint16_t*>(base + 2 * act);
  uint16_t* d_y = reinterpret_cast<uint16_t*>(base + 3 * act);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return BEAM_ERR_CUDA;
  int* err_slot = host_error_slot_dev(dev);
  // Decode sizes with page-locked buffers: one kernel reads h and x from the
  // mapped host memory and the layer writes h' and y straight to the host
  // buffers, instead of four copy-engine transfers (about 18 us at 1 token).
  if (T <= 8) {
    void* mh = mapped_host(h_host);
    void* mx = mapped_host(x_host);
    void* mho = mapped_host(h_out_host);
    void* myo = mapped_host(y_out_host);
    if (mh && mx && mho && myo && aligned16(mh) && aligned16(mx) && aligned16(mho) && aligned16(myo) &&
        mho != mx && myo != mh && myo != mx && myo != mho) {
      HostCall k;
      std::memset(&k, 0, sizeof k);
      k.device = dev;
      k.n = n;
      k.T = T;
      k.h = mh;
      k.x = mx;
      k.h_out = mho;
      k.y_out = myo;
      k.wt = *wt;
      if (fp4w != nullptr) {
        k.fp4w = *fp4w;
        k.fp4 = 1;
      }
      k.cfg = *cfg;
      k.ws = ws;
      k.ws_bytes = ws_bytes;
      k.err_out = err_slot;
      const uint64_t hash = hash_call(k);
      bool direct = true;
      {
        std::lock_guard<std::mutex> lock(g_graph_mu);
        HostGraph* g = find_graph(k, hash);
        if (g == nullptr) {
          insert_graph(k, hash)->last_use = ++g_graph_tick;
        } else {
          g->last_use = ++g_graph_tick;
          if (g->exec != nullptr || (!g->failed && capture_graph(g))) {
            if (cudaGraphLaunch(g->exec, s) != cudaSuccess) return BEAM_ERR_CUDA;
            launch_counter() = g->launches;
            direct = false;
          }
        }
      }
      if (direct) {
        launch_counter() = 0;
        if ((st = zero_copy_launches(k, s)) != BEAM_OK) return st;
      }
      if (cudaStreamSynchronize(s) != cudaSuccess) return BEAM_ERR_CUDA;
      return host_call_error(dev, err_slot != nullptr, s);
    }
  }
  if (fp4w == nullptr && T >= kPipeTokens && beam::router_tc_supported(T / pipe_chunks(T), cfg->num_experts, cfg->hidden) &&
      !beam::route_decode_supported(T, cfg->hidden, cfg->num_experts, cfg->num_groups, cfg->topk)) {
    std::lock_guard<std::mutex> lock(g_aux_mu);
    if (CopyAux* a = copy_aux(dev)) {
      DeviceInfo d;
      if ((st = device_info(&d)) != BEAM_OK) return st;
      if (ws_bytes - 4 * act < layer_ws(cfg, T, d.sms).total) return BEAM_ERR_WORKSPACE_TOO_SMALL;
      st = layer_host_pipelined(h_host, x_host, n, wt, T, cfg, h_out_host, y_out_host, d_h, d_x, d_hn, d_y,
                                base + 4 * act, d.sms, s, a, err_slot);
      if (st != BEAM_OK) return st;
      if (cudaStreamSynchronize(s) != cudaSuccess) return BEAM_ERR_CUDA;
      return host_call_error(dev, err_slot != nullptr, s);
    }
  }
  if (cudaMemcpyAsync(d_h, h_host, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) return BEAM_ERR_CUDA;
  if (cudaMemcpyAsync(d_x, x_host, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess) return BEAM_ERR_CUDA;
  if (T >= kOverlapTokens) {
    std::lock_guard<std::mutex> lock(g_aux_mu);
    if (CopyAux* a = copy_aux(dev)) {
      beam_moe_debug_t dbg;
      std::memset(&dbg, 0, sizeof dbg);
      dbg.stage_events[1] = a->after_boundary;  // recorded once h' is written
      st = layer_impl(d_h, d_x, n, wt, T, cfg, d_hn, d_y, &dbg, base + 4 * act, ws_bytes - 4 * act, stream, false,
                      nullptr, err_slot, fp4w);
      if (st != BEAM_OK) return st;
      if (cudaStreamWaitEvent(a->side, a->after_boundary, 0) != cudaSuccess ||
          cudaMemcpyAsync(h_out_host, d_hn, bytes, cudaMemcpyDeviceToHost, a->side) != cudaSuccess ||
          cudaEventRecord(a->h_copied, a->side) != cudaSuccess ||
          cudaMemcpyAsync(y_out_host, d_y, bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
          cudaStreamWaitEvent(s, a->h_copied, 0) != cudaSuccess)
        return BEAM_ERR_CUDA;
      if (cudaStreamSynchronize(s) != cudaSuccess) return BEAM_ERR_CUDA;
      return host_call_error(dev, err_slot != nullptr, s);
    }
  }
  st = layer_impl(d_h, d_x, n, wt, T, cfg, d_hn, d_y, nullptr, base + 4 * act, ws_bytes - 4 * act, stream, false,
                  nullptr, err_slot, fp4w);
  if (st != BEAM_OK) return st;
  if (cudaMemcpyAsync(h_out_host, d_hn, bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess) return BEAM_ERR_CUDA;
  if (cudaMemcpyAsync(y_out_host, d_y, bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess) return BEAM_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return BEAM_ERR_CUDA;
  return host_call_error(dev, err_slot != nullptr, s);
}

}  // namespace

beam_status_t beam_moe_layer_host(const uint16_t* h_host, const uint16_t* x_host, int n,
                                  const beam_moe_weights_t* wt, int T, const beam_moe_config_t* cfg,
                                  uint16_t* h_out_host, uint16_t* y_out_host, void* ws, size_t ws_bytes,
                                  void* stream) {
  return layer_host_impl(h_host, x_host, n, wt, nullptr, T, cfg, h_out_host, y_out_host, ws, ws_bytes, stream);
}

beam_status_t beam_moe_layer_nvfp4_host(const uint16_t* h_host, const uint16_t* x_host, int n,
                                        const beam_moe_nvfp4_weights_t* weights, int T, const beam_moe_config_t* cfg,
                                        uint16_t* h_out_host, uint16_t* y_out_host, void* ws, size_t ws_bytes,
                                        void* stream) {
  if (weights == nullptr) return BEAM_ERR_INVALID_ARG;
  const beam_moe_weights_t shared = {weights->w_post, weights->w_pre, weights->router_w, weights->bias, nullptr,
                                     nullptr};
  return layer_host_impl(h_host, x_host, n, &shared, weights, T, cfg, h_out_host, y_out_host, ws, ws_bytes, stream);
}

beam_status_t beam_release_host_graphs(void) {
  std::lock_guard<std::mutex> lock(g_graph_mu);
  for (HostGraph& g : g_graphs) {
    if (g.exec != nullptr && cudaGraphExecDestroy(g.exec) != cudaSuccess) cudaGetLastError();
    g = HostGraph{};
  }
  g_graph_tick = 0;
  return BEAM_OK;
}

beam_status_t beam_get_device_error(int* code, void* stream) {
  if (code == nullptr) return BEAM_ERR_INVALID_ARG;
  *code = 0;
  if (beam::read_and_clear_device_error(code, static_cast<cudaStream_t>(stream)) != cudaSuccess) return BEAM_ERR_CUDA;
  return *code != 0 ? BEAM_ERR_DEVICE_TIMEOUT : BEAM_OK;
}

beam_status_t beam_check_bounded_wait_pending(int* flag, int limit_ms, void* stream) {
  if (flag == nullptr || limit_ms < 1 || limit_ms > 1000 || !aligned4(flag)) return BEAM_ERR_INVALID_ARG;
  DeviceInfo d;
  beam_status_t st = device_info(&d);
  if (st != BEAM_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  launch_counter() = 0;
  if (beam::launch_bounded_wait_probe(flag, static_cast<uint64_t>(limit_ms) * 1000000ull, beam::kProbeSite, s) !=
      cudaSuccess)
    return BEAM_ERR_CUDA;
  return cuda_status(cudaStreamSynchronize(s));
}

beam_status_t beam_check_bounded_wait(int* flag, int limit_ms, int* site, void* stream) {
  if (flag == nullptr || site == nullptr || limit_ms < 1 || limit_ms > 1000 || !aligned4(flag))
    return BEAM_ERR_INVALID_ARG;
  *site = 0;
  DeviceInfo d;
  beam_status_t st = device_info(&d);
  if (st != BEAM_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int pending = 0;
  if (beam::read_and_clear_device_error(&pending, s) != cudaSuccess) return BEAM_ERR_CUDA;
  if (pending != 0) return BEAM_ERR_DEVICE_TIMEOUT;
  launch_counter() = 0;
  if (beam::launch_bounded_wait_probe(flag, static_cast<uint64_t>(limit_ms) * 1000000ull, beam::kProbeSite, s) !=
      cudaSuccess)
    return BEAM_ERR_CUDA;
  if (beam::read_and_clear_device_error(site, s) != cudaSuccess) return BEAM_ERR_CUDA;
  return *site == beam::kProbeSite ? BEAM_OK : BEAM_ERR_DEVICE_TIMEOUT;
}

}  // extern "C"
