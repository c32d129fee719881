// Internal interface between the C ABI (api.cu) and the kernel translation
// units. Plain pointers and sizes; every launcher enqueues on `stream` and
// returns the launch status.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace beam {

// Number of kernel launches issued by the calling host thread since the
// counter was last reset (for reporting).
int& launch_counter();

// ---- boundary (boundary.cu)
// n >= 1 is the index of the residual add (coefficients sqrt((n-1)/n), 1/sqrt(n))
// `pdl`: launch with programmatic stream serialization (every kernel waits for
// its predecessor before reading its outputs or writing global memory).
cudaError_t launch_boundary(const uint16_t* h, const uint16_t* x, const uint16_t* w_post, const uint16_t* w_pre,
                            int T, int H, float eps, int n, uint16_t* h_out, uint16_t* z_out, cudaStream_t stream,
                            bool pdl = false, int* zero_slot = nullptr);
bool boundary_supported(int H);
// The boundary with x = the combine of the token's K expert outputs
// (y_perm rows inv_perm[t*K+k], weights topk_w[t][k]; K <= 16), formed as
// launch_combine forms it: the same bits as combine followed by the boundary.
cudaError_t launch_boundary_combine(const uint16_t* h, const uint16_t* y_perm, const float* topk_w,
                                    const int32_t* inv_perm, int K, const uint16_t* w_post, const uint16_t* w_pre,
                                    int T, int H, float eps, int n, uint16_t* h_out, uint16_t* z_out,
                                    cudaStream_t stream, bool pdl = false);

// ---- router (router.cu)
cudaError_t launch_router_logits(const uint16_t* z, const float* W, int T, int H, int E, float* logits,
                                 cudaStream_t stream, bool pdl = false);
// Router and top-k in one launch (T <= 32, 256 experts in 8 groups): the last
// block runs the selection. `ticket` must be zero on entry and is left zero.
bool router_topk_fusable(int T, int E, int G);
cudaError_t launch_router_topk_fused(const uint16_t* z, const float* W, const float* bias, int T, int H, int E,
                                     int G, int TG, int K, float scale, float* logits, int32_t* ids, float* w,
                                     int* ticket, cudaStream_t stream, bool pdl);
// Tensor-core FP32 router for T > 128: splits W exactly into three bf16 terms
// (`w3`, router_tc_scratch_bytes) and accumulates all three in fp32.
bool router_tc_supported(int T, int E, int H);
size_t router_tc_scratch_bytes(int E, int H);
cudaError_t launch_router_tc(const uint16_t* z, const float* W, int T, int E, int H, float* logits, uint16_t* w3,
                             int num_sms, cudaStream_t stream, bool pdl);
cudaError_t launch_topk(const float* logits, const float* bias, int T, int E, int G, int TG, int K, float scale,
                        int32_t* ids, float* w, cudaStream_t stream, bool pdl = false);

// ---- decode routing (route_decode.cu)
// Boundary -> router -> top-k -> permutation -> row gather in one launch, and
// `clear_bytes` of `clear` zeroed (the experts' counters and tickets), for
// T <= 8 with 256 experts in 8 groups. `sync` (kRouteSyncInts ints, zeroed by
// a memset before the launch unless `sync_zeroed`: then an earlier kernel on
// the stream zeroed them): [0] the blocks' ticket (left zero), [1] set once
// offsets, permutation and the cleared scratch are valid, [2] set once the
// permuted rows are valid (the fused experts launch polls [1] and [2]).
// With `xq` set the permuted rows are written as NVFP4 (codes [rows][H/2] to
// `xq`, scale slots [rows][H/64][16] to `xsf`, FP32 scale g_in) instead of
// bf16 to `x_perm`.
constexpr int kRouteSyncInts = 4;
bool route_decode_supported(int T, int H, int E, int G, int K);
cudaError_t launch_route_decode(const uint16_t* h, const uint16_t* x, const uint16_t* w_post, const uint16_t* w_pre,
                                const float* W, const float* bias, int T, int H, int E, int G, int TG, int K,
                                float scale, float eps, int n, uint16_t* h_out, uint16_t* z_out, float* logits,
                                int32_t* ids, float* w, int32_t* offsets, int32_t* perm_token, int32_t* inv_perm,
                                uint16_t* x_perm, int* sync, void* clear, size_t clear_bytes, int num_sms,
                                cudaStream_t stream, bool pdl, bool sync_zeroed = false, uint8_t* xq = nullptr,
                                uint8_t* xsf = nullptr, float g_in = 0.f);

// ---- permutation (permute.cu)
size_t permute_scratch_bytes(int T, int K, int E);
// `clear` (optional): bytes zeroed before the permutation completes (the
// experts' counters and tickets), inside the kernel at small sizes.
cudaError_t launch_permute(const int32_t* ids, const uint16_t* z, int T, int K, int E, int H, int32_t* offsets,
                           int32_t* perm_token, int32_t* inv_perm, uint16_t* x_perm, void* scratch,
                           cudaStream_t stream, bool pdl = false, void* clear = nullptr, size_t clear_bytes = 0);

// ---- experts (experts.cu)
struct GemmPlan {
  int bn;               // token tile (MMA N): 16 .. 128 (256 for the down GEMM)
  int split;            // split-K factor (1 = no partial sums)
  int max_token_tiles;  // upper bound on (expert, token-tile) pairs
  int max_tiles;        // upper bound on (expert, row-block, token-tile) tiles
  bool pair;            // prefill: paired-SM launch with 256-token tiles (launch_gemm_pair)
};
// mode 0: gate/up + SwiGLU (weight rows 2F, reduction H); mode 1: down (rows H, reduction F).
// `fp4`: NVFP4 operands (256-value k-steps, token tiles of at most 32).
GemmPlan plan_gemm(int mode, int T, int K, int E, int H, int F, int num_sms, int units_per_sm = 16,
                   bool fp4 = false);
// The plans of a gate/up + down pass as run by the experts stage (the fused
// launch when fused_experts_supported, else two launches).
void plan_experts(int T, int K, int E, int H, int F, int num_sms, GemmPlan* gate_up, GemmPlan* down,
                  bool fp4 = false);
// Scratch shared by one gate/up + down pass (unit counters, split-K tickets
// and partial sums); it must be cleared with clear_gemm_scratch before the
// gate/up GEMM (one memset; each GEMM leaves its tickets at zero).
size_t gemm_scratch_bytes(const GemmPlan& gate_up, const GemmPlan& down);
cudaError_t clear_gemm_scratch(void* scratch, const GemmPlan& gate_up, const GemmPlan& down, cudaStream_t stream);
size_t gemm_clear_bytes(const GemmPlan& gate_up, const GemmPlan& down);
// Both GEMMs in one persistent launch (down units of a token tile wait for the
// gate/up tiles that produce its rows); needs equal token tiles of <= 64.
bool fused_experts_supported(const GemmPlan& gate_up, const GemmPlan& down);
// `ready` (optional): the decode routing kernel's flags [1] and [2]; the launch
// then reads offsets and scratch once [1] is set and the permuted rows once
// [2] is set, instead of waiting for the previous kernel to finish.
cudaError_t launch_fused_experts(const GemmPlan& gate_up, const GemmPlan& down, const uint16_t* w_gate_up,
                                 const uint16_t* w_down, const uint16_t* x_perm, const int32_t* offsets, int rows,
                                 int E, int H, int F, uint16_t* act, uint16_t* y_perm, void* scratch, int num_sms,
                                 cudaStream_t stream, bool pdl, const int* ready = nullptr);
// One expert GEMM on CTA pairs (clusters of two, cta_group::2 MMAs, 256-token
// tiles); mode 0 gate/up + SwiGLU, mode 1 down. `counter`: the launch's unit
// counter, zero before the launch.
cudaError_t launch_gemm_pair(int mode, const uint16_t* weights, const uint16_t* act_in, const int32_t* offsets,
                             int rows, int E, int H, int F, uint16_t* out, int* counter, int num_sms,
                             cudaStream_t stream, bool pdl);
cudaError_t launch_gemm(int mode, const GemmPlan& gate_up, const GemmPlan& down, const uint16_t* weights,
                        const uint16_t* act_in, const int32_t* offsets, int rows, int E, int H, int F, uint16_t* out,
                        void* scratch, int num_sms, cudaStream_t stream, bool pdl = false);
// ---- NVFP4 experts (nvfp4.cu, experts.cu)
// Expert weights as E2M1 codes (two per byte), E4M3 scales per 16 values in
// 512-byte atoms, and one FP32 scale per expert (layouts in beam.h).
struct Nvfp4Experts {
  const uint8_t* q_gate_up;   // [E][2F][H/2]
  const uint8_t* sf_gate_up;  // [2E][F/128][H/256][4][512]
  const uint8_t* q_down;      // [E][H][F/2]
  const uint8_t* sf_down;     // [E][H/128][F/256][4][512]
  const float* scale;         // [E]
};
bool nvfp4_experts_supported(int E, int H, int F);
cudaError_t launch_quantize_experts(const uint16_t* w_gu, const uint16_t* w_d, int E, int H, int F, uint8_t* q_gu,
                                    uint8_t* sf_gu, uint8_t* q_d, uint8_t* sf_d, float* expert_scale, int num_sms,
                                    cudaStream_t stream);
// rows x K bf16 -> codes [rows][K/2] and scale slots [rows][K/64][16] (K % 64 == 0)
cudaError_t launch_quantize_rows(const uint16_t* x, int rows, int K, float g, uint8_t* q, uint8_t* sf,
                                 cudaStream_t stream, bool pdl = false);
// Both NVFP4 GEMMs in one persistent launch (plans from plan_experts with
// fp4, token tiles <= 32): gate/up + SwiGLU writes the SwiGLU output as
// NVFP4 (act_q, act_sf, FP32 scale act_scale); down writes bf16 y_perm.
cudaError_t launch_fused_experts_fp4(const GemmPlan& gate_up, const GemmPlan& down, const Nvfp4Experts& wt,
                                     const uint8_t* xq, const uint8_t* xsf, float x_scale, const int32_t* offsets,
                                     int rows, int E, int H, int F, uint8_t* act_q, uint8_t* act_sf, float act_scale,
                                     uint16_t* y_perm, void* scratch, int num_sms, cudaStream_t stream, bool pdl,
                                     const int* ready = nullptr);
// `err_out` (optional, device-visible): receives the device error word once
// the expert launch before the combine has completed.
cudaError_t launch_combine(const uint16_t* y_perm, const float* w, const int32_t* inv_perm, int T, int K, int H,
                           uint16_t* y, cudaStream_t stream, bool pdl = false, int* err_out = nullptr);
cudaError_t read_and_clear_device_error(int* code, cudaStream_t stream);
// One bounded wait on `flag` (zeroed here) that nothing sets: records `site`.
constexpr int kProbeSite = 99;
cudaError_t launch_bounded_wait_probe(int* flag, uint64_t limit_ns, int site, cudaStream_t stream);

}  // namespace beam
