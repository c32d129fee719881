/*
 * beam.h -- C ABI of libbeam.so: the Beam 501B-A23B MoE sublayer at a
 * sandwich-norm boundary, as hand-written CUDA kernels for one GB300 (sm_103a).
 *
 * The method comes from three public pages about serving Reflection Beam:
 * the TokenSpeed blog on Reflection Beam (lightseek.org), the Gaudi cookbook
 * port "Beam-1.0-501B-A23B on Gaudi 2", and a summary of the vLLM Beam post
 * (agentlenshq). Each entry point below names the section that defines its
 * operation.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - bf16 tensors are passed as uint16_t bit patterns (bfloat16), fp32 tensors
 *   as float, indices as int32_t. All tensors are dense and row-major; the
 *   last index is contiguous.
 * - Every tensor pointer is a DEVICE pointer owned by the caller, except in
 *   beam_moe_layer_host, which also takes host buffers. The library never
 *   allocates device memory and keeps no per-call state; scratch memory comes
 *   from the caller's workspace (`ws`, `ws_bytes`, sized by the *_workspace_size
 *   queries, 256-byte aligned, no initial contents required).
 * - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream). All work is enqueued on it; no entry point synchronises, except
 *   beam_moe_layer_host and beam_get_device_error.
 * - Argument errors are detected on the host before anything is launched and
 *   return a status other than BEAM_OK; nothing is enqueued in that case.
 *   A launch failure returns BEAM_ERR_CUDA. Asynchronous device errors show up
 *   in later CUDA calls; a timed-out bounded wait inside a kernel is reported
 *   by beam_get_device_error.
 * - T == 0 is a valid empty batch: the call checks its config and returns
 *   BEAM_OK without launching anything.
 * - Alignment: every bf16 and fp32 tensor must be 16-byte aligned (128-bit
 *   vector loads and TMA); int32 tensors 4-byte aligned.
 * - Supported shapes: H % 256 == 0 and H <= 8192; F % 64 == 0 (e.g. 320, one
 *   GPU's slice of d_ff 2560 under 8-way tensor parallelism); E <= 256;
 *   E % G == 0; G <= 32; E/G <= 32; 1 <= TG <= G; 1 <= K <= 16;
 *   K <= TG * E/G; T * K < 2^31.
 */
#ifndef BEAM_H
#define BEAM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  BEAM_OK = 0,
  BEAM_ERR_INVALID_ARG = 1,         /* null pointer, negative size, bad config value */
  BEAM_ERR_MISALIGNED = 2,          /* pointer not aligned as the conventions require */
  BEAM_ERR_UNSUPPORTED_SHAPE = 3,   /* shape outside the supported set above */
  BEAM_ERR_WORKSPACE_TOO_SMALL = 4, /* ws_bytes below the matching *_workspace_size */
  BEAM_ERR_CUDA = 5,                /* a CUDA runtime call or kernel launch failed */
  BEAM_ERR_DEVICE_TIMEOUT = 6,      /* a bounded wait inside a kernel gave up */
  BEAM_ERR_UNSUPPORTED_DEVICE = 7   /* current device is not compute capability 10.3 */
} beam_status_t;

/* Shape and scalars of one MoE sublayer. Beam: hidden 5120, 256 experts in 8
 * groups, top 4 groups, top 8 experts, d_ff 2560, routed scale 2.5, eps 1e-6
 * (vLLM Beam summary, "MoE and residual stream"; TokenSpeed blog,
 * "Model architecture and precision -> Architecture"). */
typedef struct {
  int hidden;          /* H */
  int num_experts;     /* E */
  int num_groups;      /* G: contiguous groups of E/G experts */
  int topk_groups;     /* TG */
  int topk;            /* K */
  int d_ff;            /* F */
  float routed_scale;  /* 2.5 for Beam */
  float eps;           /* RMSNorm epsilon */
} beam_moe_config_t;

/* Weights of one MoE sublayer (all device pointers). */
typedef struct {
  const uint16_t* w_post;     /* bf16 [H]: RMSNorm weight after the previous sublayer */
  const uint16_t* w_pre;      /* bf16 [H]: RMSNorm weight before this MoE sublayer */
  const float* router_w;      /* fp32 [E][H] (one row per expert) */
  const float* bias;          /* fp32 [E]: correction bias, used for selection only */
  const uint16_t* w_gate_up;  /* bf16 [E][2F][H]: rows 0..F-1 gate, rows F..2F-1 up */
  const uint16_t* w_down;     /* bf16 [E][H][F] */
} beam_moe_weights_t;

/* Optional intermediate outputs of beam_moe_layer (each may be NULL). */
typedef struct {
  uint16_t* z;              /* bf16 [T][H]: pre-normed MoE input */
  float* logits;            /* fp32 [T][E]: router logits */
  int32_t* topk_ids;        /* int32 [T][K] */
  float* topk_w;            /* fp32 [T][K] */
  int32_t* expert_offsets;  /* int32 [E+1] */
  /* Optional cudaEvent_t handles (as void*, NULL to skip) recorded on the
   * stream at the stage boundaries: [0] before the boundary norm, [1] after
   * it, [2] after router + top-k, [3] after the permutation, [4] after the
   * gate/up GEMM, [5] after the down GEMM, [6] after the combine. Used for
   * per-kernel timing; the events are created and owned by the caller. */
  void* stage_events[7];
} beam_moe_debug_t;

const char* beam_status_string(beam_status_t status);
const char* beam_version(void);

/* Sandwich-norm boundary (vLLM Beam summary, "MoE and residual stream" and
 * kernel change 1; TokenSpeed blog, "MNNVL all-reduce and SandwichNorm
 * fusion"; Gaudi cookbook port, "What was built -> Model code"):
 *   y  = bf16(x / sqrt(mean(x^2) + eps) * w_post)
 *   h' = bf16(sqrt((n-1)/n) * h + y / sqrt(n))
 *   z  = bf16(h' / sqrt(mean(h'^2) + eps) * w_pre)
 * in FP32 math with the three bf16 rounding points shown. h, x: [T][H];
 * h_out, z_out: [T][H]. h_out may alias h (in-place update of the residual);
 * no other aliasing. n >= 1 is the 1-based index of this residual add. */
beam_status_t beam_boundary_norm(const uint16_t* h, const uint16_t* x, const uint16_t* w_post,
                                 const uint16_t* w_pre, int T, int H, float eps, int n,
                                 uint16_t* h_out, uint16_t* z_out, void* stream);

/* FP32 router and group-limited top-k (TokenSpeed blog, "Fused FP32
 * routing" and "Model architecture and precision -> Architecture"; vLLM Beam
 * summary, "MoE and residual stream"; Gaudi cookbook port, "Model code"):
 *   logits = z W_r^T with fp32 FMA (no TF32, no bf16), s = sigmoid(logits),
 *   s' = s + bias; group score = sum of the two largest s' in each group of
 *   E/G contiguous experts; the TG best groups, then the K best s' inside
 *   them (ties to the lower index); slots in descending s';
 *   topk_w[t][k] = routed_scale * s_k / sum_j s_j (unbiased scores).
 * z: bf16 [T][H]; router_w fp32 [E][H]; bias fp32 [E]; logits_out fp32 [T][E]
 * (required: it also serves as the scores buffer); topk_ids int32 [T][K];
 * topk_w fp32 [T][K]. */
beam_status_t beam_router_topk(const uint16_t* z, const float* router_w, const float* bias, int T,
                               const beam_moe_config_t* cfg, float* logits_out, int32_t* topk_ids,
                               float* topk_w, void* stream);

/* Permutation by expert (vLLM Beam summary, "The fused decoding graph runs
 * one MoE layer in 13 kernels": routing kernels feed grouped GEMMs). The T*K
 * pairs i = t*K + k are ordered by (expert, t): a stable counting sort built
 * from a histogram and an exclusive prefix scan, with no atomics deciding the
 * order. Outputs: expert_offsets int32 [E+1] (offsets[e]..offsets[e+1] are
 * expert e's rows), perm_token int32 [T*K] (token of each permuted row),
 * inv_perm int32 [T*K] (row of pair i), and, if x_perm is not NULL,
 * x_perm bf16 [T*K][H] with x_perm[p] = z[perm_token[p]]. */
size_t beam_moe_permute_workspace_size(const beam_moe_config_t* cfg, int T);
beam_status_t beam_moe_permute(const int32_t* topk_ids, const uint16_t* z, int T,
                               const beam_moe_config_t* cfg, int32_t* expert_offsets,
                               int32_t* perm_token, int32_t* inv_perm, uint16_t* x_perm, void* ws,
                               size_t ws_bytes, void* stream);

/* beam_moe_permute for callers that cannot provide a workspace (the pages
 * have no counterpart; this is a convenience of this library). Some callers
 * have no way to hand the library scratch memory -- for example an operator
 * plugin that only receives the tensors it declares, or a latency-critical
 * loop where a device allocation is not allowed. This variant runs the same
 * kernels as beam_moe_permute with its scratch in a fixed array inside the
 * library's device memory (131,328 bytes per GPU, held until the process
 * exits), so it takes no workspace and allocates nothing. Arguments and
 * outputs are those of beam_moe_permute. Limits: T * K <= BEAM_NO_ALLOC_MAX_PAIRS
 * and E <= 256, else BEAM_ERR_WORKSPACE_TOO_SMALL. All calls on a device share
 * the array: calls whose kernels may overlap on the GPU (unordered streams)
 * race and must not be issued. The first call on each device looks up the
 * array's device address; make it before any stream capture on that device.
 * Only a successful lookup is kept (a failed one is retried by the next call),
 * and it is kept for the life of the process: resetting the device
 * (cudaDeviceReset) after the first call is not supported. */
#define BEAM_NO_ALLOC_MAX_PAIRS 131072
beam_status_t beam_moe_permute_no_alloc(const int32_t* topk_ids, const uint16_t* z, int T,
                                        const beam_moe_config_t* cfg, int32_t* expert_offsets,
                                        int32_t* perm_token, int32_t* inv_perm, uint16_t* x_perm,
                                        void* stream);

/* Routed SwiGLU experts and weighted combine (TokenSpeed blog, "TensorRT-LLM
 * NVFP4 MoE": both expert GEMMs, SwiGLU fused into the first, weighted sum of
 * expert outputs per token; vLLM Beam summary: 256 experts, d_ff 2560):
 *   act[p]  = bf16(silu(x_perm[p] W_g^T) * (x_perm[p] W_u^T))   (gate/up GEMM)
 *   y_perm[p] = bf16(act[p] W_d^T)                              (down GEMM)
 *   y[t]   = bf16(sum_k topk_w[t][k] * y_perm[inv_perm[t*K+k]]) (combine, k in order)
 * for the expert e that owns row p. Grouped GEMMs on tcgen05 tensor cores with
 * fp32 accumulation in tensor memory, fed by TMA. The combine is atomic-free
 * and deterministic. y_out: bf16 [T][H]. */
size_t beam_moe_experts_workspace_size(const beam_moe_config_t* cfg, int T);
beam_status_t beam_moe_experts(const uint16_t* x_perm, const int32_t* expert_offsets,
                               const uint16_t* w_gate_up, const uint16_t* w_down,
                               const float* topk_w, const int32_t* inv_perm, int T,
                               const beam_moe_config_t* cfg, uint16_t* y_out, void* ws,
                               size_t ws_bytes, void* stream);

/* The three stages of beam_moe_experts, exposed for inspection and for timing
 * each kernel on its own. act: bf16 [T*K][F]; y_perm: bf16 [T*K][H].
 * beam_moe_gate_up and beam_moe_down need beam_moe_experts_workspace_size
 * bytes of workspace (their split-K partial sums). */
beam_status_t beam_moe_gate_up(const uint16_t* x_perm, const int32_t* expert_offsets,
                               const uint16_t* w_gate_up, int T, const beam_moe_config_t* cfg,
                               uint16_t* act, void* ws, size_t ws_bytes, void* stream);
beam_status_t beam_moe_down(const uint16_t* act, const int32_t* expert_offsets,
                            const uint16_t* w_down, int T, const beam_moe_config_t* cfg,
                            uint16_t* y_perm, void* ws, size_t ws_bytes, void* stream);
beam_status_t beam_moe_combine(const uint16_t* y_perm, const float* topk_w, const int32_t* inv_perm,
                               int T, const beam_moe_config_t* cfg, uint16_t* y_out, void* stream);

/* The whole sublayer: boundary -> router/top-k -> permutation -> experts ->
 * combine, as stream-ordered launches. Inputs: residual h and previous
 * sublayer output x, bf16 [T][H]; n = index of this residual add. Outputs:
 * the new residual h_out and the MoE output y_out (the next boundary's x),
 * bf16 [T][H]. h_out may alias h. dbg may be NULL. */
size_t beam_moe_workspace_size(const beam_moe_config_t* cfg, int T);
beam_status_t beam_moe_layer(const uint16_t* h, const uint16_t* x, int n,
                             const beam_moe_weights_t* weights, int T,
                             const beam_moe_config_t* cfg, uint16_t* h_out, uint16_t* y_out,
                             const beam_moe_debug_t* dbg, void* ws, size_t ws_bytes, void* stream);

/* The combine deferred to the next boundary (vLLM Beam summary, kernel
 * change list: the norm kernel that follows the MoE also combines the top-8
 * expert outputs). beam_moe_layer_uncombined runs beam_moe_layer up to and
 * including the down GEMM and leaves out the combine; *out receives the
 * addresses, inside `ws`, of the combine's inputs, valid until `ws` is next
 * used. beam_boundary_norm_combine is the next boundary with x taken as that
 * combine: x[t] = bf16(sum_k topk_w[t][k] * y_perm[inv_perm[t*K+k]]) formed
 * exactly as beam_moe_combine forms it, then beam_boundary_norm(h, x, ...);
 * the outputs are the same bits as those two calls, in one launch, and y is
 * neither written nor read. y_perm bf16 [T*K][H], topk_w fp32 [T][K],
 * inv_perm int32 [T*K] (-1: dropped pair), K <= 16. h_out may alias h; z_out
 * aliases nothing; neither may alias y_perm. Both are launched with
 * programmatic dependent launch: they read their weights (w_post, w_pre;
 * for the layer also the router and bias) before the previous kernel on the
 * stream has finished, so no kernel just before them may write those. */
typedef struct {
  const uint16_t* y_perm;   /* bf16 [T*K][H]: expert outputs, permuted order */
  const float* topk_w;      /* fp32 [T][K]: routing weights */
  const int32_t* inv_perm;  /* int32 [T*K]: row of pair t*K+k in y_perm, -1 if dropped */
} beam_moe_uncombined_t;
beam_status_t beam_moe_layer_uncombined(const uint16_t* h, const uint16_t* x, int n,
                                        const beam_moe_weights_t* weights, int T,
                                        const beam_moe_config_t* cfg, uint16_t* h_out,
                                        beam_moe_uncombined_t* out, void* ws, size_t ws_bytes,
                                        void* stream);
beam_status_t beam_boundary_norm_combine(const uint16_t* h, const uint16_t* y_perm,
                                         const float* topk_w, const int32_t* inv_perm, int K,
                                         const uint16_t* w_post, const uint16_t* w_pre, int T,
                                         int H, float eps, int n, uint16_t* h_out,
                                         uint16_t* z_out, void* stream);

/* ------------------------------------------------------------------ NVFP4 experts
 * The expert GEMMs on 4-bit weights and inputs (TokenSpeed blog, "Model
 * architecture and precision -> NVFP4 and FP8 checkpoints": each expert weight
 * is an E2M1 value, every 16 weights share an E4M3 scale and each expert has
 * an additional FP32 scale; expert inputs are quantized in the same format at
 * runtime, so the GEMMs run FP4 x FP4; "TensorRT-LLM NVFP4 MoE": the kernel
 * reads about a quarter of the BF16 weight bytes). Block-scaled tcgen05 MMAs.
 *
 * One block = 16 consecutive values along the reduction dimension of a row.
 * With FP32 scale g, its scale is s = E4M3(amax / (6 g)) and each value's code
 * q = E2M1(x / (s g)), both rounded to nearest even and saturating (448, 6),
 * every product and quotient in FP32; the value represented is q * s * g. An
 * expert's g is its largest |w| over gate, up and down divided by 6 * 448.
 * Codes are stored two per byte, element 2j in the low nibble.
 *
 * Weight layouts (produced by beam_nvfp4_quantize_experts):
 *   q_gate_up  uint8 [E][2F][H/2]  (rows 0..F-1 gate, F..2F-1 up)
 *   q_down     uint8 [E][H][F/2]
 *   sf_gate_up uint8 [2E][F/128][H/256][4][512]: plane 2e = expert e's gate
 *              rows, 2e+1 its up rows; per 128-row block and 256-value k-step
 *              four 512-byte atoms (one per 64 values); in atom c, byte
 *              (r%32)*16 + (r/32)*4 + j is the scale of row r (0..127 in the
 *              block), values 64c + 16j .. +15 of the k-step
 *   sf_down    uint8 [E][H/128][F/256][4][512], the same arrangement
 *   expert_scale float [E]
 * Activation layout (beam_nvfp4_quantize_rows and the layer's internal
 * buffers): codes uint8 [rows][K/2]; scales uint8 [rows][K/64][16], one
 * 16-byte slot per 64 values whose bytes 0..3 are the four 16-value scales
 * (bytes 4..15 are never read; beam_nvfp4_quantize_rows writes zeros there).
 * Shapes: H % 256 == 0, F % 256 == 0, E <= 256. */
typedef struct {
  const uint16_t* w_post;      /* bf16 [H] */
  const uint16_t* w_pre;       /* bf16 [H] */
  const float* router_w;       /* fp32 [E][H] */
  const float* bias;           /* fp32 [E] */
  const uint8_t* q_gate_up;    /* see above */
  const uint8_t* sf_gate_up;
  const uint8_t* q_down;
  const uint8_t* sf_down;
  const float* expert_scale;   /* [E] */
  float input_scale;           /* FP32 scale of the quantized expert input (the pre-normed z), > 0 */
  float act_scale;             /* FP32 scale of the quantized SwiGLU output (the down GEMM's input), > 0 */
} beam_moe_nvfp4_weights_t;

/* Sizes in bytes of the four weight arrays (any pointer may be NULL);
 * returns their total plus the expert scales, 0 for an unsupported config. */
size_t beam_nvfp4_expert_bytes(const beam_moe_config_t* cfg, size_t* q_gate_up, size_t* sf_gate_up,
                               size_t* q_down, size_t* sf_down);

/* Quantizes bf16 expert weights (the beam_moe_weights_t layouts) to the NVFP4
 * layouts above: one pass for each expert's largest |w|, one that writes
 * codes and scales, one for the expert scales. Every output is written. */
beam_status_t beam_nvfp4_quantize_experts(const uint16_t* w_gate_up, const uint16_t* w_down,
                                          const beam_moe_config_t* cfg, uint8_t* q_gate_up,
                                          uint8_t* sf_gate_up, uint8_t* q_down, uint8_t* sf_down,
                                          float* expert_scale, void* stream);

/* Runtime quantization of bf16 rows x [rows][K] with FP32 scale `scale`
 * (K % 64 == 0): codes q [rows][K/2], scale slots sf [rows][K/64][16]. */
beam_status_t beam_nvfp4_quantize_rows(const uint16_t* x, int rows, int K, float scale, uint8_t* q,
                                       uint8_t* sf, void* stream);

/* The NVFP4 experts stage: x_perm (bf16 [T*K][H], beam_moe_permute's rows)
 * quantized with input_scale; per expert, act = silu(gate) * up from the
 * block-scaled gate/up GEMM times the expert and input scales, quantized
 * with act_scale; y_perm = bf16(act GEMM W_down times the expert and act
 * scales); the combine as in beam_moe_experts. y_out bf16 [T][H]. `inter`
 * (may be NULL) receives the workspace addresses of the intermediates,
 * valid until `ws` is next used. */
typedef struct {
  const uint8_t* x_q;       /* [T*K][H/2] */
  const uint8_t* x_sf;      /* [T*K][H/64][16] */
  const uint8_t* act_q;     /* [T*K][F/2] */
  const uint8_t* act_sf;    /* [T*K][F/64][16] */
  const uint16_t* y_perm;   /* bf16 [T*K][H] */
} beam_moe_nvfp4_intermediates_t;
size_t beam_moe_experts_nvfp4_workspace_size(const beam_moe_config_t* cfg, int T);
beam_status_t beam_moe_experts_nvfp4(const uint16_t* x_perm, const int32_t* expert_offsets,
                                     const beam_moe_nvfp4_weights_t* weights, const float* topk_w,
                                     const int32_t* inv_perm, int T, const beam_moe_config_t* cfg,
                                     uint16_t* y_out, beam_moe_nvfp4_intermediates_t* inter, void* ws,
                                     size_t ws_bytes, void* stream);

/* beam_moe_layer with NVFP4 experts: the same boundary, FP32 routing and
 * permutation, then beam_moe_experts_nvfp4. dbg as for beam_moe_layer (its
 * stage event [3] is recorded after the input quantization). At decode sizes
 * (T <= 8, 256 experts in 8 groups) the routing launch writes the permuted
 * rows already quantized (the same codes and scales as
 * beam_nvfp4_quantize_rows), and the expert launch starts on its flags. */
size_t beam_moe_nvfp4_workspace_size(const beam_moe_config_t* cfg, int T);
beam_status_t beam_moe_layer_nvfp4(const uint16_t* h, const uint16_t* x, int n,
                                   const beam_moe_nvfp4_weights_t* weights, int T,
                                   const beam_moe_config_t* cfg, uint16_t* h_out, uint16_t* y_out,
                                   const beam_moe_debug_t* dbg, void* ws, size_t ws_bytes, void* stream);

/* beam_moe_layer with HOST input and output buffers: copies h and x (host,
 * pinned memory recommended) into the workspace, runs the layer, copies h_out
 * and y_out back to the host buffers, and synchronises the stream before it
 * returns. Up to 8 tokens, when all four host buffers are page-locked (mapped
 * into the device address space) and 16-byte aligned, one kernel reads h and x
 * from the mapped memory and the layer writes h_out and y_out to it directly
 * instead of four copy-engine transfers; the results are the same bits. h_out
 * must not alias x; y_out must alias none of the others. Weights stay device
 * pointers. Workspace: beam_moe_layer_host_workspace_size. From 8192 tokens
 * (bf16 experts, Beam-size router) the layer runs pipelined with the copies:
 * the tokens are copied in four chunks, each chunk's boundary, router and
 * top-k start once its copy has landed, and the combine and the copy of y back
 * go chunk by chunk; the results are the same bits.
 * Repeated calls on that mapped-memory path: the second call with the same
 * device, buffers, n, T, weights, config and workspace captures its launches
 * into a CUDA graph, and later calls with the same arguments replay it (one
 * launch instead of five; the same kernels and results). The library keeps up
 * to 256 such graphs per process, evicting the least recently used;
 * beam_release_host_graphs frees them. Buffer contents may change freely
 * between calls; the graphs hold only addresses.
 * After its synchronise the call reads the device error word (see
 * beam_get_device_error): if a bounded wait inside a kernel gave up, it clears
 * the word and returns BEAM_ERR_DEVICE_TIMEOUT (the outputs are then
 * incomplete). The word is shared by every call on the device, so a call may
 * also report a timeout of another call that overlapped it on the GPU. */
size_t beam_moe_layer_host_workspace_size(const beam_moe_config_t* cfg, int T);
beam_status_t beam_moe_layer_host(const uint16_t* h_host, const uint16_t* x_host, int n,
                                  const beam_moe_weights_t* weights, int T,
                                  const beam_moe_config_t* cfg, uint16_t* h_out_host,
                                  uint16_t* y_out_host, void* ws, size_t ws_bytes, void* stream);

/* beam_moe_layer_host with NVFP4 experts (the layer of beam_moe_layer_nvfp4):
 * the same host-buffer rules, mapped-memory path and graph replays.
 * Workspace: beam_moe_layer_nvfp4_host_workspace_size (0 for shapes the
 * NVFP4 experts do not support). */
size_t beam_moe_layer_nvfp4_host_workspace_size(const beam_moe_config_t* cfg, int T);
beam_status_t beam_moe_layer_nvfp4_host(const uint16_t* h_host, const uint16_t* x_host, int n,
                                        const beam_moe_nvfp4_weights_t* weights, int T,
                                        const beam_moe_config_t* cfg, uint16_t* h_out_host,
                                        uint16_t* y_out_host, void* ws, size_t ws_bytes, void* stream);

/* Frees every graph that beam_moe_layer_host has captured (their memory
 * only: a captured graph runs only when a call repeats its exact arguments,
 * so freeing or reusing buffers needs no release first). Always BEAM_OK. */
beam_status_t beam_release_host_graphs(void);

/* Reads and clears the library's device error word on the current device
 * after synchronising `stream`. *code receives 0 if no bounded wait timed
 * out, otherwise a nonzero site code; returns BEAM_ERR_DEVICE_TIMEOUT then.
 * There is one word per device for the whole process: it is not tied to a
 * stream or a call. A timeout in any call on the device (on any stream) sets
 * it until some call reads it here, in beam_check_bounded_wait or in
 * beam_moe_layer_host; callers that run layers on several streams at once
 * should read it after synchronising all of them. */
beam_status_t beam_get_device_error(int* code, void* stream);

/* Diagnostic with no counterpart in the pages: checks on the device that a
 * bounded wait gives up and reports instead of hanging. One thread waits,
 * through the same wait routine the fused experts launch uses for its
 * cross-CTA counters and routing flags, on a flag that nothing sets, for
 * `limit_ms` (1..1000) milliseconds. `flag`: 4 writable device bytes, 4-byte
 * aligned, zeroed here. Synchronises `stream`; the error word is cleared
 * before returning. Returns BEAM_OK when the wait timed out and reported its
 * site code (*site receives it), BEAM_ERR_DEVICE_TIMEOUT if another site code
 * was pending or none was recorded, BEAM_ERR_INVALID_ARG on bad arguments. */
beam_status_t beam_check_bounded_wait(int* flag, int limit_ms, int* site, void* stream);

/* The same diagnostic wait, but the site code it records is left pending in
 * the device error word (for a later beam_get_device_error or
 * beam_moe_layer_host to report and clear). Synchronises `stream`. Returns
 * BEAM_OK once the wait has given up, BEAM_ERR_INVALID_ARG on bad arguments. */
beam_status_t beam_check_bounded_wait_pending(int* flag, int limit_ms, void* stream);

/* Kernel launches issued by the most recent call of each kind on this host
 * thread's view (a count, for reporting). */
int beam_last_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* BEAM_H */
