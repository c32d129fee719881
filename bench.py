#!/usr/bin/env python
"""Throughput of the Beam MoE sublayer on GB300, on the five workloads.

One step = one pass of the whole sublayer (boundary norm -> FP32 router and
group top-k -> permutation -> gate/up GEMM with SwiGLU -> down GEMM ->
combine) over one batch of synthetic tokens, through the C ABI
(beam_moe_layer). With no arguments every workload runs in one process, in
order: the toy sublayer (16 tokens), then Beam shapes (hidden 5120, 256
experts in 8 groups, top 4 groups / top 8 experts, d_ff 2560) at 1, 64, 2048
and 16384 tokens. The headline numbers (value, ms_per_step, roofline, e2e)
are those of the largest workload, 16384 tokens; every workload's numbers
are under ``per_config``, and its agreement with the fp64 oracle under
``parity``.

Timing: W untimed warm-up steps, then K steps. Before each step a 512 MB
buffer is overwritten (L2 is 129 MB) and then read back, so L2 holds none of
the step's data and no dirty lines whose write-back would fall inside the
step; the input batch rotates over several seeded draws, so expert weights
come from HBM. Each batch's layer is captured once as a CUDA graph and every
timed step replays one, between CUDA events on the replay stream. A second
pass with CUDA events at every stage boundary (recorded by the library on the
launching stream) times each kernel. The flush is outside the events.

Parity: after the timed passes, batch 0 of each workload is checked against
the fp64 CPU oracle (which the GPU path shares no code with): routing and h'
on every token (on the 512 seeded oracle tokens at 16384 tokens), the layer
output y on a few tokens. The oracle run on the largest workload's tokens is
also timed as the CPU baseline.

Prints one JSON line (rank 0). Multi-GPU (torchrun): every rank runs the same
workloads on its own GPU (tokens are independent: replicas, weak scaling);
each value is all ranks' tokens over the slowest rank's time.

``--impl reference`` times the fp64 CPU oracle on the headline workload
instead (one token per step, host cores).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from beam_inputs import CONFIGS, make_norm_weights, make_router, sample_tokens, shared_direction  # noqa: E402

METRIC = "MoE-sublayer tokens/s on 1 GB300 + % of HBM (decode) / bf16 TC (prefill) roofline"
UNIT = "tokens/s"
STAGES = ["boundary", "router_topk", "permute", "gate_up", "down", "combine"]
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

WORKLOADS = ["toy", "decode_t1", "decode_t64", "prefill_t2048", "prefill_t16384"]
HEADLINE = "prefill_t16384"
# timed steps and seeded input batches per workload (a few seconds of GPU time each)
DEFAULT_STEPS = {"toy": 200, "decode_t1": 500, "decode_t64": 100, "prefill_t2048": 50, "prefill_t16384": 20}
DEFAULT_BATCHES = {"toy": 16, "decode_t1": 16, "decode_t64": 16, "prefill_t2048": 4, "prefill_t16384": 2}
# tokens whose layer output the oracle computes in the parity report (None: all)
PARITY_Y_TOKENS = {"toy": None, "decode_t1": None, "decode_t64": 4, "prefill_t2048": 4, "prefill_t16384": 4}
# NVFP4 experts: timed at the decode workloads after their bf16 runs (same
# weights, quantized on the device); FP32 scales of the two quantized activations
NVFP4_WORKLOADS = ["decode_t1", "decode_t64"]
NVFP4_G_IN = 2.0 ** -6
NVFP4_G_ACT = 2.0 ** -6
# the benchmark spec tolerances, also asserted by the GPU parity tests
TOL = {"h_ulp": 1, "logits_rel": 1e-5, "y_max_abs": 2e-2, "y_rel_l2": 5e-3, "near_tie_margin": 1e-5}


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None, help="timed steps of every workload (default: per workload)")
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", default="all", choices=["all"] + sorted(CONFIGS),
                   help="one workload instead of all five (it is then the headline)")
    p.add_argument("--batches", type=int, default=None, help="seeded input batches to rotate over")
    p.add_argument("--num-experts", type=int, default=None,
                   help="override E of a single --config (same per-expert shapes; small-footprint profiling)")
    p.add_argument("--tokens", type=int, default=None, help="override T of a single --config")
    p.add_argument("--d-ff", type=int, default=None, help="override d_ff of a single --config")
    p.add_argument("--l2-flush", choices=["write-read", "write"], default="write-read",
                   help="before every step: overwrite a 512 MB buffer, then (write-read) read it back so the "
                        "overwrite's dirty lines are written back before the step rather than inside it")
    p.add_argument("--moe-shape", choices=["tp8", "ep8"], default=None,
                   help="instead of the layer: time the permutation and expert stage at one GPU's share of the "
                        "layer sharded over 8 GPUs (tp8: 256 experts with d_ff 320; ep8: 32 whole experts, "
                        "routing over 256), for --tokens tokens (default 1)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-graph", action="store_true", help="time direct launches only (no CUDA-graph pass)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-parity", action="store_true", help="skip the oracle parity report")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the timed oracle sample")
    p.add_argument("--no-nvfp4", action="store_true", help="skip the NVFP4-experts runs of the decode workloads")
    p.add_argument("--nvfp4", action="store_true",
                   help="with a single --config: time the layer with NVFP4 experts instead of bf16")
    args = p.parse_args(argv)
    overrides = (args.num_experts, args.tokens, args.d_ff)
    if args.config == "all" and any(v is not None for v in overrides) and args.moe_shape is None:
        p.error("--num-experts/--tokens/--d-ff need a single --config")
    if args.config != "all":
        name = args.config
        if args.num_experts is not None:
            CONFIGS[name] = CONFIGS[name].with_(E=args.num_experts)
        if args.tokens is not None:
            CONFIGS[name] = CONFIGS[name].with_(T=args.tokens)
        if args.d_ff is not None:
            CONFIGS[name] = CONFIGS[name].with_(F=args.d_ff)
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    return args


def workloads(args):
    """(runs in order, headline run). A run is (workload name, nvfp4)."""
    if args.config == "all":
        runs = [(n, False) for n in WORKLOADS]
        if not args.no_nvfp4:
            runs += [(n, True) for n in NVFP4_WORKLOADS]
        return runs, (HEADLINE, False)
    return [(args.config, args.nvfp4)], (args.config, args.nvfp4)


def run_key(run) -> str:
    name, fp4 = run
    return f"{name}_nvfp4" if fp4 else name


def steps_for(args, name: str) -> int:
    if args.steps is not None:
        return args.steps
    return DEFAULT_STEPS.get(name, 500 if CONFIGS[name].T <= 64 else 20)


def batches_for(args, name: str) -> int:
    if args.batches is not None:
        return max(1, args.batches)
    return DEFAULT_BATCHES.get(name, 16 if CONFIGS[name].T <= 64 else 2)


# ---------------------------------------------------------------- multi-process helpers
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def whole_job(tokens_per_rank: int, world: int, rank_seconds: list) -> tuple:
    """Weak scaling: every rank processes its own tokens; the job takes as
    long as its slowest rank. Returns (tokens/s, slowest seconds)."""
    slowest = max(rank_seconds)
    return tokens_per_rank * world / slowest, slowest


def reduce_max(value: float, device) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clock, power and throttle reasons with nvidia-smi while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str, period_ms: int = 50):
        self.gpu_id, self.period = gpu_id, period_ms
        self.lines, self.proc, self.thread = [], None, None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", self.gpu_id, "-lms", str(self.period)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_id_for(device_index: int) -> str:
    import torch
    try:
        u = str(torch.cuda.get_device_properties(device_index).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        if vis:
            return vis.split(",")[device_index]
        return str(device_index)


# ---------------------------------------------------------------- peaks and traffic
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


KERNEL_SOURCES = ["experts.cu", "ptx.cuh", "common.cuh", "kernels.h"]


def kernel_source_digest() -> str:
    """sha256 over the sources that define the expert GEMM kernels."""
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "routed_expert_layer_post_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary of this kernel and
    workload, or None when there is none or it was captured from other
    kernel sources (its `source_sha256` line must match the current build)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    fields = {}
    for line in text.splitlines():
        line = line.strip().strip("`")
        if ":" in line:
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip().split()[0] if v.strip() else ""
    if fields.get("source_sha256") != kernel_source_digest():
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None




# ---------------------------------------------------------------- inputs on the device
class DeviceWeights:
    """Expert weights of the current shape, drawn on the device once and kept
    while workloads of the same shape run (20 GB at Beam shapes)."""

    def __init__(self, device):
        self.device, self.key, self.w, self.fp4 = device, None, None, None

    def get(self, cfg):
        import torch
        key = (cfg.seed, cfg.E, cfg.F, cfg.H)
        if key != self.key:
            self.w = None
            torch.cuda.empty_cache()
            # bf16 N(0, 1/sqrt(fan_in)) drawn on the device with a seeded generator
            gen = torch.Generator(device=self.device)
            gen.manual_seed(1000 + cfg.seed)
            E, F, H = cfg.E, cfg.F, cfg.H
            w_gu = torch.empty(E, 2 * F, H, dtype=torch.bfloat16, device=self.device)
            w_d = torch.empty(E, H, F, dtype=torch.bfloat16, device=self.device)
            for e in range(E):
                w_gu[e].copy_(torch.randn(2 * F, H, device=self.device, generator=gen) / H ** 0.5)
                w_d[e].copy_(torch.randn(H, F, device=self.device, generator=gen) / F ** 0.5)
            self.key, self.w, self.fp4 = key, (w_gu, w_d), None
        return self.w

    def nvfp4(self, cfg, beam):
        """The current weights quantized to NVFP4 on the device (once per weight set)."""
        w_gu, w_d = self.get(cfg)
        if getattr(self, "fp4", None) is None:
            mc = beam.make_config(cfg.H, cfg.E, cfg.G, cfg.TG, cfg.K, cfg.F)
            self.fp4 = beam.beam_nvfp4_quantize_experts(w_gu, w_d, mc)
        return self.fp4


def device_activations(cfg, B: int, device):
    """B seeded batches of (h, x), bf16 [T][H], drawn on the device with the
    workload's recipe: N(0, 1) rows, plus the shared direction where the
    workload has one."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(3000 + cfg.seed)
    u = shared_direction(cfg)
    ud = torch.from_numpy(u).to(device) if u is not None else None
    hs, xs = [], []
    for _ in range(B):
        h = torch.randn(cfg.T, cfg.H, device=device, generator=gen)
        x = torch.randn(cfg.T, cfg.H, device=device, generator=gen)
        if ud is not None:
            h += ud
            x += ud
        hs.append(h.to(torch.bfloat16))
        xs.append(x.to(torch.bfloat16))
    return hs, xs


def host_bits(t) -> np.ndarray:
    """A bf16 tensor's bit patterns as a host uint16 array."""
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


# ---------------------------------------------------------------- rooflines
def layer_floor(cfg, touched: float, peaks, fp4: bool = False) -> dict:
    """The layer's roofline: algorithmic bytes (touched expert weights, router
    weight and bias, h and x read, h' and y written, z once) over the HBM peak,
    against the expert FLOPs over the bf16 tensor peak (for NVFP4 experts the
    weights are codes plus scales and the FLOPs run at the FP4 rate, 4x bf16)."""
    T, H, F, E, K = cfg.T, cfg.H, cfg.F, cfg.E, cfg.K
    per_expert = (3 * F * H // 2 + 3 * F * H // 16) if fp4 else 3 * F * H * 2
    bytes_ = touched * per_expert + E * H * 4 + E * 4 + 5 * T * H * 2
    flops = 2.0 * T * K * 3 * H * F
    t_hbm = bytes_ / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (peaks["bf16_tflops"] * 1e12 * (4 if fp4 else 1))
    return {"bound": "hbm" if t_hbm >= t_tc else "tensor", "algorithmic_bytes": bytes_, "expert_flops": flops,
            "floor_us": 1e6 * max(t_hbm, t_tc)}


# ---------------------------------------------------------------- one workload on the GPU
def measure(run, args, env, world):
    """Times one workload (bf16 or NVFP4 experts); returns (report dict,
    capture of batch 0 for the parity check)."""
    import torch
    name, fp4 = run
    lib, beam, device = env["lib"], env["beam"], env["device"]
    cfg = CONFIGS[name]
    T, H, E, F = cfg.T, cfg.H, cfg.E, cfg.F
    mc = beam.make_config(H, E, cfg.G, cfg.TG, cfg.K, F, cfg.routed_scale, cfg.eps)
    w_gu, w_d = env["weights"].get(cfg)

    def bf(a):
        return torch.from_numpy(a.view(np.int16)).to(device).view(torch.bfloat16)

    wp, wq = make_norm_weights(cfg)
    W_r, bias = make_router(cfg)
    tens = dict(w_post=bf(wp), w_pre=bf(wq), router_w=torch.from_numpy(W_r).to(device),
                bias=torch.from_numpy(bias).to(device), w_gate_up=w_gu, w_down=w_d)
    if fp4:
        ex = env["weights"].nvfp4(cfg, beam)
        weights = beam.nvfp4_weights_struct(tens["w_post"], tens["w_pre"], tens["router_w"], tens["bias"], ex,
                                            NVFP4_G_IN, NVFP4_G_ACT)
        layer_fn, ws_fn = lib.beam_moe_layer_nvfp4, lib.beam_moe_nvfp4_workspace_size
    else:
        weights = beam.weights_struct(**tens)
        layer_fn, ws_fn = lib.beam_moe_layer, lib.beam_moe_workspace_size

    B = batches_for(args, name)
    K, W = steps_for(args, name), args.warmup
    K2 = min(K, 200)
    hs, xs = device_activations(cfg, B, device)
    hs_host = [h.cpu().pin_memory() for h in hs] if not args.no_e2e else []
    xs_host = [x.cpu().pin_memory() for x in xs] if not args.no_e2e else []
    h_out = torch.empty(T, H, dtype=torch.bfloat16, device=device)
    y_out = torch.empty(T, H, dtype=torch.bfloat16, device=device)
    offs = torch.empty(E + 1, dtype=torch.int32, device=device)
    ws_bytes = ws_fn(ctypes.byref(mc), T)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
    flush_l2 = env["flush_l2"]
    stream = torch.cuda.current_stream(device)
    sp = stream.cuda_stream

    def make_dbg(slots):
        evs = [torch.cuda.Event(enable_timing=True) if i in slots else None for i in range(7)]
        d = beam.MoeDebug()
        d.expert_offsets = offs.data_ptr()
        for i, ev in enumerate(evs):
            if ev is not None:
                ev.record(stream)      # materialise the handle
                d.stage_events[i] = ev.cuda_event
        return evs, d

    # direct-launch pass: events only at the start and end of each step, so the
    # kernels inside a step keep their programmatic-dependent-launch overlap
    main = [make_dbg({0, 6}) for _ in range(K)]
    # kernel pass: an event at every stage boundary (per-kernel durations)
    stages = [make_dbg(set(range(7))) for _ in range(K2)]
    dbg_plain = beam.MoeDebug()
    dbg_plain.expert_offsets = offs.data_ptr()
    torch.cuda.synchronize()

    def step(i, dbg):
        b = i % B
        st = layer_fn(hs[b].data_ptr(), xs[b].data_ptr(), cfg.n, ctypes.byref(weights), T, ctypes.byref(mc),
                      h_out.data_ptr(), y_out.data_ptr(), ctypes.byref(dbg), ws.data_ptr(), ws_bytes, sp)
        if st != 0:
            raise RuntimeError(f"layer ({run_key(run)}): {beam.beam_status_string(st)}")

    # warm-up; also records how many experts each batch touches
    touched = []
    for i in range(max(W, B)):
        flush_l2()
        step(i, dbg_plain)
        if i < B:
            touched.append(int((torch.diff(offs) > 0).sum().item()))
    launches_per_step = lib.beam_last_launch_count()
    torch.cuda.synchronize()
    if lib.beam_get_device_error(ctypes.byref(ctypes.c_int(0)), ctypes.c_void_p(sp)) != 0:
        raise RuntimeError(f"device wait timed out during warm-up ({name})")

    # graph pass: each seeded batch's whole layer captured once as a CUDA
    # graph; every step replays one, bracketed by events on the replay stream
    graphs = []
    if not args.no_graph:
        gstream = torch.cuda.Stream(device)
        for b in range(B):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=gstream):
                st = layer_fn(hs[b].data_ptr(), xs[b].data_ptr(), cfg.n, ctypes.byref(weights), T,
                              ctypes.byref(mc), h_out.data_ptr(), y_out.data_ptr(), None, ws.data_ptr(), ws_bytes,
                              gstream.cuda_stream)
            if st != 0:
                raise RuntimeError(f"layer (capture, {run_key(run)}): {beam.beam_status_string(st)}")
            graphs.append(g)
        for i in range(W):
            flush_l2()
            graphs[i % B].replay()
        torch.cuda.synchronize()
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]

    def replay(i, flush_mode=args.l2_flush):
        if flush_mode is not None:
            flush_l2(flush_mode)
        gev[i][0].record(stream)
        graphs[i % B].replay()
        gev[i][1].record(stream)

    barrier()
    torch.cuda.synchronize()
    with ClockSampler(gpu_id_for(device.index)) as clocks:
        for i in range(K):
            flush_l2()
            step(i, main[i][1])
        torch.cuda.synchronize()
        for i in range(K if graphs else 0):
            replay(i)
        torch.cuda.synchronize()
    graph_ms = [gev[i][0].elapsed_time(gev[i][1]) for i in range(K)] if graphs else []
    warm_ms, other_ms = [], []
    if graphs:
        for i in range(K2):
            replay(i, flush_mode=None)
        torch.cuda.synchronize()
        warm_ms = [gev[i][0].elapsed_time(gev[i][1]) for i in range(K2)]
        # the same replays after a write-only flush (L2 left full of dirty lines)
        other = "write" if args.l2_flush == "write-read" else "write-read"
        for i in range(K2):
            replay(i, flush_mode=other)
        torch.cuda.synchronize()
        other_ms = [gev[i][0].elapsed_time(gev[i][1]) for i in range(K2)]
    next_boundary = deferred_combine_report(K, lib, beam, cfg, mc, weights, tens, hs, xs, ws, ws_bytes, B,
                                            flush_l2, device) if graphs and not fp4 else None
    del graphs
    barrier()
    for i in range(K2):
        flush_l2()
        step(i, stages[i][1])
    torch.cuda.synchronize()
    if lib.beam_get_device_error(ctypes.byref(ctypes.c_int(0)), ctypes.c_void_p(sp)) != 0:
        raise RuntimeError(f"device wait timed out during the timed passes ({name})")

    step_ms = [main[i][0][0].elapsed_time(main[i][0][6]) for i in range(K)]
    stage_ms = {s: [stages[i][0][j].elapsed_time(stages[i][0][j + 1]) for i in range(K2)]
                for j, s in enumerate(STAGES)}
    staged_step_ms = [stages[i][0][0].elapsed_time(stages[i][0][6]) for i in range(K2)]
    direct_s = reduce_max(sum(step_ms) / 1e3, device)
    direct_value, direct_s = whole_job(T * K, world, [direct_s])
    # primary number: graph replays when captured, else the direct launches
    total_s = sum(graph_ms if graph_ms else step_ms) / 1e3
    slowest = reduce_max(total_s, device)
    value, slowest = whole_job(T * K, world, [slowest])
    us_per_layer = 1e3 * statistics.fmean(graph_ms if graph_ms else step_ms)

    # roofline of the dominant kernel (by mean time)
    peaks, peaks_kind = load_peaks()
    mean_stage = {s: statistics.fmean(v) for s, v in stage_ms.items()}
    rows = T * cfg.K
    touched_per_step = [touched[i % B] for i in range(K2)]
    long_step = statistics.fmean(staged_step_ms) > 1.0
    # a contraction timed inside a step of more than a millisecond runs at the
    # power-capped (sustained) rate, so it is measured against that peak
    tc_key = "bf16_tflops_sustained" if long_step and "bf16_tflops_sustained" in peaks else "bf16_tflops"
    tc_kind = f"{peaks_kind} {'sustained' if tc_key.endswith('sustained') else 'burst'}"
    # When both expert GEMMs share one launch the library records the launch
    # as the gate/up stage and the down stage is empty: the dominant kernel is
    # then the fused one and its algorithmic bytes cover both weight sets.
    fused = mean_stage["down"] < 0.05 * mean_stage["gate_up"]
    if fp4:
        # NVFP4: codes (half a byte per weight) plus one E4M3 scale per 16
        # weights; the input and SwiGLU rows as codes and scale slots, y_perm bf16
        dom = "experts_fused_nvfp4"
        w_bytes = 3 * F * H // 2 + 3 * F * H // 16
        act_bytes = rows * (H // 2 + H // 4) + 2 * rows * (F // 2 + F // 4) + rows * H * 2
        flops = 2.0 * rows * 3 * F * H
    elif fused:
        dom = "experts_fused"
        w_bytes = 3 * F * H * 2
        act_bytes = rows * H * 2 + 2 * rows * F * 2 + rows * H * 2
        flops = 2.0 * rows * 3 * F * H
    else:
        dom = max(("gate_up", "down"), key=lambda s: mean_stage[s])
        if dom == "gate_up":
            w_bytes = 2 * F * H * 2
            act_bytes = rows * H * 2 + rows * F * 2
            flops = 2.0 * rows * 2 * F * H
        else:
            w_bytes = H * F * 2
            act_bytes = rows * F * 2 + rows * H * 2
            flops = 2.0 * rows * H * F
    bytes_total = sum(tc * w_bytes + act_bytes for tc in touched_per_step)
    dom_stage = "gate_up" if (fused or fp4) else dom
    dom_s = sum(stage_ms[dom_stage]) / 1e3
    t_hbm = bytes_total / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops * K2 / (peaks["bf16_tflops"] * 1e12)
    if t_hbm >= t_tc:
        achieved = bytes_total / dom_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "peak_source": peaks_kind}
    else:
        achieved = flops * K2 / dom_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks[tc_key], "unit": "TFLOP/s",
                "frac": achieved / peaks[tc_key], "peak_source": tc_kind}
    roof.update({"traffic": profiled_traffic(dom, cfg.name), "kernel": dom,
                 "algorithmic_bytes_per_launch": bytes_total / K2,
                 "launch_us": 1e3 * statistics.fmean(stage_ms[dom_stage]),
                 "timing": f"CUDA events around the kernel on its stream, {K2} steps of a second pass with an event "
                           "at every stage boundary"})
    # both expert GEMMs against the tensor peak, the layer against its roofline
    gemm_s = (sum(stage_ms["gate_up"]) + sum(stage_ms["down"])) / 1e3 / K2
    expert_flops = 2.0 * rows * 3 * F * H
    expert_gemms = {"us": 1e6 * gemm_s, "tflops": expert_flops / gemm_s / 1e12, "peak": peaks[tc_key],
                    "peak_source": tc_kind, "frac_of_bf16_peak": expert_flops / gemm_s / 1e12 / peaks[tc_key]}
    floor = layer_floor(cfg, statistics.fmean(touched_per_step), peaks, fp4)
    floor["frac"] = floor["floor_us"] / us_per_layer
    floor["peak_source"] = peaks_kind

    # end to end through the host-buffer entry point: H2D of h, x and D2H of h', y inside the timed region
    e2e = None
    host_fn = lib.beam_moe_layer_nvfp4_host if fp4 else lib.beam_moe_layer_host
    host_name = "beam_moe_layer_nvfp4_host" if fp4 else "beam_moe_layer_host"
    if not args.no_e2e:
        hbytes = (lib.beam_moe_layer_nvfp4_host_workspace_size if fp4 else
                  lib.beam_moe_layer_host_workspace_size)(ctypes.byref(mc), T)
        ws_h = torch.empty(hbytes, dtype=torch.uint8, device=device)
        ho = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()
        yo = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()
        # a serving loop's staging buffers: each step's batch is written into
        # the same page-locked h and x (host to host, before the timed call)
        hi = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()
        xi = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()
        Ke = K2
        tot = 0.0
        for i in range(Ke + 3):
            b = i % B
            hi.copy_(hs_host[b])
            xi.copy_(xs_host[b])
            flush_l2()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            st = host_fn(hi.data_ptr(), xi.data_ptr(), cfg.n, ctypes.byref(weights), T, ctypes.byref(mc),
                         ho.data_ptr(), yo.data_ptr(), ws_h.data_ptr(), hbytes, sp)
            dt = time.perf_counter() - t0
            if st != 0:
                raise RuntimeError(f"{host_name} ({name}): {beam.beam_status_string(st)}")
            if i >= 3:
                tot += dt
        tot = reduce_max(tot, device)
        e2e = {"value": T * Ke * world / tot, "unit": UNIT, "h2d_bytes_per_step": 2 * T * H * 2,
               "d2h_bytes_per_step": 2 * T * H * 2, "steps": Ke, "us_per_layer": 1e6 * tot / Ke,
               "timing": f"host clock around {host_name} (returns after a stream synchronise); the same "
                         "page-locked h, x, h', y buffers every step, refilled with the step's batch before the "
                         "timed call"}
        del ws_h

    # batch 0 once more with every debug output, for the parity check
    dbg = {"logits": torch.empty(T, E, dtype=torch.float32, device=device),
           "topk_ids": torch.empty(T, cfg.K, dtype=torch.int32, device=device)}
    d = beam.MoeDebug()
    d.logits = dbg["logits"].data_ptr()
    d.topk_ids = dbg["topk_ids"].data_ptr()
    step(0, d)
    torch.cuda.synchronize()
    capture = {"h": host_bits(hs[0]), "x": host_bits(xs[0]), "h_out": host_bits(h_out), "y": host_bits(y_out),
               "logits": dbg["logits"].cpu().numpy(), "ids": dbg["topk_ids"].cpu().numpy(),
               "wp": wp, "wq": wq, "W_r": W_r, "bias": bias, "w_gu": w_gu, "w_d": w_d}

    capture["nvfp4"] = fp4
    report = {"workload": name, "experts": "nvfp4" if fp4 else "bf16", "T": T, "tokens_per_s": value,
              "us_per_layer": us_per_layer,
              "ms_per_step": 1e3 * slowest / K, "steps": K, "warmup": W, "batches": B,
              "timing": ("CUDA-graph replay of the whole layer per step (one graph per seeded batch), events "
                         "on the replay stream" if graph_ms else "direct launches, events on the launch stream"),
              "direct_launch": {"value": direct_value, "unit": UNIT, "us_per_layer": 1e3 * statistics.fmean(step_ms)},
              "graph_warm_l2_us_per_layer": 1e3 * statistics.fmean(warm_ms) if warm_ms else None,
              f"graph_{'write_only' if args.l2_flush == 'write-read' else 'write_read'}_flush_us_per_layer":
                  1e3 * statistics.fmean(other_ms) if other_ms else None,
              "stage_us": stage_report(stage_ms, routing_fused(cfg, T)),
              "us_per_layer_with_stage_events": 1e3 * statistics.fmean(staged_step_ms),
              "next_boundary": next_boundary,
              "touched_experts_mean": statistics.fmean(touched_per_step),
              "roofline": roof, "layer_roofline": floor, "expert_gemms": expert_gemms, "e2e": e2e,
              "gpu_launches_per_step": launches_per_step, "gpu_launches": launches_per_step * K,
              "clocks": clocks.summary()}
    return report, capture


# ---------------------------------------------------------------- parity against the oracle
def expert_reader(w_gu, w_d, F: int):
    """expert_fn for the oracle: expert e's bf16 bits copied from the device
    weights, decoded to float64 by the oracle's own reader."""
    from oracle.experts import decoded_expert

    def fn(e):
        gu = host_bits(w_gu[e])[None]
        d = host_bits(w_d[e])[None]
        return decoded_expert(gu, d, 0, F)
    return fn


def parity_report(name, cap, timed_seconds=None, workers=None):
    """Batch 0 of a workload against the fp64 oracle.

    Routing, logits and h' are compared on every token (the workload's seeded
    oracle sample where it has one), the layer output y on a few of them.
    With ``timed_seconds`` the y tokens are evaluated one at a time, each
    call timed, until that much CPU time has passed (the CPU baseline).
    Returns (report, timing or None)."""
    from oracle import bf16 as obf
    from oracle.boundary import boundary
    from oracle.layer import layer
    from oracle.routing import near_tie, route, router_logits
    cfg = CONFIGS[name]
    workers = workers or max(1, len(os.sched_getaffinity(0)))
    tokens = sample_tokens(cfg)
    h64, x64 = obf.decode(cap["h"][tokens]), obf.decode(cap["x"][tokens])
    wp64, wq64 = obf.decode(cap["wp"]), obf.decode(cap["wq"])
    h_new, z, _ = boundary(h64, x64, wp64, wq64, cfg.n, cfg.eps)
    L = router_logits(z, cap["W_r"])
    r = route(L, cap["bias"], cfg.G, cfg.TG, cfg.K, cfg.routed_scale)
    tie = near_tie(r, TOL["near_tie_margin"])
    gids = cap["ids"][tokens]
    same = np.all(gids == r["ids"], axis=1)
    h_ulp = int(obf.ulp_distance(cap["h_out"][tokens], obf.encode(h_new)).max())
    Lg = cap["logits"][tokens].astype(np.float64)
    logit_rel = float(np.max(np.abs(Lg - L).max(axis=1) / np.maximum(np.abs(L).max(axis=1), 1e-300)))

    # layer output on the first few tokens of the sample (one token with NVFP4
    # experts, whose oracle quantizes each touched expert on the host first)
    fp4 = cap.get("nvfp4", False)
    ny = 1 if fp4 else PARITY_Y_TOKENS.get(name)
    ysel = tokens if ny is None else tokens[:ny]
    efn = expert_reader(cap["w_gu"], cap["w_d"], cfg.F)
    common = dict(n=cfg.n, eps=cfg.eps, G=cfg.G, TG=cfg.TG, K=cfg.K, routed_scale=cfg.routed_scale,
                  workers=workers)
    if fp4:
        from oracle import nvfp4 as onv

        def ffn(e, X):
            Wg, Wu, Wd = efn(e)
            ex = onv.Nvfp4Expert(Wg.astype(np.float32), Wu.astype(np.float32), Wd.astype(np.float32))
            return onv.ffn(X, ex, NVFP4_G_IN, NVFP4_G_ACT)
        common["ffn"] = ffn
    else:
        common["expert_fn"] = efn
    args_l = (obf.decode(cap["h"]), obf.decode(cap["x"]), wp64, wq64, cap["W_r"], cap["bias"])
    timing = None
    if timed_seconds is None:
        ref = layer(*args_l, tokens=ysel, **common)
        y_ref, y_ids = ref["y"], ref["ids"]
    else:
        # the CPU baseline: the oracle as it stands, one token per call, its
        # experts read from the weights and decoded to fp64 on every call
        ys, idl, el, done = [], [], 0.0, 0
        for t in tokens:
            t0 = time.perf_counter()
            ref = layer(*args_l, tokens=np.array([t]), **common)
            el += time.perf_counter() - t0
            ys.append(ref["y"][0])
            idl.append(ref["ids"][0])
            done += 1
            if el >= timed_seconds:
                break
        ysel = tokens[:done]
        y_ref, y_ids = np.array(ys), np.array(idl)
        timing = {"tokens": done, "seconds": el, "workers": workers}
    yg = obf.decode(cap["y"][ysel])
    ysame = np.all(cap["ids"][ysel] == y_ids, axis=1)
    diff = yg[ysame] - y_ref[ysame]
    y_max = float(np.abs(diff).max()) if diff.size else 0.0
    y_rel = float(np.linalg.norm(diff) / max(np.linalg.norm(y_ref[ysame]), 1e-300)) if diff.size else 0.0
    cond = None
    if (~ysame).any():
        # routing-conditioned check: the oracle evaluated with the GPU's choices
        c = layer(*args_l, tokens=ysel[~ysame], ids_override=cap["ids"][ysel[~ysame]], **common)
        dc = yg[~ysame] - c["y"]
        cond = {"tokens": int((~ysame).sum()), "max_abs": float(np.abs(dc).max()),
                "rel_l2": float(np.linalg.norm(dc) / max(np.linalg.norm(c["y"]), 1e-300))}
    ok = (int((~same & ~tie).sum()) == 0 and h_ulp <= TOL["h_ulp"] and logit_rel <= TOL["logits_rel"]
          and y_max <= TOL["y_max_abs"] and y_rel <= TOL["y_rel_l2"]
          and (cond is None or (cond["max_abs"] <= TOL["y_max_abs"] and cond["rel_l2"] <= TOL["y_rel_l2"])))
    rep = {"routing_tokens": int(tokens.size), "near_ties": int(tie.sum()),
           "differing_rows": int((~same).sum()), "differing_non_near_tie": int((~same & ~tie).sum()),
           "h_worst_ulp": h_ulp, "logits_max_rel": logit_rel, "y_tokens": int(ysel.size),
           "y_max_abs": y_max, "y_rel_l2": y_rel, "y_routing_conditioned": cond, "pass": bool(ok)}
    return rep, timing


# ---------------------------------------------------------------- the reference arm
def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    _, (headline, _) = workloads(args)
    cfg = CONFIGS[headline]
    from beam_inputs import expert_weights, make_activations
    from oracle import bf16 as obf
    from oracle.layer import layer
    workers = max(1, len(os.sched_getaffinity(0)))
    wp, wq = make_norm_weights(cfg)
    W_r, bias = make_router(cfg)
    cache = {}

    def expert_fn(e):
        if e not in cache:
            cache[e] = tuple(obf.decode(m) for m in expert_weights(cfg, e))
        return cache[e]

    h, x = make_activations(cfg.with_(T=1), batch=0)
    args_l = (obf.decode(h), obf.decode(x), obf.decode(wp), obf.decode(wq), W_r, bias)
    kw = dict(n=cfg.n, eps=cfg.eps, G=cfg.G, TG=cfg.TG, K=cfg.K, routed_scale=cfg.routed_scale,
              expert_fn=expert_fn, workers=workers)
    steps = args.steps if args.steps is not None else 20
    for _ in range(args.warmup):
        layer(*args_l, **kw)
    t0 = time.perf_counter()
    for _ in range(steps):
        layer(*args_l, **kw)
    el = time.perf_counter() - t0
    value = steps / el
    sample = (f"1 token of {cfg.name} per step (a seed-0 token of that workload's recipe, its 8 experts decoded "
              f"to fp64 once and reused), fp64 numpy oracle, {workers} worker threads")
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 0, "steps": steps,
           "warmup": args.warmup, "ms_per_step": 1e3 * el / steps, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": config_block(cfg, world=1, l2=None),
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": workers, "kind": "oracle", "sample": sample},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)
    return 0


def config_block(cfg, world: int, l2) -> dict:
    c = {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "E": cfg.E, "G": cfg.G, "TG": cfg.TG, "K": cfg.K,
         "F": cfg.F, "n": cfg.n, "parallelism": f"replicas x{world}",
         "weights": "expert weights bf16 N(0, 1/sqrt(fan_in)) drawn on the device; router, norms and bias from "
                    "beam_inputs; activations N(0, 1) (plus the workload's shared direction) drawn on the device"}
    if l2 is not None:
        c["l2"] = l2
    return c


# ---------------------------------------------------------------- our implementation
def run_ours(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)

    import routed_expert_layer_post_gb300 as beam
    from routed_expert_layer_post_gb300 import build as beam_build
    beam_build.build()
    lib = beam.library()

    flush = torch.empty(512 << 20, dtype=torch.uint8, device=device)
    flush_words = flush.view(torch.int64)

    def flush_l2(mode=args.l2_flush):
        # The overwrite (4x L2) evicts every line of the previous step but
        # leaves L2 full of dirty lines; reading the buffer back writes those
        # back first, so the step starts from a cold, clean L2.
        flush.zero_()
        if mode == "write-read":
            flush_words.sum()

    env = {"lib": lib, "beam": beam, "device": device, "flush_l2": flush_l2, "weights": DeviceWeights(device)}
    runs, head_run = workloads(args)
    reports, captures = {}, {}
    for run in runs:
        key = run_key(run)
        reports[key], captures[key] = measure(run, args, env, world)
        torch.cuda.empty_cache()

    # parity against the oracle (and the timed oracle sample) on rank 0 of a 1-GPU run
    cpu = None
    if rank == 0 and world == 1 and not args.no_parity:
        for run in runs:
            key, name = run_key(run), run[0]
            timed = (not args.no_cpu_baseline) and run == head_run
            rep, timing = parity_report(name, captures[key], timed_seconds=args.cpu_seconds if timed else None)
            reports[key]["parity"] = rep
            if timing is not None:
                cpu = {"value": timing["tokens"] / timing["seconds"], "unit": UNIT, "cores": timing["workers"],
                       "kind": "oracle",
                       "sample": f"{timing['tokens']} tokens of {name} (its seeded oracle sample, one token per "
                                 f"call, each call's experts read from the bf16 weights and decoded to fp64), fp64 "
                                 f"numpy oracle, {timing['workers']} worker threads, {timing['seconds']:.1f} s"}
    captures.clear()

    if rank == 0:
        headline = head_run[0]
        head = reports[run_key(head_run)]
        cfg = CONFIGS[headline]
        B = batches_for(args, headline)
        l2 = ("512 MB buffer overwritten " + ("and read back " if args.l2_flush == "write-read" else "")
              + f"before every step (outside the timed events); inputs rotate over {B} seeded batches")
        out = {"metric": METRIC, "value": head["tokens_per_s"], "unit": UNIT, "n_gpus": world,
               "steps": head["steps"], "warmup": head["warmup"], "ms_per_step": head["ms_per_step"],
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
               "data": "synthetic", "config": config_block(cfg, world, l2), "timing": head["timing"],
               "us_per_layer": head["us_per_layer"], "roofline": head["roofline"],
               "layer_roofline": head["layer_roofline"], "expert_gemms": head["expert_gemms"],
               "cpu_baseline": cpu, "e2e": head["e2e"], "gpu_launches": head["gpu_launches"],
               "clocks": head["clocks"],
               "parity": {k: reports[k].get("parity") for k in reports},
               "parity_tolerances": TOL,
               "per_config": reports}
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def deferred_combine_report(steps, lib, beam, cfg, mc, weights, tens, hs, xs, ws, ws_bytes, B, flush_l2, device):
    """Decode sizes: the step followed by the next sublayer's boundary, timed
    as CUDA-graph replays two ways -- the combine as its own kernel
    (beam_moe_layer, beam_boundary_norm) and the combine fused into that
    boundary (beam_moe_layer_uncombined, beam_boundary_norm_combine)."""
    import torch
    T, H = cfg.T, cfg.H
    if T > 64:
        return None
    Kr = min(steps, 200)
    h1 = torch.empty(T, H, dtype=torch.bfloat16, device=device)
    y = torch.empty(T, H, dtype=torch.bfloat16, device=device)
    h2 = torch.empty(T, H, dtype=torch.bfloat16, device=device)
    z2 = torch.empty(T, H, dtype=torch.bfloat16, device=device)
    wp, wq = tens["w_post"].data_ptr(), tens["w_pre"].data_ptr()
    n2 = cfg.n + 1
    gstream = torch.cuda.Stream(device)
    gs = gstream.cuda_stream

    def separate(b):
        st = lib.beam_moe_layer(hs[b].data_ptr(), xs[b].data_ptr(), cfg.n, ctypes.byref(weights), T,
                                ctypes.byref(mc), h1.data_ptr(), y.data_ptr(), None, ws.data_ptr(), ws_bytes, gs)
        st = st or lib.beam_boundary_norm(h1.data_ptr(), y.data_ptr(), wp, wq, T, H, cfg.eps, n2, h2.data_ptr(),
                                          z2.data_ptr(), gs)
        return st

    def fused(b):
        out = beam.MoeUncombined()
        st = lib.beam_moe_layer_uncombined(hs[b].data_ptr(), xs[b].data_ptr(), cfg.n, ctypes.byref(weights), T,
                                           ctypes.byref(mc), h1.data_ptr(), ctypes.byref(out), ws.data_ptr(),
                                           ws_bytes, gs)
        st = st or lib.beam_boundary_norm_combine(h1.data_ptr(), out.y_perm, out.topk_w, out.inv_perm, cfg.K, wp,
                                                  wq, T, H, cfg.eps, n2, h2.data_ptr(), z2.data_ptr(), gs)
        return st

    res = {}
    for name, fn in (("separate", separate), ("fused", fused)):
        graphs = []
        for b in range(B):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=gstream):
                st = fn(b)
            if st != 0:
                raise RuntimeError(f"{name} next-boundary step: {beam.beam_status_string(st)}")
            graphs.append(g)
        stream = torch.cuda.current_stream(device)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(Kr)]
        for i in range(3):
            flush_l2()
            graphs[i % B].replay()
        for i in range(Kr):
            flush_l2()
            evs[i][0].record(stream)
            graphs[i % B].replay()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        res[name] = 1e3 * statistics.fmean(a.elapsed_time(b) for a, b in evs)
        del graphs
    return {"separate_us": round(res["separate"], 2), "fused_us": round(res["fused"], 2),
            "saved_us": round(res["separate"] - res["fused"], 2),
            "timing": f"{Kr} CUDA-graph replays each after the L2 flush: the step plus the next sublayer's "
                      "boundary, with the combine as its own kernel or fused into that boundary"}


def routing_fused(cfg, T):
    """The library's condition for its one-launch decode routing (up to 8
    tokens, 256 experts in 8 groups, at most 64 (token, expert) pairs)."""
    return 1 <= T <= 8 and cfg.E == 256 and cfg.G == 8 and T * cfg.K <= 64 and cfg.H % 256 == 0 and cfg.H <= 5120


def stage_report(stage_ms, fused_routing):
    """Mean microseconds per stage. With the one-launch decode routing the
    library records that launch as the boundary stage and the next two stages
    are empty (two back-to-back events): reported as "routing_fused"."""
    mean = {s: 1e3 * statistics.fmean(v) for s, v in stage_ms.items()}
    if fused_routing:
        mean = {"routing_fused": mean["boundary"], **{s: v for s, v in mean.items()
                                                      if s not in ("boundary", "router_topk", "permute")}}
    return {s: round(v, 2) for s, v in mean.items()}


def run_shard_shape(args):
    """The permutation and the expert stage (gate/up + SwiGLU, down, combine)
    at one GPU's share of a Beam layer sharded over eight GPUs, the shapes on
    which the pages compare MoE kernels: one JSON line, CUDA-graph replays
    after the L2 flush. Routing is drawn over all 256 experts; under EP8 the
    permutation drops the pairs of the other GPUs' experts."""
    import torch
    import routed_expert_layer_post_gb300 as beam
    from routed_expert_layer_post_gb300 import build as beam_build
    from beam_inputs import random_topk_ids
    beam_build.build()
    lib = beam.library()
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    base = CONFIGS["decode_t1"]
    T = args.tokens or 1
    E_route = base.E
    if args.moe_shape == "tp8":
        E, F = base.E, base.F // 8
    else:
        E, F = base.E // 8, base.F
    H, K = base.H, base.K
    mc = beam.make_config(H, E, 8, 4, K, F, base.routed_scale, base.eps)
    gen = torch.Generator(device=device)
    gen.manual_seed(2000)
    w_gu = (torch.randn(E, 2 * F, H, device=device, generator=gen) / H ** 0.5).to(torch.bfloat16)
    w_d = (torch.randn(E, H, F, device=device, generator=gen) / F ** 0.5).to(torch.bfloat16)
    B = args.batches if args.batches is not None else 16
    ids, zs, ws_ = [], [], []
    for b in range(B):
        ids.append(torch.from_numpy(random_topk_ids(T, E_route, K, seed=3000 + b).astype(np.int32)).to(device))
        zs.append((torch.randn(T, H, device=device, generator=gen)).to(torch.bfloat16))
        w = torch.rand(T, K, device=device, generator=gen) + 0.1
        ws_.append((base.routed_scale * w / w.sum(dim=1, keepdim=True)).contiguous())
    rows = T * K
    offs = torch.empty(E + 1, dtype=torch.int32, device=device)
    perm = torch.empty(rows, dtype=torch.int32, device=device)
    inv = torch.empty(rows, dtype=torch.int32, device=device)
    x_perm = torch.empty(rows, H, dtype=torch.bfloat16, device=device)
    y = torch.empty(T, H, dtype=torch.bfloat16, device=device)
    pws = torch.empty(max(256, lib.beam_moe_permute_workspace_size(ctypes.byref(mc), T)), dtype=torch.uint8,
                      device=device)
    ews = torch.empty(max(256, lib.beam_moe_experts_workspace_size(ctypes.byref(mc), T)), dtype=torch.uint8,
                      device=device)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=device)
    gstream = torch.cuda.Stream(device)
    gs = gstream.cuda_stream
    graphs, touched = [], []
    for b in range(B):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=gstream):
            st = lib.beam_moe_permute(ids[b].data_ptr(), zs[b].data_ptr(), T, ctypes.byref(mc), offs.data_ptr(),
                                      perm.data_ptr(), inv.data_ptr(), x_perm.data_ptr(), pws.data_ptr(),
                                      pws.numel(), gs)
            st = st or lib.beam_moe_experts(x_perm.data_ptr(), offs.data_ptr(), w_gu.data_ptr(), w_d.data_ptr(),
                                            ws_[b].data_ptr(), inv.data_ptr(), T, ctypes.byref(mc), y.data_ptr(),
                                            ews.data_ptr(), ews.numel(), gs)
        if st != 0:
            raise RuntimeError(f"shard-shape step: {beam.beam_status_string(st)}")
        graphs.append(g)
        ib = ids[b].cpu().numpy().reshape(-1)
        touched.append(len(np.unique(ib[ib < E])))
    stream = torch.cuda.current_stream(device)
    Kr = args.steps if args.steps is not None else 500
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(Kr)]
    words = flush.view(torch.int64)
    for i in range(args.warmup + Kr):
        flush.zero_()
        words.sum()
        j = i - args.warmup
        if j >= 0:
            evs[j][0].record(stream)
        graphs[i % B].replay()
        if j >= 0:
            evs[j][1].record(stream)
    torch.cuda.synchronize()
    us = [1e3 * a.elapsed_time(b) for a, b in evs]
    mean_us = statistics.fmean(us)
    peaks, peaks_kind = load_peaks()
    bytes_step = statistics.fmean(touched[i % B] for i in range(Kr)) * 3 * F * H * 2 + 2 * rows * H * 2
    achieved = bytes_step / (mean_us * 1e-6) / 1e9
    out = {"metric": f"MoE expert stage at the {args.moe_shape.upper()} per-GPU shape (permutation + gate/up "
                     "+ down + combine)",
           "value": T / (mean_us * 1e-6), "unit": UNIT, "us_per_call": mean_us, "n_gpus": 1, "steps": Kr,
           "warmup": args.warmup, "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
           "config": {"workload": f"{args.moe_shape}_t{T}", "T": T, "H": H, "E_local": E, "E_routed": E_route,
                      "K": K, "F": F, "l2": "512 MB buffer overwritten and read back before every call"},
           "touched_experts_mean": statistics.fmean(touched),
           "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                        "frac": achieved / peaks["hbm_gbs"], "peak_source": peaks_kind,
                        "algorithmic_bytes": bytes_step,
                        "note": "weights of the touched local experts plus the token rows in and out; the "
                                "whole call, so launch and routing-side latency count against it"}}
    print(json.dumps(out), flush=True)
    return 0




def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.moe_shape is not None:
        return run_shard_shape(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
