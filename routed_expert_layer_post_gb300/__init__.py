"""Python binding of libbeam.so, the GB300 (sm_103a) Beam MoE sublayer.

Argument marshalling only: every step runs in the library's CUDA kernels.
Tensors are PyTorch CUDA tensors (PyTorch supplies device memory and the
current stream); the functions carry the C ABI's names and pass raw device
pointers, sizes and ``torch.cuda.current_stream()`` through. There is no CPU
fallback: if libbeam.so is missing or the device is not a GB300, the calls
raise.

See include/beam.h for the layouts, ownership and error behaviour of each
entry point.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

import torch

__all__ = [
    "BeamError", "MoeConfig", "MoeWeights", "MoeDebug", "make_config", "library",
    "beam_boundary_norm", "beam_router_topk", "beam_moe_permute", "beam_moe_experts",
    "beam_moe_gate_up", "beam_moe_down", "beam_moe_combine", "beam_moe_layer",
    "beam_moe_layer_host", "beam_moe_layer_uncombined", "beam_boundary_norm_combine", "MoeUncombined",
    "beam_moe_workspace_size", "beam_moe_permute_workspace_size",
    "beam_moe_experts_workspace_size", "beam_moe_layer_host_workspace_size",
    "beam_get_device_error", "beam_check_bounded_wait", "beam_check_bounded_wait_pending",
    "beam_release_host_graphs", "MoeNvfp4Weights", "MoeNvfp4Intermediates", "Nvfp4Experts",
    "beam_nvfp4_quantize_experts", "beam_nvfp4_quantize_rows", "nvfp4_weights_struct", "beam_moe_experts_nvfp4",
    "beam_moe_layer_nvfp4", "beam_moe_nvfp4_workspace_size", "beam_moe_layer_nvfp4_host",
    "beam_moe_layer_nvfp4_host_workspace_size", "beam_last_launch_count", "beam_status_string", "Workspace",
]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libbeam.so")

c_int, c_float, c_size_t, c_void_p = ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p


class BeamError(RuntimeError):
    pass


class MoeConfig(ctypes.Structure):
    _fields_ = [("hidden", c_int), ("num_experts", c_int), ("num_groups", c_int),
                ("topk_groups", c_int), ("topk", c_int), ("d_ff", c_int),
                ("routed_scale", c_float), ("eps", c_float)]


class MoeWeights(ctypes.Structure):
    _fields_ = [("w_post", c_void_p), ("w_pre", c_void_p), ("router_w", c_void_p),
                ("bias", c_void_p), ("w_gate_up", c_void_p), ("w_down", c_void_p)]


class MoeDebug(ctypes.Structure):
    _fields_ = [("z", c_void_p), ("logits", c_void_p), ("topk_ids", c_void_p),
                ("topk_w", c_void_p), ("expert_offsets", c_void_p), ("stage_events", c_void_p * 7)]


class MoeUncombined(ctypes.Structure):
    _fields_ = [("y_perm", c_void_p), ("topk_w", c_void_p), ("inv_perm", c_void_p)]


class MoeNvfp4Weights(ctypes.Structure):
    _fields_ = [("w_post", c_void_p), ("w_pre", c_void_p), ("router_w", c_void_p), ("bias", c_void_p),
                ("q_gate_up", c_void_p), ("sf_gate_up", c_void_p), ("q_down", c_void_p), ("sf_down", c_void_p),
                ("expert_scale", c_void_p), ("input_scale", c_float), ("act_scale", c_float)]


class MoeNvfp4Intermediates(ctypes.Structure):
    _fields_ = [("x_q", c_void_p), ("x_sf", c_void_p), ("act_q", c_void_p), ("act_sf", c_void_p),
                ("y_perm", c_void_p)]


def make_config(hidden: int, num_experts: int, num_groups: int, topk_groups: int, topk: int,
                d_ff: int, routed_scale: float = 2.5, eps: float = 1e-6) -> MoeConfig:
    return MoeConfig(hidden, num_experts, num_groups, topk_groups, topk, d_ff, routed_scale, eps)


_SIGNATURES = {
    "beam_status_string": (ctypes.c_char_p, [c_int]),
    "beam_version": (ctypes.c_char_p, []),
    "beam_last_launch_count": (c_int, []),
    "beam_boundary_norm": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_int, c_float, c_int,
                                   c_void_p, c_void_p, c_void_p]),
    "beam_router_topk": (c_int, [c_void_p, c_void_p, c_void_p, c_int, ctypes.POINTER(MoeConfig), c_void_p,
                                 c_void_p, c_void_p, c_void_p]),
    "beam_moe_permute_workspace_size": (c_size_t, [ctypes.POINTER(MoeConfig), c_int]),
    "beam_moe_permute": (c_int, [c_void_p, c_void_p, c_int, ctypes.POINTER(MoeConfig), c_void_p, c_void_p,
                                 c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "beam_moe_experts_workspace_size": (c_size_t, [ctypes.POINTER(MoeConfig), c_int]),
    "beam_moe_experts": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int,
                                 ctypes.POINTER(MoeConfig), c_void_p, c_void_p, c_size_t, c_void_p]),
    "beam_moe_gate_up": (c_int, [c_void_p, c_void_p, c_void_p, c_int, ctypes.POINTER(MoeConfig), c_void_p,
                                 c_void_p, c_size_t, c_void_p]),
    "beam_moe_down": (c_int, [c_void_p, c_void_p, c_void_p, c_int, ctypes.POINTER(MoeConfig), c_void_p,
                              c_void_p, c_size_t, c_void_p]),
    "beam_moe_combine": (c_int, [c_void_p, c_void_p, c_void_p, c_int, ctypes.POINTER(MoeConfig), c_void_p,
                                 c_void_p]),
    "beam_moe_workspace_size": (c_size_t, [ctypes.POINTER(MoeConfig), c_int]),
    "beam_moe_layer_uncombined": (c_int, [c_void_p, c_void_p, c_int, ctypes.POINTER(MoeWeights), c_int,
                                          ctypes.POINTER(MoeConfig), c_void_p, ctypes.POINTER(MoeUncombined),
                                          c_void_p, c_size_t, c_void_p]),
    "beam_boundary_norm_combine": (c_int, [c_void_p, c_void_p, c_void_p, c_void_p, c_int, c_void_p, c_void_p,
                                           c_int, c_int, c_float, c_int, c_void_p, c_void_p, c_void_p]),
    "beam_moe_layer": (c_int, [c_void_p, c_void_p, c_int, ctypes.POINTER(MoeWeights), c_int,
                               ctypes.POINTER(MoeConfig), c_void_p, c_void_p, ctypes.POINTER(MoeDebug),
                               c_void_p, c_size_t, c_void_p]),
    "beam_moe_layer_host_workspace_size": (c_size_t, [ctypes.POINTER(MoeConfig), c_int]),
    "beam_moe_layer_host": (c_int, [c_void_p, c_void_p, c_int, ctypes.POINTER(MoeWeights), c_int,
                                    ctypes.POINTER(MoeConfig), c_void_p, c_void_p, c_void_p, c_size_t,
                                    c_void_p]),
    "beam_moe_layer_nvfp4_host_workspace_size": (c_size_t, [ctypes.POINTER(MoeConfig), c_int]),
    "beam_moe_layer_nvfp4_host": (c_int, [c_void_p, c_void_p, c_int, ctypes.POINTER(MoeNvfp4Weights), c_int,
                                          ctypes.POINTER(MoeConfig), c_void_p, c_void_p, c_void_p, c_size_t,
                                          c_void_p]),
    "beam_get_device_error": (c_int, [ctypes.POINTER(c_int), c_void_p]),
    "beam_check_bounded_wait": (c_int, [c_void_p, c_int, ctypes.POINTER(c_int), c_void_p]),
    "beam_check_bounded_wait_pending": (c_int, [c_void_p, c_int, c_void_p]),
    "beam_release_host_graphs": (c_int, []),
    "beam_moe_permute_no_alloc": (c_int, [c_void_p, c_void_p, c_int, ctypes.POINTER(MoeConfig), c_void_p,
                                          c_void_p, c_void_p, c_void_p, c_void_p]),
    "beam_nvfp4_expert_bytes": (c_size_t, [ctypes.POINTER(MoeConfig), ctypes.POINTER(c_size_t),
                                           ctypes.POINTER(c_size_t), ctypes.POINTER(c_size_t),
                                           ctypes.POINTER(c_size_t)]),
    "beam_nvfp4_quantize_experts": (c_int, [c_void_p, c_void_p, ctypes.POINTER(MoeConfig), c_void_p, c_void_p,
                                            c_void_p, c_void_p, c_void_p, c_void_p]),
    "beam_nvfp4_quantize_rows": (c_int, [c_void_p, c_int, c_int, c_float, c_void_p, c_void_p, c_void_p]),
    "beam_moe_experts_nvfp4_workspace_size": (c_size_t, [ctypes.POINTER(MoeConfig), c_int]),
    "beam_moe_experts_nvfp4": (c_int, [c_void_p, c_void_p, ctypes.POINTER(MoeNvfp4Weights), c_void_p, c_void_p,
                                       c_int, ctypes.POINTER(MoeConfig), c_void_p,
                                       ctypes.POINTER(MoeNvfp4Intermediates), c_void_p, c_size_t, c_void_p]),
    "beam_moe_nvfp4_workspace_size": (c_size_t, [ctypes.POINTER(MoeConfig), c_int]),
    "beam_moe_layer_nvfp4": (c_int, [c_void_p, c_void_p, c_int, ctypes.POINTER(MoeNvfp4Weights), c_int,
                                     ctypes.POINTER(MoeConfig), c_void_p, c_void_p, ctypes.POINTER(MoeDebug),
                                     c_void_p, c_size_t, c_void_p]),
}

_lib: Optional[ctypes.CDLL] = None


def library() -> ctypes.CDLL:
    """Load libbeam.so (built in-tree by ``build.py``); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise BeamError(f"libbeam.so not found at {LIB_PATH}: build it with "
                            "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def beam_status_string(status: int) -> str:
    return library().beam_status_string(status).decode()


def _check(name: str, status: int) -> None:
    if status != 0:
        raise BeamError(f"{name} failed: {beam_status_string(status)} (status {status})")


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _p(t: Optional[torch.Tensor], dtype: Optional[torch.dtype] = None) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise BeamError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise BeamError("expected a contiguous tensor")
    if dtype is not None and t.dtype != dtype:
        raise BeamError(f"expected dtype {dtype}, got {t.dtype}")
    return t.data_ptr()


class Workspace:
    """A reusable device byte buffer for the library's scratch needs (grown on demand)."""

    def __init__(self, device: Optional[torch.device] = None):
        self.device = device
        self.buf: Optional[torch.Tensor] = None

    def get(self, nbytes: int) -> torch.Tensor:
        if self.buf is None or self.buf.numel() < nbytes:
            dev = self.device or torch.device("cuda", torch.cuda.current_device())
            self.buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
        return self.buf


_default_ws: dict = {}


def _ws(nbytes: int, ws: Optional[Workspace]) -> torch.Tensor:
    if ws is None:
        dev = torch.cuda.current_device()
        ws = _default_ws.setdefault(dev, Workspace(torch.device("cuda", dev)))
    return ws.get(nbytes)


def beam_moe_workspace_size(cfg: MoeConfig, T: int) -> int:
    return library().beam_moe_workspace_size(ctypes.byref(cfg), T)


def beam_moe_permute_workspace_size(cfg: MoeConfig, T: int) -> int:
    return library().beam_moe_permute_workspace_size(ctypes.byref(cfg), T)


def beam_moe_experts_workspace_size(cfg: MoeConfig, T: int) -> int:
    return library().beam_moe_experts_workspace_size(ctypes.byref(cfg), T)


def beam_moe_layer_host_workspace_size(cfg: MoeConfig, T: int) -> int:
    return library().beam_moe_layer_host_workspace_size(ctypes.byref(cfg), T)


def beam_last_launch_count() -> int:
    return library().beam_last_launch_count()


def beam_boundary_norm(h, x, w_post, w_pre, eps: float, n: int, h_out=None, z_out=None):
    """Returns (h_out, z). ``h_out`` may be ``h`` itself (in-place residual update)."""
    T, H = h.shape
    h_out = torch.empty_like(h) if h_out is None else h_out
    z_out = torch.empty_like(h) if z_out is None else z_out
    bf = torch.bfloat16
    _check("beam_boundary_norm", library().beam_boundary_norm(
        _p(h, bf), _p(x, bf), _p(w_post, bf), _p(w_pre, bf), T, H, eps, n, _p(h_out, bf), _p(z_out, bf),
        _stream()))
    return h_out, z_out


def beam_router_topk(z, router_w, bias, cfg: MoeConfig, logits=None, ids=None, w=None):
    """Returns (logits fp32 [T][E], topk_ids int32 [T][K], topk_w fp32 [T][K])."""
    T = z.shape[0]
    dev = z.device
    logits = torch.empty(T, cfg.num_experts, dtype=torch.float32, device=dev) if logits is None else logits
    ids = torch.empty(T, cfg.topk, dtype=torch.int32, device=dev) if ids is None else ids
    w = torch.empty(T, cfg.topk, dtype=torch.float32, device=dev) if w is None else w
    _check("beam_router_topk", library().beam_router_topk(
        _p(z, torch.bfloat16), _p(router_w, torch.float32), _p(bias, torch.float32), T, ctypes.byref(cfg),
        _p(logits, torch.float32), _p(ids, torch.int32), _p(w, torch.float32), _stream()))
    return logits, ids, w


def beam_moe_permute(ids, z, cfg: MoeConfig, gather: bool = True, ws: Optional[Workspace] = None):
    """Returns (expert_offsets [E+1], perm_token [T*K], inv_perm [T*K], x_perm [T*K][H] or None)."""
    T = ids.shape[0]
    dev = ids.device
    rows = T * cfg.topk
    offsets = torch.empty(cfg.num_experts + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(rows, dtype=torch.int32, device=dev)
    inv = torch.empty(rows, dtype=torch.int32, device=dev)
    x_perm = torch.empty(rows, cfg.hidden, dtype=torch.bfloat16, device=dev) if gather else None
    nbytes = beam_moe_permute_workspace_size(cfg, T)
    buf = _ws(nbytes, ws)
    _check("beam_moe_permute", library().beam_moe_permute(
        _p(ids, torch.int32), _p(z, torch.bfloat16) if z is not None else None, T, ctypes.byref(cfg),
        _p(offsets), _p(perm), _p(inv), _p(x_perm), buf.data_ptr(), buf.numel(), _stream()))
    return offsets, perm, inv, x_perm


def beam_moe_experts(x_perm, offsets, w_gate_up, w_down, topk_w, inv_perm, cfg: MoeConfig, T: int,
                     y_out=None, ws: Optional[Workspace] = None):
    """Returns y bf16 [T][H]."""
    y_out = torch.empty(T, cfg.hidden, dtype=torch.bfloat16, device=x_perm.device) if y_out is None else y_out
    buf = _ws(beam_moe_experts_workspace_size(cfg, T), ws)
    bf = torch.bfloat16
    _check("beam_moe_experts", library().beam_moe_experts(
        _p(x_perm, bf), _p(offsets, torch.int32), _p(w_gate_up, bf), _p(w_down, bf), _p(topk_w, torch.float32),
        _p(inv_perm, torch.int32), T, ctypes.byref(cfg), _p(y_out, bf), buf.data_ptr(), buf.numel(), _stream()))
    return y_out


def beam_moe_gate_up(x_perm, offsets, w_gate_up, cfg: MoeConfig, T: int, act=None,
                     ws: Optional[Workspace] = None):
    """Returns act bf16 [T*K][F] = silu(x W_g^T) * (x W_u^T) per expert."""
    act = torch.empty(T * cfg.topk, cfg.d_ff, dtype=torch.bfloat16, device=x_perm.device) if act is None else act
    buf = _ws(beam_moe_experts_workspace_size(cfg, T), ws)
    bf = torch.bfloat16
    _check("beam_moe_gate_up", library().beam_moe_gate_up(
        _p(x_perm, bf), _p(offsets, torch.int32), _p(w_gate_up, bf), T, ctypes.byref(cfg), _p(act, bf),
        buf.data_ptr(), buf.numel(), _stream()))
    return act


def beam_moe_down(act, offsets, w_down, cfg: MoeConfig, T: int, y_perm=None, ws: Optional[Workspace] = None):
    """Returns y_perm bf16 [T*K][H] = act W_d^T per expert."""
    y_perm = (torch.empty(T * cfg.topk, cfg.hidden, dtype=torch.bfloat16, device=act.device)
              if y_perm is None else y_perm)
    buf = _ws(beam_moe_experts_workspace_size(cfg, T), ws)
    bf = torch.bfloat16
    _check("beam_moe_down", library().beam_moe_down(
        _p(act, bf), _p(offsets, torch.int32), _p(w_down, bf), T, ctypes.byref(cfg), _p(y_perm, bf),
        buf.data_ptr(), buf.numel(), _stream()))
    return y_perm


def beam_moe_combine(y_perm, topk_w, inv_perm, cfg: MoeConfig, T: int, y_out=None):
    y_out = torch.empty(T, cfg.hidden, dtype=torch.bfloat16, device=y_perm.device) if y_out is None else y_out
    _check("beam_moe_combine", library().beam_moe_combine(
        _p(y_perm, torch.bfloat16), _p(topk_w, torch.float32), _p(inv_perm, torch.int32), T, ctypes.byref(cfg),
        _p(y_out, torch.bfloat16), _stream()))
    return y_out


def weights_struct(w_post, w_pre, router_w, bias, w_gate_up, w_down) -> MoeWeights:
    """The weights as the C struct of device pointers; the struct keeps the
    tensors alive for as long as it lives."""
    bf = torch.bfloat16
    s = MoeWeights(_p(w_post, bf), _p(w_pre, bf), _p(router_w, torch.float32), _p(bias, torch.float32),
                   _p(w_gate_up, bf), _p(w_down, bf))
    s._keep = (w_post, w_pre, router_w, bias, w_gate_up, w_down)
    return s


def beam_moe_layer(h, x, n: int, weights: MoeWeights, cfg: MoeConfig, h_out=None, y_out=None,
                   debug: bool = False, ws: Optional[Workspace] = None):
    """One MoE sublayer. Returns (h_out, y, dbg) where dbg holds z, logits,
    topk_ids, topk_w and expert_offsets when ``debug`` is set (else None)."""
    T = h.shape[0]
    dev = h.device
    h_out = torch.empty_like(h) if h_out is None else h_out
    y_out = torch.empty_like(h) if y_out is None else y_out
    dbg, dbg_struct = None, None
    if debug:
        dbg = {"z": torch.empty_like(h),
               "logits": torch.empty(T, cfg.num_experts, dtype=torch.float32, device=dev),
               "topk_ids": torch.empty(T, cfg.topk, dtype=torch.int32, device=dev),
               "topk_w": torch.empty(T, cfg.topk, dtype=torch.float32, device=dev),
               "expert_offsets": torch.empty(cfg.num_experts + 1, dtype=torch.int32, device=dev)}
        dbg_struct = MoeDebug(*(dbg[k].data_ptr() for k in ("z", "logits", "topk_ids", "topk_w",
                                                             "expert_offsets")))
    buf = _ws(beam_moe_workspace_size(cfg, T), ws)
    bf = torch.bfloat16
    _check("beam_moe_layer", library().beam_moe_layer(
        _p(h, bf), _p(x, bf), n, ctypes.byref(weights), T, ctypes.byref(cfg), _p(h_out, bf), _p(y_out, bf),
        ctypes.byref(dbg_struct) if dbg_struct is not None else None, buf.data_ptr(), buf.numel(), _stream()))
    return h_out, y_out, dbg


def _ws_view(buf: torch.Tensor, ptr: int, dtype, shape):
    """A tensor over `buf` (a uint8 workspace) starting at device address `ptr`."""
    off = ptr - buf.data_ptr()
    nbytes = math.prod(shape) * torch.empty((), dtype=dtype).element_size()
    if off < 0 or off + nbytes > buf.numel():
        raise BeamError("address outside the workspace")
    return buf[off:off + nbytes].view(dtype).view(*shape)


def beam_moe_layer_uncombined(h, x, n: int, weights: MoeWeights, cfg: MoeConfig, h_out=None,
                              ws: Optional[Workspace] = None):
    """The layer without its combine. Returns (h_out, (y_perm, topk_w, inv_perm)), the last three
    views of the workspace (valid until it is next used), ready for beam_boundary_norm_combine."""
    T = h.shape[0]
    h_out = torch.empty_like(h) if h_out is None else h_out
    buf = _ws(beam_moe_workspace_size(cfg, T), ws)
    out = MoeUncombined()
    bf = torch.bfloat16
    _check("beam_moe_layer_uncombined", library().beam_moe_layer_uncombined(
        _p(h, bf), _p(x, bf), n, ctypes.byref(weights), T, ctypes.byref(cfg), _p(h_out, bf), ctypes.byref(out),
        buf.data_ptr(), buf.numel(), _stream()))
    if T == 0:
        return h_out, None
    K, H = cfg.topk, cfg.hidden
    return h_out, (_ws_view(buf, out.y_perm, bf, (T * K, H)), _ws_view(buf, out.topk_w, torch.float32, (T, K)),
                   _ws_view(buf, out.inv_perm, torch.int32, (T * K,)))


def beam_boundary_norm_combine(h, y_perm, topk_w, inv_perm, w_post, w_pre, eps: float, n: int, h_out=None,
                               z_out=None):
    """The boundary with x = the combine of (y_perm, topk_w, inv_perm). Returns (h_out, z)."""
    T, H = h.shape
    K = topk_w.shape[1] if T > 0 else 1
    h_out = torch.empty_like(h) if h_out is None else h_out
    z_out = torch.empty_like(h) if z_out is None else z_out
    bf = torch.bfloat16
    _check("beam_boundary_norm_combine", library().beam_boundary_norm_combine(
        _p(h, bf), _p(y_perm, bf), _p(topk_w, torch.float32), _p(inv_perm, torch.int32), K, _p(w_post, bf),
        _p(w_pre, bf), T, H, eps, n, _p(h_out, bf), _p(z_out, bf), _stream()))
    return h_out, z_out


def beam_moe_layer_host(h_host: torch.Tensor, x_host: torch.Tensor, n: int, weights: MoeWeights,
                        cfg: MoeConfig, h_out_host=None, y_out_host=None, ws: Optional[Workspace] = None):
    """The layer on HOST bf16 tensors (pinned recommended); copies in and out and synchronises."""
    T = h_host.shape[0]
    for t in (h_host, x_host):
        if t.is_cuda or not t.is_contiguous() or t.dtype != torch.bfloat16:
            raise BeamError("beam_moe_layer_host expects contiguous bf16 host tensors")
    h_out_host = torch.empty_like(h_host) if h_out_host is None else h_out_host
    y_out_host = torch.empty_like(h_host) if y_out_host is None else y_out_host
    buf = _ws(beam_moe_layer_host_workspace_size(cfg, T), ws)
    _check("beam_moe_layer_host", library().beam_moe_layer_host(
        h_host.data_ptr(), x_host.data_ptr(), n, ctypes.byref(weights), T, ctypes.byref(cfg),
        h_out_host.data_ptr(), y_out_host.data_ptr(), buf.data_ptr(), buf.numel(), _stream()))
    return h_out_host, y_out_host


def beam_moe_layer_nvfp4_host_workspace_size(cfg: MoeConfig, T: int) -> int:
    return library().beam_moe_layer_nvfp4_host_workspace_size(ctypes.byref(cfg), T)


def beam_moe_layer_nvfp4_host(h_host: torch.Tensor, x_host: torch.Tensor, n: int, weights: MoeNvfp4Weights,
                              cfg: MoeConfig, h_out_host=None, y_out_host=None, ws: Optional[Workspace] = None):
    """beam_moe_layer_host with NVFP4 experts."""
    T = h_host.shape[0]
    for t in (h_host, x_host):
        if t.is_cuda or not t.is_contiguous() or t.dtype != torch.bfloat16:
            raise BeamError("beam_moe_layer_nvfp4_host expects contiguous bf16 host tensors")
    h_out_host = torch.empty_like(h_host) if h_out_host is None else h_out_host
    y_out_host = torch.empty_like(h_host) if y_out_host is None else y_out_host
    buf = _ws(beam_moe_layer_nvfp4_host_workspace_size(cfg, T), ws)
    _check("beam_moe_layer_nvfp4_host", library().beam_moe_layer_nvfp4_host(
        h_host.data_ptr(), x_host.data_ptr(), n, ctypes.byref(weights), T, ctypes.byref(cfg),
        h_out_host.data_ptr(), y_out_host.data_ptr(), buf.data_ptr(), buf.numel(), _stream()))
    return h_out_host, y_out_host


def beam_get_device_error() -> int:
    """Synchronises the current stream; returns 0 or the site code of a timed-out device wait."""
    code = c_int(0)
    status = library().beam_get_device_error(ctypes.byref(code), _stream())
    if status not in (0, 6):
        _check("beam_get_device_error", status)
    return code.value


def beam_release_host_graphs() -> None:
    """Frees the CUDA graphs that repeated host-buffer layer calls captured."""
    _check("beam_release_host_graphs", library().beam_release_host_graphs())


def beam_check_bounded_wait(limit_ms: int = 50) -> int:
    """Runs the device bounded-wait check (a wait on a flag nothing sets);
    returns the site code it reported. Raises if it did not time out cleanly."""
    flag = torch.zeros(4, dtype=torch.int32, device="cuda")
    site = c_int(0)
    _check("beam_check_bounded_wait", library().beam_check_bounded_wait(flag.data_ptr(), limit_ms,
                                                                      ctypes.byref(site), _stream()))
    return site.value


def beam_check_bounded_wait_pending(limit_ms: int = 50) -> None:
    """Runs the device bounded-wait check and leaves its site code pending in
    the device error word (for the next error query or host-buffer layer call
    to report)."""
    flag = torch.zeros(4, dtype=torch.int32, device="cuda")
    _check("beam_check_bounded_wait_pending",
           library().beam_check_bounded_wait_pending(flag.data_ptr(), limit_ms, _stream()))


# ---------------------------------------------------------------- NVFP4 experts
class Nvfp4Experts:
    """Device tensors of NVFP4 expert weights (layouts in beam.h): codes and
    scale atoms of gate/up and down, and the per-expert FP32 scales."""

    def __init__(self, q_gate_up, sf_gate_up, q_down, sf_down, expert_scale):
        self.q_gate_up, self.sf_gate_up = q_gate_up, sf_gate_up
        self.q_down, self.sf_down = q_down, sf_down
        self.expert_scale = expert_scale


def beam_nvfp4_quantize_experts(w_gate_up, w_down, cfg: MoeConfig) -> Nvfp4Experts:
    """Quantizes bf16 expert weights [E][2F][H] and [E][H][F] to NVFP4."""
    sizes = [c_size_t(0) for _ in range(4)]
    if library().beam_nvfp4_expert_bytes(ctypes.byref(cfg), *(ctypes.byref(v) for v in sizes)) == 0:
        raise BeamError("beam_nvfp4_expert_bytes: unsupported config")
    dev = w_gate_up.device
    bufs = [torch.empty(v.value, dtype=torch.uint8, device=dev) for v in sizes]
    scale = torch.empty(cfg.num_experts, dtype=torch.float32, device=dev)
    bf = torch.bfloat16
    _check("beam_nvfp4_quantize_experts", library().beam_nvfp4_quantize_experts(
        _p(w_gate_up, bf), _p(w_down, bf), ctypes.byref(cfg), *(b.data_ptr() for b in bufs), scale.data_ptr(),
        _stream()))
    return Nvfp4Experts(bufs[0], bufs[1], bufs[2], bufs[3], scale)


def beam_nvfp4_quantize_rows(x, scale: float):
    """bf16 rows [R][K] -> (codes uint8 [R][K/2], scale slots uint8 [R][K/64][16])."""
    R, K = x.shape
    q = torch.empty(R, K // 2, dtype=torch.uint8, device=x.device)
    sf = torch.empty(R, K // 64, 16, dtype=torch.uint8, device=x.device)
    _check("beam_nvfp4_quantize_rows", library().beam_nvfp4_quantize_rows(
        _p(x, torch.bfloat16), R, K, scale, q.data_ptr(), sf.data_ptr(), _stream()))
    return q, sf


def nvfp4_weights_struct(w_post, w_pre, router_w, bias, experts: Nvfp4Experts, input_scale: float,
                         act_scale: float) -> MoeNvfp4Weights:
    bf = torch.bfloat16
    s = MoeNvfp4Weights(_p(w_post, bf), _p(w_pre, bf), _p(router_w, torch.float32), _p(bias, torch.float32),
                        _p(experts.q_gate_up, torch.uint8), _p(experts.sf_gate_up, torch.uint8),
                        _p(experts.q_down, torch.uint8), _p(experts.sf_down, torch.uint8),
                        _p(experts.expert_scale, torch.float32), input_scale, act_scale)
    s._keep = (w_post, w_pre, router_w, bias, experts)  # the struct holds raw pointers: keep the tensors alive
    return s


def beam_moe_experts_nvfp4(x_perm, offsets, weights: MoeNvfp4Weights, topk_w, inv_perm, cfg: MoeConfig, T: int,
                           y_out=None, ws: Optional[Workspace] = None):
    """The NVFP4 experts stage. Returns (y bf16 [T][H], intermediates dict of
    workspace views: x_q, x_sf, act_q, act_sf, y_perm)."""
    y_out = torch.empty(T, cfg.hidden, dtype=torch.bfloat16, device=x_perm.device) if y_out is None else y_out
    buf = _ws(library().beam_moe_experts_nvfp4_workspace_size(ctypes.byref(cfg), T), ws)
    inter = MoeNvfp4Intermediates()
    _check("beam_moe_experts_nvfp4", library().beam_moe_experts_nvfp4(
        _p(x_perm, torch.bfloat16), _p(offsets, torch.int32), ctypes.byref(weights), _p(topk_w, torch.float32),
        _p(inv_perm, torch.int32), T, ctypes.byref(cfg), _p(y_out, torch.bfloat16), ctypes.byref(inter),
        buf.data_ptr(), buf.numel(), _stream()))
    if T == 0:
        return y_out, None
    rows, H, F = T * cfg.topk, cfg.hidden, cfg.d_ff
    views = {"x_q": _ws_view(buf, inter.x_q, torch.uint8, (rows, H // 2)),
             "x_sf": _ws_view(buf, inter.x_sf, torch.uint8, (rows, H // 64, 16)),
             "act_q": _ws_view(buf, inter.act_q, torch.uint8, (rows, F // 2)),
             "act_sf": _ws_view(buf, inter.act_sf, torch.uint8, (rows, F // 64, 16)),
             "y_perm": _ws_view(buf, inter.y_perm, torch.bfloat16, (rows, H))}
    return y_out, views


def beam_moe_nvfp4_workspace_size(cfg: MoeConfig, T: int) -> int:
    return library().beam_moe_nvfp4_workspace_size(ctypes.byref(cfg), T)


def beam_moe_layer_nvfp4(h, x, n: int, weights: MoeNvfp4Weights, cfg: MoeConfig, h_out=None, y_out=None,
                         debug: bool = False, ws: Optional[Workspace] = None):
    """One MoE sublayer with NVFP4 experts. Returns (h_out, y, dbg) as beam_moe_layer."""
    T = h.shape[0]
    dev = h.device
    h_out = torch.empty_like(h) if h_out is None else h_out
    y_out = torch.empty_like(h) if y_out is None else y_out
    dbg, dbg_struct = None, None
    if debug:
        dbg = {"z": torch.empty_like(h),
               "logits": torch.empty(T, cfg.num_experts, dtype=torch.float32, device=dev),
               "topk_ids": torch.empty(T, cfg.topk, dtype=torch.int32, device=dev),
               "topk_w": torch.empty(T, cfg.topk, dtype=torch.float32, device=dev),
               "expert_offsets": torch.empty(cfg.num_experts + 1, dtype=torch.int32, device=dev)}
        dbg_struct = MoeDebug(*(dbg[k].data_ptr() for k in ("z", "logits", "topk_ids", "topk_w",
                                                             "expert_offsets")))
    buf = _ws(beam_moe_nvfp4_workspace_size(cfg, T), ws)
    bf = torch.bfloat16
    _check("beam_moe_layer_nvfp4", library().beam_moe_layer_nvfp4(
        _p(h, bf), _p(x, bf), n, ctypes.byref(weights), T, ctypes.byref(cfg), _p(h_out, bf), _p(y_out, bf),
        ctypes.byref(dbg_struct) if dbg_struct is not None else None, buf.data_ptr(), buf.numel(), _stream()))
    return h_out, y_out, dbg
