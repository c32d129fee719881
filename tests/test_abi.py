"""CPU-side checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments on the host before touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "beam.h")


@pytest.fixture(scope="module")
def beam():
    from routed_expert_layer_post_gb300 import build as b
    b.build()
    import routed_expert_layer_post_gb300 as m
    return m


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(beam_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_layer_entry_points():
    names = declared_functions()
    for n in ("beam_boundary_norm", "beam_router_topk", "beam_moe_permute", "beam_moe_experts", "beam_moe_layer"):
        assert n in names


def test_library_exports_every_declared_symbol(beam):
    lib = ctypes.CDLL(beam.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding knows the signature of every one of them
    assert set(declared_functions()) <= set(beam._SIGNATURES)


def test_status_strings(beam):
    assert beam.beam_status_string(0) == "ok"
    assert "workspace" in beam.beam_status_string(4)
    assert beam.library().beam_version().decode().startswith("beam")


def _cfg(beam, **kw):
    base = dict(hidden=5120, num_experts=256, num_groups=8, topk_groups=4, topk=8, d_ff=2560)
    base.update(kw)
    return beam.make_config(**base)


def test_config_validation(beam):
    lib = beam.library()
    ok = _cfg(beam)
    assert lib.beam_moe_workspace_size(ctypes.byref(ok), 64) > 0
    bad = [
        (_cfg(beam, num_experts=250), 1),           # E % G != 0
        (_cfg(beam, topk_groups=9), 1),             # TG > G
        (_cfg(beam, topk=200), 1),                  # K > TG * E/G
        (_cfg(beam, hidden=5000), 3),               # H % 256 != 0
        (_cfg(beam, d_ff=2500), 3),                 # F % 128 != 0
        (_cfg(beam, num_experts=512, num_groups=16), 3),
        (_cfg(beam, topk=17), 3),
        (_cfg(beam, hidden=0), 1),
    ]
    for c, want in bad:
        assert lib.beam_moe_workspace_size(ctypes.byref(c), 64) == 0
        st = lib.beam_router_topk(None, None, None, 4, ctypes.byref(c), None, None, None, None)
        assert st == want, (c.hidden, c.num_experts, c.topk, st)
    nan_eps = _cfg(beam)
    nan_eps.eps = float("nan")
    assert lib.beam_router_topk(None, None, None, 4, ctypes.byref(nan_eps), None, None, None, None) == 1


def test_host_side_rejections(beam):
    lib = beam.library()
    c = _cfg(beam)
    p16 = 0x10000            # a 16-byte aligned fake pointer (never dereferenced: rejected first)
    # empty batch is a valid no-op
    assert lib.beam_boundary_norm(None, None, None, None, 0, 5120, 1e-6, 3, None, None, None) == 0
    assert lib.beam_moe_layer(None, None, 3, ctypes.byref(beam.MoeWeights()), 0, ctypes.byref(c), None, None,
                              None, None, 0, None) == 0
    # null pointers, bad n, bad eps, bad H
    assert lib.beam_boundary_norm(None, p16, p16, p16, 4, 5120, 1e-6, 3, p16 + 64, p16 + 128, None) == 1
    assert lib.beam_boundary_norm(p16, p16, p16, p16, 4, 5120, 1e-6, 0, p16 + 64, p16 + 128, None) == 1
    assert lib.beam_boundary_norm(p16, p16, p16, p16, 4, 5120, -1.0, 3, p16 + 64, p16 + 128, None) == 1
    assert lib.beam_boundary_norm(p16, p16, p16, p16, 4, 5000, 1e-6, 3, p16 + 64, p16 + 128, None) == 3
    # misaligned
    assert lib.beam_boundary_norm(p16 + 2, p16, p16, p16, 4, 5120, 1e-6, 3, p16 + 64, p16 + 128, None) == 2
    # forbidden aliasing (z over h_out)
    assert lib.beam_boundary_norm(p16, p16 + 32, p16, p16, 4, 5120, 1e-6, 3, p16 + 64, p16 + 64, None) == 1
    # negative T
    assert lib.beam_router_topk(None, None, None, -1, ctypes.byref(c), None, None, None, None) == 1
    # workspace too small / misaligned workspace
    assert lib.beam_moe_permute(p16, p16, 4, ctypes.byref(c), p16, p16, p16, None, p16, 16, None) == 4
    assert lib.beam_moe_permute(p16, p16, 4, ctypes.byref(c), p16, p16, p16, None, p16 + 16, 1 << 30, None) == 2
    assert lib.beam_moe_experts(p16, p16, p16, p16, p16, p16, 4, ctypes.byref(c), p16, p16, 100, None) == 4
    # x_perm requested without z
    assert lib.beam_moe_permute(p16, None, 4, ctypes.byref(c), p16, p16, p16, p16, p16, 1 << 30, None) == 1
    # a null weight inside the weights struct
    w = beam.MoeWeights(p16, p16, p16, p16, None, p16)
    assert lib.beam_moe_layer(p16, p16, 3, ctypes.byref(w), 4, ctypes.byref(c), p16, p16, None, p16, 1 << 40,
                              None) == 1
    assert lib.beam_get_device_error(None, None) == 1


def test_workspace_sizes_grow_with_tokens(beam):
    lib = beam.library()
    c = _cfg(beam)
    # decode sizes include split-K partial sums, so T=1 can exceed T=64
    sizes = [lib.beam_moe_workspace_size(ctypes.byref(c), T) for T in (1, 64, 2048, 16384)]
    assert sizes[0] > 0 and sizes[1:] == sorted(sizes[1:])
    # the layer workspace covers x_perm, act and y_perm at least
    T = 2048
    assert sizes[2] >= T * 8 * (2 * 5120 + 2560) * 2
    assert lib.beam_moe_layer_host_workspace_size(ctypes.byref(c), T) >= sizes[2] + 4 * T * 5120 * 2
    fp4 = lib.beam_moe_nvfp4_workspace_size(ctypes.byref(c), T)
    assert fp4 > 0 and lib.beam_moe_layer_nvfp4_host_workspace_size(ctypes.byref(c), T) >= fp4 + 4 * T * 5120 * 2


def test_nvfp4_host_entry_rejects_bad_arguments(beam):
    lib = beam.library()
    c = _cfg(beam)
    p16 = ctypes.c_void_p(1 << 20)
    # no weights; then a workspace too small (checked before any device work)
    assert lib.beam_moe_layer_nvfp4_host(p16, p16, 3, None, 4, ctypes.byref(c), p16, p16, p16, 1 << 30, None) == 1
    w = beam.MoeNvfp4Weights()
    assert lib.beam_moe_layer_nvfp4_host(p16, p16, 3, ctypes.byref(w), 4, ctypes.byref(c), p16, p16, p16, 64,
                                         None) == 4


def test_bounded_wait_check_rejects_bad_arguments(beam):
    lib = beam.library()
    site = ctypes.c_int(7)
    assert lib.beam_check_bounded_wait(None, 50, ctypes.byref(site), None) == 1
    assert lib.beam_check_bounded_wait(ctypes.c_void_p(256), 0, ctypes.byref(site), None) == 1
    assert lib.beam_check_bounded_wait(ctypes.c_void_p(256), 5000, ctypes.byref(site), None) == 1
    assert lib.beam_check_bounded_wait(ctypes.c_void_p(258), 50, ctypes.byref(site), None) == 1  # misaligned
    pend = lib.beam_check_bounded_wait_pending
    assert pend(None, 50, None) == 1
    assert pend(ctypes.c_void_p(256), 0, None) == 1
    assert pend(ctypes.c_void_p(256), 5000, None) == 1
    assert pend(ctypes.c_void_p(258), 50, None) == 1


def test_deferred_combine_rejects_bad_arguments(beam):
    lib = beam.library()
    c = _cfg(beam)
    p16 = 0x10000
    fn = lib.beam_boundary_norm_combine
    # (h, y_perm, topk_w, inv_perm, K, w_post, w_pre, T, H, eps, n, h_out, z_out, stream)
    assert fn(None, None, None, None, 8, None, None, 0, 5120, 1e-6, 3, None, None, None) == 0  # empty batch
    assert fn(p16, p16 + 256, p16, p16, 0, p16, p16, 4, 5120, 1e-6, 3, p16 + 64, p16 + 128, None) == 1  # K = 0
    assert fn(p16, p16 + 256, p16, p16, 17, p16, p16, 4, 5120, 1e-6, 3, p16 + 64, p16 + 128, None) == 3  # K > 16
    assert fn(p16, p16 + 256, p16, p16, 8, p16, p16, 4, 5000, 1e-6, 3, p16 + 64, p16 + 128, None) == 3  # H
    assert fn(p16, p16 + 256, p16, p16, 8, p16, p16, 4, 5120, 1e-6, 0, p16 + 64, p16 + 128, None) == 1  # n
    assert fn(p16, None, p16, p16, 8, p16, p16, 4, 5120, 1e-6, 3, p16 + 64, p16 + 128, None) == 1  # null y_perm
    assert fn(p16, p16 + 256, p16 + 2, p16, 8, p16, p16, 4, 5120, 1e-6, 3, p16 + 64, p16 + 128, None) == 2
    assert fn(p16, p16 + 256, p16, p16, 8, p16, p16, 4, 5120, 1e-6, 3, p16 + 64, p16 + 64, None) == 1  # z on h'
    assert fn(p16, p16 + 256, p16, p16, 8, p16, p16, 4, 5120, 1e-6, 3, p16 + 256, p16 + 128, None) == 1  # h' on y
    out = beam.MoeUncombined()
    w = beam.MoeWeights(p16, p16, p16, p16, p16, p16)
    lu = lib.beam_moe_layer_uncombined
    assert lu(p16, p16, 3, ctypes.byref(w), 4, ctypes.byref(c), p16, None, p16, 1 << 40, None) == 1  # no out
    assert lu(None, None, 3, ctypes.byref(w), 0, ctypes.byref(c), None, ctypes.byref(out), None, 0, None) == 0
    assert out.y_perm is None and out.topk_w is None and out.inv_perm is None
    bad = beam.MoeWeights(p16, p16, None, p16, p16, p16)
    assert lu(p16, p16, 3, ctypes.byref(bad), 4, ctypes.byref(c), p16, ctypes.byref(out), p16, 1 << 40, None) == 1
    # beam_moe_layer still needs y_out
    assert lib.beam_moe_layer(p16, p16, 3, ctypes.byref(w), 4, ctypes.byref(c), p16, None, None, p16, 1 << 40,
                              None) == 1
