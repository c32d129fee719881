"""GPU parity of the NVFP4 experts (E2M1 values, E4M3 scale per 16, FP32
scale) against the oracle's NVFP4 definition (oracle.nvfp4), through the C
ABI: the two quantizers bit-exact, the experts stage's intermediate codes and
its down GEMM output, and the whole sublayer with NVFP4 experts."""
import numpy as np
import pytest
import torch

from beam_inputs import CONFIGS, make_activations, random_topk_ids
from oracle import bf16 as obf
from oracle import nvfp4 as q
from oracle.routing import near_tie
from tests.gpu_support import WORKERS, beam_module, bits_of, dev_bf16, f64_of, layer_errors, model

pytestmark = pytest.mark.gpu

G_IN = 2.0 ** -6    # FP32 scales of the two quantized activations (z and the SwiGLU output)
G_ACT = 2.0 ** -6


def _host_u8(t):
    return t.contiguous().cpu().numpy().view(np.uint8)


def unpack_atoms(sf, planes, rows, K):
    """The weight-scale atom layout of beam.h back to logical [planes * rows][K/16] codes."""
    a = np.asarray(sf, dtype=np.uint8).reshape(planes, rows // 128, K // 256, 4, 512)
    out = np.empty((planes, rows, K // 16), dtype=np.uint8)
    r = np.arange(128)
    for c in range(4):
        for j in range(4):
            # byte (r%32)*16 + (r/32)*4 + j of atom c holds row r, group 16s + 4c + j
            vals = a[:, :, :, c, (r % 32) * 16 + (r // 32) * 4 + j]        # [planes][blocks][steps][128]
            out[:, :, 4 * c + j::16] = vals.transpose(0, 1, 3, 2).reshape(planes, rows, K // 256)
    return out.reshape(planes * rows, K // 16)


def unpack_slots(sf):
    """[rows][K/64][16] activation scale slots -> logical [rows][K/16] codes."""
    s = np.asarray(sf, dtype=np.uint8)
    return s[:, :, :4].reshape(s.shape[0], -1)


def test_quantize_rows_is_bit_exact():
    beam = beam_module()
    rng = np.random.default_rng(21)
    rows, K = 37, 5120
    x = rng.standard_normal((rows, K)).astype(np.float32) * np.exp(rng.uniform(-3, 3, (rows, 1))).astype(np.float32)
    x[3, 64:128] = 0.0                     # whole zero blocks
    x[5, :16] = -x[5, :16]
    x[7, 16:32] = 1e-9                     # a block whose scale underflows to 0
    bits = obf.encode(x.astype(np.float64))
    xq, xsf = beam.beam_nvfp4_quantize_rows(dev_bf16(bits), G_IN)
    torch.cuda.synchronize()
    codes, scales = q.quantize(obf.decode(bits).astype(np.float32), G_IN)
    assert np.array_equal(q.unpack_codes(_host_u8(xq)), codes)
    sl = _host_u8(xsf).reshape(rows, K // 64, 16)
    assert np.array_equal(unpack_slots(sl), scales)
    assert not sl[:, :, 4:].any()


@pytest.mark.parametrize("name", ["toy_f256", "beam"])
def test_quantize_experts_is_bit_exact(name):
    beam = beam_module()
    if name == "toy_f256":
        cfg = CONFIGS["toy"].with_(F=256)
        from beam_inputs import make_all_expert_weights
        W_gu, W_d = make_all_expert_weights(cfg, workers=WORKERS)
        w_gu, w_d = dev_bf16(W_gu), dev_bf16(W_d)
        check = range(cfg.E)
    else:
        m = model("decode_t64")
        cfg, (w_gu, w_d) = m.cfg, m.dev
        W_gu, W_d = m.W_gu_bits, m.W_d_bits
        check = (0, 255)
    mc = beam.make_config(cfg.H, cfg.E, cfg.G, cfg.TG, cfg.K, cfg.F)
    ex = beam.beam_nvfp4_quantize_experts(w_gu, w_d, mc)
    torch.cuda.synchronize()
    E, H, F = cfg.E, cfg.H, cfg.F
    qgu = _host_u8(ex.q_gate_up).reshape(E, 2 * F, H // 2)
    qd = _host_u8(ex.q_down).reshape(E, H, F // 2)
    sgu = unpack_atoms(_host_u8(ex.sf_gate_up), 2 * E, F, H).reshape(E, 2 * F, H // 16)
    sd = unpack_atoms(_host_u8(ex.sf_down), E, H, F).reshape(E, H, F // 16)
    gs = ex.expert_scale.cpu().numpy()
    for e in check:
        ref = _oracle_expert(W_gu, W_d, e, F)
        assert gs[e] == ref.g, (e, gs[e], ref.g)
        assert np.array_equal(q.unpack_codes(qgu[e, :F]), ref.gate[0]) and np.array_equal(sgu[e, :F], ref.gate[1])
        assert np.array_equal(q.unpack_codes(qgu[e, F:]), ref.up[0]) and np.array_equal(sgu[e, F:], ref.up[1])
        assert np.array_equal(q.unpack_codes(qd[e]), ref.down[0]) and np.array_equal(sd[e], ref.down[1])


def _stage(beam, cfg, w_gu_dev, w_d_dev, W_gu, W_d, T, seed, skew=0.0):
    """Random routing -> permutation -> NVFP4 experts stage; returns what the
    checks need, with the oracle's experts quantized from the bf16 bits."""
    mc = beam.make_config(cfg.H, cfg.E, cfg.G, cfg.TG, cfg.K, cfg.F)
    ex = beam.beam_nvfp4_quantize_experts(w_gu_dev, w_d_dev, mc)
    rng = np.random.default_rng(seed)
    z_bits = obf.encode(rng.standard_normal((T, cfg.H)))
    ids = torch.from_numpy(random_topk_ids(T, cfg.E, cfg.K, seed=seed, skew=skew).astype(np.int32)).cuda()
    z = dev_bf16(z_bits)
    offsets, perm, inv, x_perm = beam.beam_moe_permute(ids, z, mc)
    w = torch.rand(T, cfg.K, device="cuda", generator=torch.Generator("cuda").manual_seed(seed)) + 0.1
    w = (2.5 * w / w.sum(dim=1, keepdim=True)).contiguous()
    zero = torch.zeros(1, dtype=torch.bfloat16, device="cuda")
    wt = beam.nvfp4_weights_struct(zero, zero, torch.zeros(1, device="cuda"), torch.zeros(1, device="cuda"), ex,
                                   G_IN, G_ACT)
    y, inter = beam.beam_moe_experts_nvfp4(x_perm, offsets, wt, w, inv, mc, T)
    torch.cuda.synchronize()
    assert beam.beam_get_device_error() == 0
    return dict(mc=mc, ex=ex, z_bits=z_bits, off=offsets.cpu().numpy(), perm=perm.cpu().numpy(),
                inv=inv.cpu().numpy(), w=w.cpu().numpy(), y=y, inter={k: v.clone() for k, v in inter.items()})


_ORACLE_EXPERTS = {}


def _oracle_expert(W_gu, W_d, e, F):
    """The oracle's NVFP4 quantization of expert e of the packed bf16 weights (cached per process)."""
    key = (id(W_gu), e)
    if key not in _ORACLE_EXPERTS:
        Wg = obf.decode(W_gu[e, :F]).astype(np.float32)
        Wu = obf.decode(W_gu[e, F:]).astype(np.float32)
        Wd = obf.decode(W_d[e]).astype(np.float32)
        _ORACLE_EXPERTS[key] = q.Nvfp4Expert(Wg, Wu, Wd)
    return _ORACLE_EXPERTS[key]


@pytest.mark.parametrize("T,skew", [(16, 0.0), (64, 1.2)])
def test_experts_stage_toy_shapes(T, skew):
    beam = beam_module()
    cfg = CONFIGS["toy"].with_(F=256)
    from beam_inputs import make_all_expert_weights
    W_gu, W_d = make_all_expert_weights(cfg, workers=WORKERS)
    r = _stage(beam, cfg, dev_bf16(W_gu), dev_bf16(W_d), W_gu, W_d, T, seed=500 + T, skew=skew)
    _check_stage(cfg, r, W_gu, W_d, experts=range(cfg.E))


@pytest.mark.parametrize("T", [1, 8, 64])
def test_experts_stage_beam_shapes(T):
    beam = beam_module()
    m = model("decode_t64")
    cfg = m.cfg
    r = _stage(beam, cfg, m.dev[0], m.dev[1], m.W_gu_bits, m.W_d_bits, T, seed=600 + T)
    touched = [e for e in range(cfg.E) if r["off"][e + 1] > r["off"][e]]
    _check_stage(cfg, r, m.W_gu_bits, m.W_d_bits, experts=touched[:3])


def _check_stage(cfg, r, W_gu, W_d, experts):
    H, F = cfg.H, cfg.F
    rows = r["perm"].shape[0]
    inter = r["inter"]
    # the quantized input rows: bit-exact
    xq = q.unpack_codes(_host_u8(inter["x_q"]))
    xs = unpack_slots(_host_u8(inter["x_sf"]))
    xc, xsc = q.quantize(obf.decode(r["z_bits"][r["perm"]]).astype(np.float32), G_IN)
    assert np.array_equal(xq, xc) and np.array_equal(xs, xsc)
    aq = q.unpack_codes(_host_u8(inter["act_q"]))
    asf = unpack_slots(_host_u8(inter["act_sf"]))
    y_perm = f64_of(inter["y_perm"])
    code_diff = scale_diff = total = 0
    for e in experts:
        lo, hi = int(r["off"][e]), int(r["off"][e + 1])
        if hi == lo:
            continue
        ex = _oracle_expert(W_gu, W_d, e, F)
        Y, ac, as_ = q.ffn(obf.decode(r["z_bits"][r["perm"][lo:hi]]), ex, G_IN, G_ACT, return_act=True)
        # the SwiGLU output's codes: decided in FP32 from the GPU's FP32 sums,
        # so a value within rounding of a decision boundary may differ
        code_diff += int((aq[lo:hi] != ac).sum())
        scale_diff += int((asf[lo:hi] != as_).sum())
        total += ac.size
        # the down GEMM on the GPU's own SwiGLU codes: fp32 accumulation, one bf16 rounding
        _, _, Wd = ex.values()
        ref = q.dequantize(aq[lo:hi], asf[lo:hi], G_ACT) @ Wd.T
        err = np.abs(y_perm[lo:hi] - ref)
        assert np.all(err <= 2.0 ** -8 * np.abs(ref) + 1e-4), (e, float(err.max()))
        # and against the oracle's own act: the whole expert within the layer tolerance
        mx, rel = layer_errors(y_perm[lo:hi], Y)
        assert mx <= 2e-2 and rel <= 5e-3, (e, mx, rel)
    print(f"act codes differing {code_diff}/{total}, scales differing {scale_diff}/{total // 16}")
    assert code_diff <= max(4, total // 10000) and scale_diff <= max(2, total // 160000)


@pytest.mark.parametrize("name,tokens", [("toy_f256", None), ("decode_t1", None), ("decode_t64", [37])])
def test_layer_nvfp4_matches_oracle(name, tokens):
    beam = beam_module()
    if name == "toy_f256":
        cfg = CONFIGS["toy"].with_(F=256)
        from beam_inputs import make_all_expert_weights, make_norm_weights, make_router
        W_gu, W_d = make_all_expert_weights(cfg, workers=WORKERS)
        w_gu, w_d = dev_bf16(W_gu), dev_bf16(W_d)
        hb, xb = make_activations(cfg)
        wp, wq = make_norm_weights(cfg)
        W_r, bias = make_router(cfg)
    else:
        m = model("decode_t64")
        cfg = m.cfg if name == "decode_t64" else CONFIGS["decode_t1"]
        W_gu, W_d, (w_gu, w_d) = m.W_gu_bits, m.W_d_bits, m.dev
        hb, xb = make_activations(cfg)
        wp, wq, W_r, bias = m.wp_bits, m.wq_bits, m.W_r, m.bias
    mc = beam.make_config(cfg.H, cfg.E, cfg.G, cfg.TG, cfg.K, cfg.F, cfg.routed_scale, cfg.eps)
    ex = beam.beam_nvfp4_quantize_experts(w_gu, w_d, mc)
    wt = beam.nvfp4_weights_struct(dev_bf16(wp), dev_bf16(wq), torch.from_numpy(W_r).cuda(),
                                   torch.from_numpy(bias).cuda(), ex, G_IN, G_ACT)
    h_out, y, dbg = beam.beam_moe_layer_nvfp4(dev_bf16(hb), dev_bf16(xb), cfg.n, wt, mc, debug=True)
    torch.cuda.synchronize()
    assert beam.beam_get_device_error() == 0
    tokens = np.arange(cfg.T) if tokens is None else np.array(tokens)
    from oracle.layer import layer
    cache = {}

    def ffn(e, X):
        if e not in cache:
            cache[e] = _oracle_expert(W_gu, W_d, e, cfg.F)
        return q.ffn(X, cache[e], G_IN, G_ACT)

    ref = layer(obf.decode(hb), obf.decode(xb), obf.decode(wp), obf.decode(wq), W_r, bias, n=cfg.n, eps=cfg.eps,
                G=cfg.G, TG=cfg.TG, K=cfg.K, routed_scale=cfg.routed_scale, ffn=ffn, tokens=tokens, workers=WORKERS)
    ids = dbg["topk_ids"].cpu().numpy()[tokens]
    same = np.all(ids == ref["ids"], axis=1)
    assert np.all(same | near_tie(ref["route"]))
    obf_h = bits_of(h_out)[tokens]
    assert int(obf.ulp_distance(obf_h, obf.encode(ref["h_new"])).max()) <= 1
    mx, rel = layer_errors(f64_of(y)[tokens][same], ref["y"][same])
    print(f"{name} NVFP4 layer: tokens {tokens.size}, max|dy| {mx:.3e}, rel-L2 {rel:.3e}")
    assert mx <= 2e-2 and rel <= 5e-3, (mx, rel)


_FP4_EXPERTS = {}


@pytest.mark.parametrize("T", [1, 3, 8])
def test_decode_routing_writes_rows_like_the_quantizer(T):
    """At decode sizes the routing kernel writes the permuted rows as NVFP4
    itself. The layer output must be bit-identical to the experts stage fed
    with the same routing and the standalone row quantizer."""
    beam = beam_module()
    m = model("decode_t64")
    cfg = m.cfg.with_(T=T)
    mc = beam.make_config(cfg.H, cfg.E, cfg.G, cfg.TG, cfg.K, cfg.F, cfg.routed_scale, cfg.eps)
    if "beam" not in _FP4_EXPERTS:
        _FP4_EXPERTS["beam"] = beam.beam_nvfp4_quantize_experts(m.dev[0], m.dev[1], mc)
    wt = beam.nvfp4_weights_struct(dev_bf16(m.wp_bits), dev_bf16(m.wq_bits), torch.from_numpy(m.W_r).cuda(),
                                   torch.from_numpy(m.bias).cuda(), _FP4_EXPERTS["beam"], G_IN, G_ACT)
    hb, xb = make_activations(cfg)
    _, y, dbg = beam.beam_moe_layer_nvfp4(dev_bf16(hb), dev_bf16(xb), cfg.n, wt, mc, debug=True)
    offsets, _, inv, x_perm = beam.beam_moe_permute(dbg["topk_ids"], dbg["z"], mc)
    y2, _ = beam.beam_moe_experts_nvfp4(x_perm, offsets, wt, dbg["topk_w"], inv, mc, T)
    torch.cuda.synchronize()
    assert beam.beam_get_device_error() == 0
    assert torch.equal(offsets, dbg["expert_offsets"])
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("T,pinned_out", [(1, True), (8, False), (64, True), (300, True)])
def test_nvfp4_host_buffer_entry_point_matches_device(T, pinned_out):
    """beam_moe_layer_nvfp4_host (mapped host memory up to 8 tokens with
    page-locked buffers, copies otherwise) gives the bits of the device entry
    point."""
    beam = beam_module()
    m = model("decode_t64")
    cfg = m.cfg.with_(T=T)
    mc = beam.make_config(cfg.H, cfg.E, cfg.G, cfg.TG, cfg.K, cfg.F, cfg.routed_scale, cfg.eps)
    if "beam" not in _FP4_EXPERTS:
        _FP4_EXPERTS["beam"] = beam.beam_nvfp4_quantize_experts(m.dev[0], m.dev[1], mc)
    wt = beam.nvfp4_weights_struct(dev_bf16(m.wp_bits), dev_bf16(m.wq_bits), torch.from_numpy(m.W_r).cuda(),
                                   torch.from_numpy(m.bias).cuda(), _FP4_EXPERTS["beam"], G_IN, G_ACT)
    hb, xb = make_activations(cfg, batch=700 + T)
    h_dev, y_dev, _ = beam.beam_moe_layer_nvfp4(dev_bf16(hb), dev_bf16(xb), cfg.n, wt, mc)
    h_host = torch.from_numpy(hb.view(np.int16)).view(torch.bfloat16).pin_memory()
    x_host = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).pin_memory()
    h_out = torch.empty_like(h_host)
    y_out = torch.empty_like(h_host)
    if pinned_out:
        h_out, y_out = h_out.pin_memory(), y_out.pin_memory()
    for _ in range(3):  # the second identical call captures a graph (mapped path), the third replays it
        h_out, y = beam.beam_moe_layer_nvfp4_host(h_host, x_host, cfg.n, wt, mc, h_out_host=h_out, y_out_host=y_out)
        assert torch.equal(y.view(torch.int16), y_dev.cpu().view(torch.int16))
        assert torch.equal(h_out.view(torch.int16), h_dev.cpu().view(torch.int16))
