"""Host-side logic of bench.py: whole-job aggregation over ranks (gloo,
world size 2 on CPU), clock-record parsing, peaks and argument defaults."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, seconds, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    slowest = bench.reduce_max(seconds[rank], torch.device("cpu"))
    bench.barrier()
    value, slow = bench.whole_job(100, world, [slowest])
    out[rank] = (slowest, value)
    dist.destroy_process_group()


def test_whole_job_over_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, [1.5, 2.0], out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        slowest, value = out[r]
        assert slowest == 2.0                     # max over ranks
        assert value == pytest.approx(100 * 2 / 2.0)  # all ranks' tokens over the slowest rank's time


def test_clock_summary_parsing():
    c = bench.ClockSampler("0")
    c.lines = ["0, 1965, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
               "0, 1980, 2070, 1100.0, 0x4, Not Active, Not Active, Not Active, Active",
               "garbage", "0, 2010, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active"]
    s = c.summary()
    assert s["sm_mhz"] == 1980 and s["sm_max_mhz"] == 2070 and s["reasons"] == ["sw_power_cap"]
    assert s["samples"] == 3


def test_defaults_and_peaks():
    a = bench.parse_args([])
    assert a.config == "all" and a.warmup >= 3 and a.impl == "ours"
    runs, head = bench.workloads(a)
    names = ["toy", "decode_t1", "decode_t64", "prefill_t2048", "prefill_t16384"]
    assert runs == [(n, False) for n in names] + [("decode_t1", True), ("decode_t64", True)]
    assert head == ("prefill_t16384", False)
    assert [bench.run_key(r) for r in runs[-2:]] == ["decode_t1_nvfp4", "decode_t64_nvfp4"]
    assert all(bench.steps_for(a, n) > 0 and bench.batches_for(a, n) > 0 for n in names)
    assert bench.workloads(bench.parse_args(["--no-nvfp4"]))[0] == [(n, False) for n in names]
    one = bench.parse_args(["--config", "decode_t1", "--steps", "7"])
    assert bench.workloads(one) == ([("decode_t1", False)], ("decode_t1", False))
    assert bench.steps_for(one, "decode_t1") == 7
    fp4 = bench.parse_args(["--config", "decode_t64", "--nvfp4"])
    assert bench.workloads(fp4) == ([("decode_t64", True)], ("decode_t64", True))
    with pytest.raises(SystemExit):
        bench.parse_args(["--tokens", "8"])  # overrides need a single workload
    peaks, kind = bench.load_peaks()
    assert peaks["hbm_gbs"] > 1000 and kind in ("measured", "fallback")
    assert bench.whole_job(8, 1, [0.5]) == (16.0, 0.5)


def _toy_capture():
    """A capture of the toy workload whose 'GPU' outputs are the oracle's own
    (to test the parity report's bookkeeping on CPU)."""
    import numpy as np
    from beam_inputs import CONFIGS, make_activations, make_all_expert_weights, make_norm_weights, make_router
    from oracle import bf16 as obf
    from oracle.experts import decoded_expert
    from oracle.layer import layer
    cfg = CONFIGS["toy"]
    h, x = make_activations(cfg)
    wp, wq = make_norm_weights(cfg)
    W_r, bias = make_router(cfg)
    W_gu, W_d = make_all_expert_weights(cfg, workers=1, cache=False)
    ref = layer(obf.decode(h), obf.decode(x), obf.decode(wp), obf.decode(wq), W_r, bias, n=cfg.n, eps=cfg.eps,
                G=cfg.G, TG=cfg.TG, K=cfg.K, routed_scale=cfg.routed_scale,
                expert_fn=lambda e: decoded_expert(W_gu, W_d, e, cfg.F))
    t16 = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)  # noqa: E731
    return {"h": h, "x": x, "h_out": obf.encode(ref["h_new"]), "y": obf.encode(ref["y"]),
            "logits": ref["logits"].astype(np.float32), "ids": ref["ids"].copy(), "wp": wp, "wq": wq,
            "W_r": W_r, "bias": bias, "w_gu": t16(W_gu), "w_d": t16(W_d)}, ref


def test_parity_report_counts_and_flags_disagreements():
    import numpy as np
    from oracle.routing import near_tie
    cap, ref = _toy_capture()
    rep, timing = bench.parity_report("toy", cap, workers=1)
    assert timing is None
    assert rep["pass"] and rep["differing_rows"] == 0 and rep["h_worst_ulp"] == 0
    assert rep["routing_tokens"] == 16 and rep["y_tokens"] == 16 and rep["y_max_abs"] < 2e-2
    # one token routed to another expert (not a near-tie) must fail the report
    t = int(np.flatnonzero(~near_tie(ref["route"]))[0])
    bad = dict(cap, ids=cap["ids"].copy())
    bad["ids"][t, 0] = next(e for e in range(16) if e not in bad["ids"][t])
    rep2, _ = bench.parity_report("toy", bad, workers=1)
    assert rep2["differing_non_near_tie"] == 1 and not rep2["pass"]
    # an h' two ulps off must fail it too
    off = dict(cap, h_out=cap["h_out"].copy())
    off["h_out"][3, 5] += 2
    rep3, _ = bench.parity_report("toy", off, workers=1)
    assert rep3["h_worst_ulp"] == 2 and not rep3["pass"]
    # the timed variant evaluates tokens one at a time and reports its timing
    rep4, timing = bench.parity_report("toy", cap, timed_seconds=0.0, workers=1)
    assert timing["tokens"] == 1 and rep4["y_tokens"] == 1 and rep4["pass"]
