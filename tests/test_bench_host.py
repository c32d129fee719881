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
    assert a.config == "decode_t1" and a.warmup >= 3 and a.steps > 0 and a.impl == "ours"
    peaks, kind = bench.load_peaks()
    assert peaks["hbm_gbs"] > 1000 and kind in ("measured", "fallback")
    assert bench.whole_job(8, 1, [0.5]) == (16.0, 0.5)
