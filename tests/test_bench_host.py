"""Host-side logic of the benchmark on the CPU: argument handling, the
max-over-ranks / sum-of-work reduction across a world of 2 gloo ranks, the
clock-sample parser and the weight byte count."""
from __future__ import annotations

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench
from quantized_swiglu_mlp_gb300 import inputs


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, results):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # rank r "took" 10*(r+1) ms and processed 100*(r+1) units
    ms, units = bench.reduce_timing(10.0 * (rank + 1), 100.0 * (rank + 1))
    bench.barrier()
    results[rank] = (ms, units, bench.dist_info())
    dist.destroy_process_group()


def test_reduce_timing_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        ms, units, (world, rank, local) = results[r]
        assert ms == 20.0 and units == 300.0
        assert (world, rank, local) == (2, r, r)


def test_reduce_timing_single_process():
    assert bench.reduce_timing(5.0, 7.0) == (5.0, 7.0)


def test_clock_summary_parser():
    s = bench.ClockSampler(0)
    s.lines = ["0, 1965, 2070, 900.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
               "0, 1980, 2070, 905.0, 0x0, Not Active, Not Active, Not Active, Not Active",
               "garbage"]
    out = s.summary()
    assert out["sm_mhz"] == pytest.approx(1972.5) and out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap"] and out["samples"] == 2


def test_decode_weight_bytes():
    case = inputs.workload_case("decode")
    # packed 2 x 8192 x 1024 B + scales/biases 2 x 2 x 8192 x 32 x 2 B
    assert bench.weight_bytes(case) == 18_874_368


def test_warmup_floor():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_peaks_fallback_or_measured():
    peaks, src = bench.load_peaks()
    assert src in ("measured", "fallback")
    assert peaks["hbm_gbs"] > 1000 and peaks["bf16_tflops"] > 100


def test_peaks_per_key(tmp_path):
    f = tmp_path / "peaks.json"
    f.write_text('{"hbm_gbs": 7100.5, "bf16_tflops": {"value": 2010}}')
    peaks, src = bench.load_peaks(str(f))
    assert src == "measured"
    assert peaks["hbm_gbs"] == 7100.5 and peaks["bf16_tflops"] == 2010.0
    assert peaks["bf16_tflops_sustained"] == bench.FALLBACK_PEAKS["bf16_tflops_sustained"]
    f.write_text('{"hbm_gbs": 7100.5}')
    peaks, src = bench.load_peaks(str(f))
    assert src == "fallback" and peaks["hbm_gbs"] == 7100.5
    peaks, src = bench.load_peaks(str(tmp_path / "missing.json"))
    assert src == "fallback" and peaks == bench.FALLBACK_PEAKS
