"""CPU tests of the benchmark's host logic: the multi-rank aggregation over a
2-rank gloo process group (max time over ranks, whole-job throughput of
independent replicas), the accounting formulas, the clock-log parsing and
the rule that ncu traffic is reported only for unchanged kernel sources."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import synth


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [3.0, 5.0][rank]
    ms = bench.max_over_ranks(local_ms, world, dist)
    out[rank] = ms
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_max_and_job_throughput():
    world = 2
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, start_method="spawn")
    assert out[0] == 5.0 and out[1] == 5.0          # every rank sees the slowest time
    # two replicas of a 1 TFLOP step in 5 ms: 400 TFLOP/s for the job
    assert bench.job_throughput(1e12, 2, 5.0) == pytest.approx(400.0)
    assert bench.max_over_ranks(7.5, 1) == 7.5


def test_layer_accounting():
    r = synth.RECIPES["clamped_glu_fwd"]
    fwd, bwd = bench.layer_flops(r)
    assert fwd == 2 * 8192 * 4 * 3 * 2880 * 2880 and bwd == 2 * fwd
    bf, bb = bench.layer_bytes(r, 128)
    w = 128 * 3 * 2880 * 2880 * 2
    assert bf == pytest.approx(2 * 8192 * 2880 * 2 + w + 8192 * 4 * 8)
    assert bb > 128 * 3 * 2880 * 2880 * 4          # includes the fp32 weight gradients
    work = bench.kernel_work(r, 128)
    total_flops = sum(f for f, _ in work.values())
    assert total_flops == pytest.approx(fwd + bwd)  # the GEMM kernels carry all layer FLOPs


def test_clock_summary():
    lines = ["0, 2070, 2070, 900.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "0, 1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
             "0, 2010, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "garbage line"]
    s = bench.summarize_clocks(lines)
    assert s["sm_mhz"] == 2010 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 3
    assert bench.summarize_clocks([])["samples"] == 0


def test_traffic_requires_matching_sources(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (prof / ("k_%s.txt" % bench.WORKLOAD)).write_text("source_hash=deadbeef\ndram_bytes_per_launch=123\n")
    monkeypatch.setattr(bench, "csrc_hash", lambda: "0123abcd")
    assert bench.committed_traffic("k") is None
    monkeypatch.setattr(bench, "csrc_hash", lambda: "deadbeef")
    assert bench.committed_traffic("k") == 123.0


def test_peaks_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peaks, src = bench.load_peaks()
    assert src == "fallback" and peaks["hbm_gbs"] == 6800.0
    (tmp_path / "MEASURED_PEAKS.json").write_text('{"hbm_gbs": 7000, "bf16_tflops": 2000}')
    peaks, src = bench.load_peaks()
    assert src == "measured" and peaks["bf16_tflops_sustained"] == 2000.0


def test_zipf_routing_stats():
    r = synth.RECIPES["zipf_sweep"].scaled(T=512, H=64, I=64)
    case = synth.make_case(r, with_dy=False)
    zero, ratio = synth.routing_stats(case.topk_idx, r.E)
    assert zero >= 0.25 and ratio > 10.0
    # each token picks k distinct experts
    ids = case.topk_idx
    assert all(len(set(row.tolist())) == r.k for row in ids)


def test_stats_ms_percentiles():
    s = bench.stats_ms([float(v) for v in range(1, 12)])   # 1 .. 11 ms
    assert s["median"] == 6.0 and s["p10"] == 2.0 and s["p90"] == 10.0 and s["n"] == 11


def test_oracle_sample_is_bounded_and_consistent():
    """The CPU sample used by cpu_baseline and by the reference arm: a token
    prefix touching at most max_experts experts, whose timed passes run the
    oracle on host fp64 copies made beforehand."""
    r = synth.RECIPES["clamped_glu_fwd"].scaled(T=64, H=64, I=64, E=32)
    case = synth.make_case(r)
    smp = bench.OracleSample(case, max_experts=6)
    assert 1 <= smp.n_max <= r.T
    assert len(smp.experts(smp.n_max)) <= 6
    if smp.n_max < r.T:   # the next token would bring in a seventh expert
        nxt = set(case.topk_idx[:smp.n_max + 1].reshape(-1).tolist())
        assert len(nxt) > 6
    assert set(smp.wgu) == set(smp.experts(smp.n_max))
    assert smp.step(smp.n_max) > 0.0
