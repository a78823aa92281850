"""Host-side pieces of bench.py (no GPU): traffic records, kernel source lists, JSON helpers."""

import os

import bench


def test_kernel_source_lists_exist():
    for kernel, names in bench.KERNEL_SOURCES.items():
        for n in names:
            assert os.path.exists(os.path.join(bench.ROOT, "context_paged_attention_gb300", "csrc", n)), (kernel, n)
        assert len(bench.source_digest(kernel)) == 16


def test_traffic_file_parses():
    # every record names a known kernel; a stale digest simply yields None
    with open(bench.TRAFFIC_FILE) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                kv = dict(x.split("=", 1) for x in line.split())
                assert kv["kernel"] in bench.KERNEL_SOURCES
                assert int(kv["dram_bytes_per_launch"]) > 0
    assert bench.recorded_traffic("gqa_partial", "no-such-workload") is None


def test_peaks_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    peak, src = bench.load_peaks()
    assert src == "fallback" and peak == bench.FALLBACK_HBM_GBS


def test_clock_summary_window_and_reasons():
    s = bench.ClockSampler(0)
    s.samples = [(0.5, 1900.0, 2070.0, set()), (1.0, 2070.0, 2070.0, set()), (1.5, 2050.0, 2070.0, {"sw_power_cap"}),
                 (2.0, 2070.0, 2070.0, set()), (3.0, 1000.0, 2070.0, {"hw_slowdown"})]
    out = s.summary(0.9, 2.1)
    assert out["window_samples"] == 3 and out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]
    # no sample inside the window: the nearest one stands in, and says so
    out = s.summary(2.6, 2.7)
    assert out["window_samples"] == 0 and out["samples"] == 1 and out["reasons"] == ["hw_slowdown"]


def test_clock_reason_bits():
    # NVML clock-event reason masks (nvml.h): SwPowerCap 0x4, HwSlowdown 0x8,
    # SwThermalSlowdown 0x20, HwThermalSlowdown 0x40
    assert bench._REASON_BITS == {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                                  "hw_thermal_slowdown": 0x40}


def test_launch_counts_and_bytes():
    from context_paged_attention_gb300 import workloads as W

    dec = W.tiny_fp32()
    mixed = W.mixed_step(seed=1, n_decode=2, n_extend=2, dec_ctx=(1, 50), ext_new=(2, 5), ext_ctx=(0, 30),
                         token_multiple=16)
    assert bench.launches_per_step(dec, True) == 2 and bench.launches_per_step(dec, False) == 3
    assert bench.launches_per_step(mixed, True) == 4 and bench.launches_per_step(mixed, False) == 5
    # fused: merged output instead of P partials; the KV bytes are the same
    f, u = bench.algorithmic_bytes(dec, True), bench.algorithmic_bytes(dec, False)
    assert f["kv"] == u["kv"] == dec.kv_bytes_read() and f["partial"] < u["partial"]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        # each replica reports its own step time; the job takes the slowest
        got = bench.max_over_ranks(dist, [1.0 + rank, 10.0 * rank], "cpu")
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_replica_timing_reduction_gloo():
    """Two CPU ranks (gloo): the max over ranks, and the job throughput of
    world x per-rank bytes over the slowest step."""
    import socket

    import torch.multiprocessing as mp

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == [2.0, 10.0] and out[1] == [2.0, 10.0]
    assert bench.job_throughput(2, 1e9, 2.0) == 2 * 1e9 / 2e-3 / 1e9
    assert bench.max_over_ranks(None, [3.0], "cpu") == [3.0]
