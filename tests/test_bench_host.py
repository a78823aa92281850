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
