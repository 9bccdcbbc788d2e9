"""Host-side pieces of bench.py that decide what a JSON line claims: the DRAM
traffic is reported only for the kernel source it was captured on, the
timing notes say how the region was timed, and the window's flop count is
the visible pairs of the band mask (no GPU needed)."""
import json

import numpy as np

import bench
import oracle
from scaled_dot_product_18_b300 import inputs as I


def test_traffic_is_reported_only_for_the_captured_source(tmp_path, monkeypatch):
    entry = {"kernel_src_sha": bench.kernel_source_sha("fwd"), "dram_bytes_per_launch": 123.0, "from": "test"}
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"w": entry, "stale": dict(entry, kernel_src_sha="0")}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.committed_traffic("w") == 123.0
    assert bench.committed_traffic("stale") is None  # the kernel changed since the capture
    assert bench.committed_traffic("absent") is None


def test_source_hash_covers_the_kernel_files():
    for kind, files in bench.KERNEL_SOURCES.items():
        assert files[0].endswith(".cu") and "ptx_sm103.cuh" in files
    h = bench.kernel_source_sha("fwd")
    assert len(h) == 16 and h == bench.kernel_source_sha("fwd")
    assert bench.kernel_source_sha("mha") != h  # the block also hashes the GEMM source


def test_timing_notes():
    flushed = bench.timing_note(20, True, "attn_fwd")
    graph = bench.timing_note(20, False, "attn_fwd")
    assert "flushed" in flushed["l2"] and "events" in flushed["timed"]
    assert graph["l2"] == "inputs larger than L2" and "graph" in graph["timed"]
    # the default workload is larger than L2, the small ones fit
    assert I.WORKLOADS["c5_b1h32n16384d128_causal"].algorithmic_bytes() > bench.L2_BYTES
    assert I.WORKLOADS["c3_b16h12n512d64_keylens_x1.5"].algorithmic_bytes() <= bench.L2_BYTES
    assert bench.FLUSH_BYTES > bench.L2_BYTES


def test_window_flops_count_the_visible_pairs():
    w = I.Workload("t", 2, 3, 300, 64, True)
    for window in (1, 17, 128, 299, 300, 1000):
        vis = int(oracle.visible_mask(w.N, True, None, window).sum())
        assert bench.window_flops(w, window) == 4.0 * w.B * w.H * vis * w.d
