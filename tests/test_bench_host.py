"""Host-side logic of bench.py (no GPU): the committed DRAM-traffic figure is reported only
for the engine source it was captured on, and the measured peaks file sets the roofline
denominators."""
import json
import os

import bench


def test_traffic_reported_only_for_the_captured_engine_source(tmp_path, monkeypatch):
    key = "iso_leaf_tree_gemm_kernel<EPI_BF16>/M4096"
    prof = tmp_path / "profiles"
    prof.mkdir()
    good = {key: {"source_hash": bench.kernel_source_hash(), "dram_bytes_per_launch": 123.0}}
    (prof / "traffic.json").write_text(json.dumps(good))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # the engine sources are read from ROOT as well: point them at the real ones
    src = tmp_path / "parallelism_invariant_logprob_gb300" / "csrc"
    src.mkdir(parents=True)
    real = os.path.join(os.path.dirname(os.path.abspath(bench.__file__)), "parallelism_invariant_logprob_gb300",
                        "csrc")
    for f in bench.ENGINE_SOURCES:
        (src / f).write_bytes(open(os.path.join(real, f), "rb").read())
    assert bench.committed_traffic(key) == 123.0
    # a comment or blank-line edit keeps it
    orig = open(os.path.join(real, "gemm_tcgen05.cu"), "rb").read()
    (src / "gemm_tcgen05.cu").write_bytes(orig + b"\n// a note\n\n/* and another */\n")
    assert bench.committed_traffic(key) == 123.0
    # a changed engine source: the old figure is not reported
    (src / "gemm_tcgen05.cu").write_bytes(orig + b"\nstatic int x;\n")
    assert bench.committed_traffic(key) is None
    assert bench.committed_traffic("no such kernel") is None


def test_peaks_from_measured_file_or_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    fb = bench.load_peaks()
    assert fb["src"] == "fallback" and fb["hbm"] == 6800.0 and fb["tc"] == 1900.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(
        json.dumps({"hbm_gbs": 6684.5, "bf16_tflops": 1932.6, "bf16_tflops_sustained": 1700.0}))
    m = bench.load_peaks()
    assert m["src"] == "measured" and m["hbm"] == 6684.5 and m["tc"] == 1932.6
