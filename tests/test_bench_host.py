"""Host-side pieces of bench.py that need no GPU: the oracle baseline timing,
the choice of roofline denominator and the staleness rule for the committed
DRAM-traffic figure."""
import hashlib
import json
import os

import bench
from quantized_moe_routed_gb300.inputs import (WORKLOADS, algorithmic_bytes, make_expert_weights, make_topk_ids,
                                               make_topk_w, make_x)


def test_cpu_baseline_reports_all_cores_and_one_thread():
    wl = WORKLOADS["tiny"]
    x, ids, w = make_x(wl), make_topk_ids(wl), make_topk_w(wl)
    S = {"wl": wl, "x": x, "ids": ids, "w": w, "W": make_expert_weights(wl, device="cpu"),
         "bytes": algorithmic_bytes(wl, ids)}
    cb = bench.cpu_baseline(S, seconds=0.2)
    assert cb["kind"] == "oracle" and cb["unit"] == "GB/s" and cb["value"] > 0
    assert cb["cores"] == (os.cpu_count() or 1)
    st = cb["single_thread"]
    assert st["cores"] == 1 and st["value"] > 0 and st["unit"] == "GB/s"


def test_peaks_prefers_the_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.peaks() == (6800.0, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6701.5}))
    assert bench.peaks() == (6701.5, "measured")


def test_traffic_is_reported_only_for_the_profiled_sources(tmp_path, monkeypatch):
    csrc = tmp_path / "quantized_moe_routed_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "moe_kernels.cu").write_bytes(b"kernel v1\n")
    (csrc / "moe_device.cuh").write_bytes(b"helpers v1\n")
    sha = hashlib.sha256(b"kernel v1\nhelpers v1\n").hexdigest()
    (tmp_path / "profiles" / "moe_step_kernel_decode.md").write_text(
        f"# summary\nkernel_source_sha256: {sha}\ntraffic_bytes_per_launch: 57300480\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic() == 57300480
    (csrc / "moe_device.cuh").write_bytes(b"helpers v2\n")       # a source changed since the capture
    assert bench.measured_traffic() is None
