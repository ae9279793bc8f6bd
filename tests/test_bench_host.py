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
    for f, body in (("moe_small.cu", b"kernel v1\n"), ("moe_device.cuh", b"helpers v1\n"),
                    ("moe_tcgen05.cuh", b"tc v1\n")):
        (csrc / f).write_bytes(body)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = hashlib.sha256(b"kernel v1\nhelpers v1\ntc v1\n").hexdigest()
    assert bench.kernel_source_sha("moe_small_kernel") == sha
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(
        {"moe_small_kernel/decode": {"kernel": "moe_small_kernel", "workload": "decode",
                                     "dram_bytes_per_launch": 56773376, "kernel_source_sha256": sha}}))
    assert bench.measured_traffic("moe_small_kernel", "decode") == 56773376
    assert bench.measured_traffic("moe_small_kernel", "spec_verify") is None   # not captured
    (csrc / "moe_device.cuh").write_bytes(b"helpers v2\n")       # a source changed since the capture
    assert bench.measured_traffic("moe_small_kernel", "decode") is None


def test_cpu_model_is_named():
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()
