"""CPU: the host-side logic of bench.py -- the algorithmic work per token that every roofline
fraction divides by, the check that a stored DRAM-traffic figure belongs to the current kernel
sources, and the reference arm's JSON line (on a tiny sample of the stream)."""
import json
import os
import shutil
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_algorithmic_work_per_token():
    # forward: q, k (16 key heads x 128, bf16), v, out (32 value heads x 128, bf16), g, beta (fp32)
    assert bench.BYTES_PER_TOKEN == 16 * 128 * 2 * 2 + 32 * 128 * 2 * 2 + 32 * 4 * 2 == 24832
    # per value head: the chunk's products 2 C (3K + 2V), the state's 3 K V, the C^2 / 6 of the solve
    assert abs(bench.FLOP_PER_TOKEN / 5.81e6 - 1) < 2e-3
    # prologue: 8192 channels read and written in bf16, a and b read, g and beta written in fp32
    assert bench.CH == 8192 and bench.PRO_BYTES_PER_TOKEN == 33152
    # decode: 256 requests, each its 32 fp32 128 x 128 states read and written
    assert bench.DEC_BYTES == 256 * (32 * 128 * 128 * 8 + 16 * 128 * 4 + 32 * 128 * 4 + 32 * 8 + 4)
    assert abs(bench.BWD_FLOP_PER_TOKEN / 16.8e6 - 1) < 0.01
    assert abs(bench.FP32_ALU_TFLOPS - 80.5) < 0.1


def test_stored_traffic_is_tied_to_the_kernel_sources(tmp_path, monkeypatch):
    # the committed figures belong to the committed sources
    for key in ("prologue", "decode", "emit_records", "sum_u_records", "sum_m_records"):
        assert bench.stored_traffic(key) is not None, key
    assert bench.stored_traffic("no such kernel") is None
    # a copy of the tree whose prologue source differs: its figure no longer counts
    (tmp_path / "profiles").mkdir()
    shutil.copy(os.path.join(ROOT, "profiles", "traffic.json"), tmp_path / "profiles")
    csrc = tmp_path / "gated_delta_rule_07_gb300" / "csrc"
    shutil.copytree(os.path.join(ROOT, "gated_delta_rule_07_gb300", "csrc"), csrc)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.stored_traffic("prologue") is not None
    with open(csrc / "gdn_prologue.cu", "a") as f:
        f.write("\n// edited\n")
    assert bench.stored_traffic("prologue") is None
    assert bench.stored_traffic("decode") is not None


def test_peaks_come_from_the_measured_file_when_present():
    hbm, tf, tf_sus, src = bench.peaks()
    if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")):
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        assert src == "measured" and hbm == float(d["hbm_gbs"]) and tf == float(d["bf16_tflops"])
    else:
        assert src == "fallback"


def test_reference_arm_line(monkeypatch):
    pytest.importorskip("oracle")
    monkeypatch.setattr(bench, "T_FULL", 256)
    args = types.SimpleNamespace(steps=1, warmup=0, ref_tokens=64)
    assert bench.run_reference(args, 2, 1) is None  # only rank 0 reports
    res = bench.run_reference(args, 1, 0)
    assert res["impl"] == "reference" and res["metric"] == bench.METRIC
    assert res["value"] > 0 and res["unit"] == "tokens/s" and res["higher_is_better"] is True
    assert res["cpu_baseline"]["kind"] == "oracle" and res["cpu_baseline"]["value"] == res["value"]
    assert res["e2e"] == {"value": res["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                          "d2h_bytes_per_step": 0}
    json.dumps(res)
