"""Host-side bookkeeping of bench.py: the DRAM traffic of a profiled kernel
is reported only while its source is the one the capture was taken on, and
the bf16 denominators are put side by side with the theoretical rate
computed from the SM count, the per-SM rate and the clock."""
import hashlib
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _tree(tmp_path, src_text, recorded_text):
    csrc = tmp_path / "exact_attention_40_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text(src_text)
    (tmp_path / "profiles").mkdir()
    rec = {"k_workload": {"kernel": "k", "source": "exact_attention_40_gb300/csrc/k.cu",
                          "source_sha256": hashlib.sha256(recorded_text.encode()).hexdigest(),
                          "bytes_per_launch": 12345}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))


def test_traffic_reported_for_the_profiled_source(tmp_path, monkeypatch):
    _tree(tmp_path, "kernel v1\n", "kernel v1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_traffic("k.cu", "k_workload") == 12345


def test_traffic_null_once_the_source_changed(tmp_path, monkeypatch):
    _tree(tmp_path, "kernel v2\n", "kernel v1\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.load_traffic("k.cu", "k_workload") is None
    assert bench.load_traffic("k.cu", "other_workload") is None
    assert bench.load_traffic("missing.cu", "k_workload") is None


def test_committed_traffic_records_name_existing_sources():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        data = json.load(f)
    for key, ent in data.items():
        assert os.path.exists(os.path.join(ROOT, ent["source"])), key
        assert ent["bytes_per_launch"] == ent["dram_read_bytes"] + ent["dram_write_bytes"], key


def test_bf16_peaks_side_by_side():
    peaks = {"bf16": 1885.7, "bf16_sus": 1703.3, "src": "measured"}
    side = bench.bf16_peaks(peaks, 152, 2070.0)
    assert side["bf16_burst_measured"] == 1885.7
    assert side["bf16_sustained_measured"] == 1703.3
    # 152 SMs x 8192 FLOP/clk x 2.07 GHz
    assert side["bf16_theoretical"] == pytest.approx(2577.53088, rel=1e-12)
    assert side["used_for_roofline"].startswith("bf16_burst_measured")


def test_spread_of_per_step_times():
    st = bench.spread([3.0, 1.0, 2.0, 10.0])
    assert st["ms_mean"] == 4.0
    assert st["ms_median"] == 2.5
    assert (st["ms_min"], st["ms_max"], st["calls"]) == (1.0, 10.0, 4)
