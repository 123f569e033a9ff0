"""CPU checks of bench.py's bookkeeping: the kernel-source hash that keys the committed ncu traffic
records ignores comments but not code, every traffic record names a workload kernel family, and
the host CPU description is a non-empty string."""
import json
import os

import bench


def test_source_hash_ignores_comments_but_not_code(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "k.cu").write_text("// header\nint f(int x) { return x + 1; }  // inc\n/* block\n */\n")
    h0 = bench.kernel_sources_hash(["k.cu"])
    (tmp_path / "k.cu").write_text("// a different header\n\nint f(int x) { return x + 1; }\n")
    assert bench.kernel_sources_hash(["k.cu"]) == h0
    (tmp_path / "k.cu").write_text("int f(int x) { return x + 2; }\n")
    assert bench.kernel_sources_hash(["k.cu"]) != h0


def test_traffic_records_are_well_formed():
    path = os.path.join(os.path.dirname(bench.__file__), "profiles", "traffic.json")
    records = json.load(open(path))
    assert "packed_B256" in records
    for key, rec in records.items():
        assert rec["dram_bytes_per_launch"] > 0, key
        assert len(rec["sources_hash"]) == 16, key
        assert rec.get("command", "").lstrip().startswith("ncu ") or "phases" in rec, key


def test_cpu_model_is_described():
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()


def test_both_arms_name_the_same_packed_workload():
    """The GPU arm and the oracle arm describe the packed decode with one config: its text and
    sizes, and the state bytes of one step (read and written once)."""
    name, sizes = bench.packed_workload_config(256, 16, 32, 128, 128)
    assert "B=256" in name and "HV=32" in name and "K=V=128" in name and "f32 state" in name
    assert sizes["state_bytes_per_step"] == 2 * 256 * 32 * 128 * 128 * 4
    _, half = bench.packed_workload_config(256, 16, 32, 128, 128, "bf16")
    assert half["state_bytes_per_step"] * 2 == sizes["state_bytes_per_step"]


def test_oracle_baselines_of_the_buffered_and_fused_lines():
    """The buffered baseline runs whole L-step cycles (every phase equally often) and the fused one
    at least one call; both report a positive figure from one thread."""
    b = bench.cpu_baseline_buffered(2, 4, 16, 16, 4, seed=1, budget_s=0.05)
    assert b["value"] > 0 and b["kind"] == "oracle" and b["cores"] == 1
    assert "whole 4-step cycles" in b["sample"]
    f = bench.cpu_baseline_fused(4, 16, seed=1, budget_s=0.05)
    assert f["value"] > 0 and f["kind"] == "oracle" and "single-token" in f["sample"]


def test_oracle_baselines_of_the_mamba_and_projection_lines():
    m = bench.cpu_baseline_mamba(64, 16, seed=1, budget_s=0.05)
    assert m["value"] > 0 and m["kind"] == "oracle" and "single-row" in m["sample"]
    g = bench.cpu_baseline_gemv(2, 300, 128, seed=1, budget_s=0.05, rows=64)
    assert g["value"] > 0 and "64 of the 300 weight rows" in g["sample"]


def test_secondary_rows_cover_the_hot_path_rows_and_summarise():
    import bench
    names = [n for n, _ in bench.SECONDARY_ROWS]
    assert len(names) == len(set(names))
    workloads = {o["workload"] for _, o in bench.SECONDARY_ROWS}
    assert {"packed", "buffered", "fused", "stack", "mamba", "gemv", "front"} <= workloads
    line = {"config": {"workload": "w"}, "metric": "m", "value": 1.0, "unit": "GB/s",
            "us_per_step": 2.0, "roofline": {"frac": 0.5, "achieved": 3.0}, "per_layer_us": 4.0}
    s = bench.secondary_summary(line)
    assert s["roofline_frac"] == 0.5 and s["per_layer_us"] == 4.0 and s["us_per_call"] == 2.0
