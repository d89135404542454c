"""bench.py's host-side logic (no GPU): the DRAM-traffic record is used only
when it was taken on the current kernel sources, workload and step, and
the peak denominators come from MEASURED_PEAKS.json when it is present."""
import hashlib
import json
import os
import shutil

import pytest

import bench

KERNEL = os.path.join(bench.ROOT, "paged_kv_cache_309_gb300", "csrc", "decode.cu")
HEADER = os.path.join(bench.ROOT, "paged_kv_cache_309_gb300", "csrc", "pa_internal.cuh")


def _sources_hash():
    hs = hashlib.sha256()
    for p in (KERNEL, HEADER):
        with open(p, "rb") as f:
            hs.update(f.read())
    return hs.hexdigest()[:16]


@pytest.fixture
def root(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def _write_record(root, **kw):
    rec = dict(workload="long_context_decode_b8_ctx32k-128k_bs16", step="fused", kv_dtype="bf16",
               source_sha256_16=_sources_hash(), dram_bytes_per_decode_call=1234)
    rec.update(kw)
    (root / "profiles" / "decode_traffic.json").write_text(json.dumps(rec))


def test_traffic_used_when_sources_workload_and_step_match(root):
    _write_record(root)
    assert bench.traffic_record(KERNEL, "long_context_decode_b8_ctx32k-128k_bs16", "fused",
                                "bf16") == 1234


@pytest.mark.parametrize("change", [dict(source_sha256_16="0" * 16),
                                    dict(workload="other"), dict(step="two-call"),
                                    dict(kv_dtype="e4m3")])
def test_traffic_null_when_anything_differs(root, change):
    _write_record(root, **change)
    assert bench.traffic_record(KERNEL, "long_context_decode_b8_ctx32k-128k_bs16", "fused",
                                "bf16") is None


def test_traffic_null_when_a_hashed_source_changes(root, tmp_path):
    _write_record(root)
    src = tmp_path / "csrc"
    src.mkdir()
    shutil.copy(KERNEL, src / "decode.cu")
    shutil.copy(HEADER, src / "pa_internal.cuh")
    with open(src / "pa_internal.cuh", "a") as f:
        f.write("\n// edited\n")
    assert bench.traffic_record(str(src / "decode.cu"), "long_context_decode_b8_ctx32k-128k_bs16",
                                "fused", "bf16") is None


def test_traffic_null_without_a_record(root):
    assert bench.traffic_record(KERNEL, "long_context_decode_b8_ctx32k-128k_bs16", "fused",
                                "bf16") is None


def test_committed_records_name_their_hashed_sources():
    with open(os.path.join(bench.ROOT, "profiles", "decode_traffic.json")) as f:
        d = json.load(f)
    assert d["hashed_sources"] == ["paged_kv_cache_309_gb300/csrc/decode.cu",
                                   "paged_kv_cache_309_gb300/csrc/pa_internal.cuh"]
    assert d["records"]
    keys = set()
    for rec in d["records"]:
        assert rec["dram_bytes_per_decode_call"] == rec["dram_bytes_read"] + rec["dram_bytes_write"]
        assert "--clock-control none" in rec["command"]
        key = (rec["workload"], rec["step"], rec["kv_dtype"])
        assert key not in keys  # one record per workload, step and KV format
        keys.add(key)


def test_traffic_picks_the_matching_record(root):
    recs = [dict(workload=f"w{i}", step="fused", kv_dtype=k, source_sha256_16=_sources_hash(),
                 dram_bytes_per_decode_call=100 + i) for i, k in enumerate(["bf16", "e4m3"])]
    (root / "profiles" / "decode_traffic.json").write_text(json.dumps({"records": recs}))
    assert bench.traffic_record(KERNEL, "w1", "fused", "e4m3") == 101
    assert bench.traffic_record(KERNEL, "w0", "fused", "bf16") == 100
    assert bench.traffic_record(KERNEL, "w1", "fused", "bf16") is None


def test_peak_from_measured_file_else_fallback(root):
    assert bench.hbm_peak() == (bench.FALLBACK_HBM_GBS, "fallback")
    (root / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6677.5}))
    assert bench.hbm_peak() == (6677.5, "measured")


def test_host_cpu_reports_model_and_cores():
    h = bench.host_cpu()
    assert h["nproc"] >= 1 and isinstance(h["cpu_model"], str) and h["cpu_model"]
