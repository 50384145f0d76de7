"""Host logic of bench.py that needs no GPU: the DRAM traffic taken from a
committed capture is reported only while the kernel source and the workload
are those the capture was taken on."""
import hashlib
import json
import os
import sys
from types import SimpleNamespace

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _tree(tmp_path, source: bytes, recorded_sha: str, workload: str):
    csrc = tmp_path / "speculative_decoding_verification_42_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_bytes(source)
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({
        "k_x": {"source": "k.cu", "source_sha256": recorded_sha, "workload": workload,
                "dram_bytes_per_launch": 1234567}}))


def test_traffic_reported_for_the_captured_source_and_workload(tmp_path, monkeypatch):
    import bench
    src = b"__global__ void k_x() {}\n"
    _tree(tmp_path, src, hashlib.sha256(src).hexdigest(), "B=1 V=8")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._traffic("k_x", SimpleNamespace(name="B=1 V=8")) == 1234567.0


def test_traffic_null_once_the_source_changed(tmp_path, monkeypatch):
    import bench
    src = b"__global__ void k_x() {}\n"
    _tree(tmp_path, src + b"// edited\n", hashlib.sha256(src).hexdigest(), "B=1 V=8")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._traffic("k_x", SimpleNamespace(name="B=1 V=8")) is None


def test_traffic_null_for_another_workload_or_kernel(tmp_path, monkeypatch):
    import bench
    src = b"__global__ void k_x() {}\n"
    _tree(tmp_path, src, hashlib.sha256(src).hexdigest(), "B=1 V=8")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._traffic("k_x", SimpleNamespace(name="B=2 V=8")) is None
    assert bench._traffic("k_y", SimpleNamespace(name="B=1 V=8")) is None


def test_traffic_picks_the_record_of_the_workload(tmp_path, monkeypatch):
    import bench
    src = b"__global__ void k_x() {}\n"
    sha = hashlib.sha256(src).hexdigest()
    _tree(tmp_path, src, sha, "B=1 V=8")
    recs = [{"source": "k.cu", "source_sha256": sha, "workload": "B=1 V=8", "dram_bytes_per_launch": 10},
            {"source": "k.cu", "source_sha256": sha, "workload": "B=2 V=8", "dram_bytes_per_launch": 20}]
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"k_x": recs}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._traffic("k_x", SimpleNamespace(name="B=2 V=8")) == 20.0
    assert bench._traffic("k_x", SimpleNamespace(name="B=3 V=8")) is None


def test_committed_traffic_records_name_existing_sources():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        d = json.load(f)
    for kernel, recs in d.items():
        for e in (recs if isinstance(recs, list) else [recs]):
            path = os.path.join(ROOT, "speculative_decoding_verification_42_gb300", "csrc", e["source"])
            assert os.path.exists(path), kernel
            assert e["dram_bytes_per_launch"] > 0, kernel
