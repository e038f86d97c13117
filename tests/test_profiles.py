"""The committed ncu records under profiles/ are well formed: each names the kernel
source files its hash covers (all present in the package), the capture command,
and DRAM bytes that add up.  bench.py reports a record's traffic only while those
files still hash to the recorded value."""
import glob
import hashlib
import json
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "moe_gemm_exl3_gb300", "csrc")
RECORDS = sorted(glob.glob(os.path.join(ROOT, "profiles", "*.json")))


def test_records_exist():
    assert RECORDS, "no ncu records under profiles/"


@pytest.mark.parametrize("path", RECORDS, ids=[os.path.basename(p) for p in RECORDS])
def test_record_fields(path):
    with open(path) as f:
        d = json.load(f)
    assert d["source_files"], "a record must list the sources its hash covers"
    for s in d["source_files"]:
        assert os.path.exists(os.path.join(CSRC, s)), s
    assert len(d["source_sha256_16"]) == 16
    assert d["dram_bytes_per_launch"] == d["dram_bytes_read"] + d["dram_bytes_write"]
    assert "ncu" in d["command"] and "--clock-control none" in d["command"]


def test_bench_reads_a_record_only_while_its_sources_match(tmp_path, monkeypatch):
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    src = tmp_path / "moe_gemm_exl3_gb300" / "csrc"
    src.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (src / "k.cu").write_bytes(b"kernel v1")
    rec = {"source_files": ["k.cu"], "dram_bytes_per_launch": 123,
           "source_sha256_16": hashlib.sha256(b"kernel v1").hexdigest()[:16]}
    (tmp_path / "profiles" / "k.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profile_traffic("k.json") == 123
    (src / "k.cu").write_bytes(b"kernel v2")
    assert bench.profile_traffic("k.json") is None
    assert bench.profile_traffic("missing.json") is None
