"""The committed DRAM-traffic entries (profiles/traffic.json) are used by the
benchmark only while the kernel source they were captured from is unchanged;
a changed source turns the figure into null rather than a stale number."""
import hashlib
import json
import os

import bench


def _tree(tmp_path, source_text, recorded_sha):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "k.cu").write_text(source_text)
    entry = {"source": "k.cu", "source_sha256_16": recorded_sha,
             "kernels": {"k": {"read": 1, "write": 2, "us": 3.0}}, "bytes_per_launch": 3}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"case": entry}))
    return entry


def test_entry_used_while_source_unchanged(tmp_path, monkeypatch):
    src = "// kernel\n"
    entry = _tree(tmp_path, src, hashlib.sha256(src.encode()).hexdigest()[:16])
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic("case") == entry
    assert bench.measured_traffic("missing") is None


def test_entry_dropped_once_source_changed(tmp_path, monkeypatch):
    _tree(tmp_path, "// kernel, edited\n", hashlib.sha256(b"// kernel\n").hexdigest()[:16])
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic("case") is None


def test_committed_entries_are_well_formed():
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        data = json.load(f)
    for key, e in data.items():
        if key == "note":
            continue
        assert os.path.exists(os.path.join(bench.ROOT, e["source"])), key
        assert len(e["source_sha256_16"]) == 16
        assert e["kernels"] and all(k["read"] > 0 and k["write"] > 0 for k in e["kernels"].values())
        assert e["bytes_per_launch"] > 0
