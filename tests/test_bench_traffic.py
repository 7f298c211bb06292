"""bench.py reports the dominant kernel's DRAM traffic from the committed ncu
summary only while the kernel source still hashes to the sha recorded there;
any other source gives null (the counters would describe another kernel)."""
import hashlib
import os

import bench


def _setup(tmp_path, src_text, sha, traffic="123456789"):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "gemm_tc_qwen3_8b_b1.md").write_text(
        "# summary\n<!-- kernel_sha: %s -->\n<!-- traffic_bytes_per_launch: %s -->\ntext\n"
        % (sha, traffic))
    src = tmp_path / "gemm_tc.cu"
    src.write_text(src_text)
    return str(src)


def _sha(text):
    return hashlib.sha256(text.encode()).hexdigest()[:16]


def test_traffic_reported_for_the_profiled_source(tmp_path, monkeypatch):
    src = _setup(tmp_path, "kernel v1\n", _sha("kernel v1\n"))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_from_profile(src) == 123456789.0


def test_traffic_null_once_the_source_changed(tmp_path, monkeypatch):
    src = _setup(tmp_path, "kernel v2\n", _sha("kernel v1\n"))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_from_profile(src) is None


def test_traffic_null_without_a_summary_or_a_number(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    src = tmp_path / "gemm_tc.cu"
    src.write_text("kernel v1\n")
    assert bench.traffic_from_profile(str(src)) is None
    os.remove(src)
    src = _setup(tmp_path, "kernel v1\n", _sha("kernel v1\n"), traffic="n/a")
    assert bench.traffic_from_profile(src) is None


def test_committed_summary_matches_its_recorded_format():
    # the committed summary carries both fields, the sha as 16 hex digits
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                        "profiles", "gemm_tc_qwen3_8b_b1.md")
    meta = {}
    for line in open(path):
        if line.startswith("<!-- ") and ":" in line:
            k, v = line[5:].split("-->")[0].split(":", 1)
            meta[k.strip()] = v.strip()
    assert len(meta["kernel_sha"]) == 16
    int(meta["kernel_sha"], 16)
    assert float(meta["traffic_bytes_per_launch"]) > 0
