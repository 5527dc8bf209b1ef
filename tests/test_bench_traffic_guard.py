"""bench.py reports the ncu DRAM traffic of the dominant kernel only while the
kernel source is byte-identical to the one the counters were taken from (CPU)."""

import hashlib
import os

import bench

SRC = os.path.join("muon_newton_schulz_expert_gb300", "csrc", "gemm_tc.cu")
PROF = os.path.join("profiles", "ns_gemm_kernels_profile8.md")


def _tree(tmp_path, source, profile_lines):
    (tmp_path / SRC).parent.mkdir(parents=True)
    (tmp_path / SRC).write_bytes(source)
    (tmp_path / PROF).parent.mkdir(parents=True)
    (tmp_path / PROF).write_text("# summary\n\nsome: text\n" + "\n".join(profile_lines) + "\n")


def test_traffic_only_for_the_captured_source(tmp_path, monkeypatch):
    source = b"// kernel\nint x;\n"
    sha = hashlib.sha256(source).hexdigest()
    _tree(tmp_path, source, ["traffic_kernel: ns_axpy_tc", "traffic_bytes_per_matrix: 90335808",
                             f"source_sha256: {sha}"])
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.axpy_traffic_per_matrix() == 90335808
    (tmp_path / SRC).write_bytes(source + b"// edited\n")   # any change to the source
    assert bench.axpy_traffic_per_matrix() is None


def test_no_traffic_without_a_recorded_figure(tmp_path, monkeypatch):
    source = b"int y;\n"
    _tree(tmp_path, source, [f"source_sha256: {hashlib.sha256(source).hexdigest()}"])
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.axpy_traffic_per_matrix() is None
    (tmp_path / PROF).unlink()
    assert bench.axpy_traffic_per_matrix() is None
