"""bench.py reports the ncu DRAM traffic of the dominant kernel only while the
kernel source is byte-identical to the one the counters were taken from, and
the figure comes from a machine-readable record that --ingest-ncu writes from
an ncu CSV (CPU)."""

import json

import bench

HEADER = ['"ID"', '"Kernel Name"', '"dram__bytes_read.sum"', '"dram__bytes_write.sum"']


def _setup(tmp_path, monkeypatch, source=b"// kernel\nint x;\n"):
    src = tmp_path / "gemm_tc.cu"
    src.write_bytes(source)
    rec = tmp_path / "ns_axpy_traffic.json"
    monkeypatch.setattr(bench, "KERNEL_SOURCE", str(src))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return src, rec


def _csv(tmp_path, rows, units=("", "", "Mbyte", "Mbyte")):
    lines = [",".join(HEADER), ",".join(f'"{u}"' for u in units)]
    lines += [",".join(f'"{v}"' for v in r) for r in rows]
    p = tmp_path / "raw.csv"
    p.write_text("\n".join(lines) + "\n")
    return str(p)


def test_ingest_averages_the_axpy_launches_and_guards_on_the_source(tmp_path, monkeypatch):
    src, rec = _setup(tmp_path, monkeypatch)
    csv_path = _csv(tmp_path, [
        ("1", "ns_gemm_kernel<0, false, false, 1, 1>(...)", "200.0", "35.0"),    # X X^T: ignored
        ("2", "ns_gemm_kernel<2, false, true, 1, 1>(...)", "415.946496", "306.739968"),
        ("3", "ns_gemm_kernel<2, false, true, 1, 1>(...)", "415.946496", "306.739968"),
    ])
    bench.ingest_ncu(csv_path, 8, "ncu ...")
    data = json.loads(rec.read_text())
    assert data["launches"] == 2 and data["matrices_per_launch"] == 8
    assert data["traffic_bytes_per_matrix"] == (415946496 + 306739968) // 8
    assert bench.axpy_traffic_per_matrix() == (415946496 + 306739968) // 8
    src.write_bytes(src.read_bytes() + b"// edited\n")   # any change to the kernel source
    assert bench.axpy_traffic_per_matrix() is None


def test_no_traffic_without_a_record(tmp_path, monkeypatch):
    _setup(tmp_path, monkeypatch)
    assert bench.axpy_traffic_per_matrix() is None


def test_byte_units_and_thousands_separators(tmp_path, monkeypatch):
    _, rec = _setup(tmp_path, monkeypatch)
    csv_path = _csv(tmp_path, [("1", "ns_gemm_kernel<2, false, false, 0, 0>(...)", "1,000", "600")],
                    units=("", "", "byte", "byte"))
    bench.ingest_ncu(csv_path, 2, "")
    assert json.loads(rec.read_text())["traffic_bytes_per_matrix"] == 800
