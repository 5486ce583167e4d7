"""The bench's source fingerprint covers code, not comments: a captured DRAM-traffic figure
stays valid across comment edits and lapses on any change of code."""
import os

import bench


def _write(tmp, name, text):
    with open(os.path.join(tmp, name), "w", encoding="utf-8") as fh:
        fh.write(text)


def test_fingerprint_ignores_comments_and_blank_lines(tmp_path, monkeypatch):
    pkg = tmp_path / "persistent_gemm_tile_gb300"
    pkg.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    _write(pkg, "k.cuh", "int f(int x) {\n    return x + 1;  // one more\n}\n")
    base = bench.source_fingerprint(["k.cuh"])
    _write(pkg, "k.cuh", "// a new header comment\n\nint f(int x) {\n    return x + 1;  // reworded\n}\n")
    assert bench.source_fingerprint(["k.cuh"]) == base
    _write(pkg, "k.cuh", "int f(int x) {\n    return x + 2;  // one more\n}\n")
    assert bench.source_fingerprint(["k.cuh"]) != base
    assert len(base) == 16 and int(base, 16) >= 0


def test_traffic_lapses_when_code_changes(tmp_path, monkeypatch):
    pkg = tmp_path / "persistent_gemm_tile_gb300"
    pkg.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    _write(pkg, "k.cuh", "int g;\n")
    fp = bench.source_fingerprint(["k.cuh"])
    monkeypatch.setitem(bench.PROFILED_TRAFFIC, "probe", (123.0, ["k.cuh"], fp))
    assert bench.profiled_traffic("probe") == 123.0
    _write(pkg, "k.cuh", "int g;  // comment only\n")
    assert bench.profiled_traffic("probe") == 123.0
    _write(pkg, "k.cuh", "long g;\n")
    assert bench.profiled_traffic("probe") is None
