"""bench.py's per-launch DRAM traffic lookup (CPU only).

The bench line's roofline.traffic comes from a committed ncu summary, but only while the
kernel's source files are the ones the counters were taken on. A changed kernel gives null
rather than a stale number. These tests run the lookup on files written to a temporary root,
and check the format of the committed summaries.
"""
import glob
import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _write_profile(root, digest, traffic="123456789", files="src/k.cu, src/p.cuh"):
    os.makedirs(os.path.join(root, "profiles"), exist_ok=True)
    with open(os.path.join(root, "profiles", "kern_work_traffic.txt"), "w") as f:
        f.write("# DRAM traffic of one launch (test fixture)\n")
        f.write(f"source_files: {files}\n")
        f.write(f"source_sha256_16: {digest}\n")
        f.write(f"traffic_bytes_per_launch: {traffic}\n")


def _write_sources(root, text_k="kernel v1", text_p="header v1"):
    os.makedirs(os.path.join(root, "src"), exist_ok=True)
    with open(os.path.join(root, "src", "k.cu"), "w") as f:
        f.write(text_k)
    with open(os.path.join(root, "src", "p.cuh"), "w") as f:
        f.write(text_p)


def test_matching_digest_gives_traffic(bench, tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    _write_sources(tmp_path)
    _write_profile(tmp_path, bench.source_digest(["src/k.cu", "src/p.cuh"]))
    assert bench.traffic_from_profile("kern", "work") == 123456789.0


@pytest.mark.parametrize("which", ["kernel", "header"])
def test_changed_source_gives_none(bench, tmp_path, monkeypatch, which):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    _write_sources(tmp_path)
    _write_profile(tmp_path, bench.source_digest(["src/k.cu", "src/p.cuh"]))
    if which == "kernel":
        _write_sources(tmp_path, text_k="kernel v2")
    else:
        _write_sources(tmp_path, text_p="header v2")
    assert bench.traffic_from_profile("kern", "work") is None


def test_missing_or_malformed_gives_none(bench, tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.traffic_from_profile("kern", "work") is None  # no summary
    _write_sources(tmp_path)
    digest = bench.source_digest(["src/k.cu", "src/p.cuh"])
    _write_profile(tmp_path, digest, traffic="n/a")
    assert bench.traffic_from_profile("kern", "work") is None  # not a number
    _write_profile(tmp_path, digest, files="src/k.cu, src/gone.cuh")
    assert bench.traffic_from_profile("kern", "work") is None  # a listed source is missing


def test_digest_depends_on_file_order_and_content(bench, tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    _write_sources(tmp_path)
    a = bench.source_digest(["src/k.cu", "src/p.cuh"])
    assert len(a) == 16 and all(c in "0123456789abcdef" for c in a)
    assert bench.source_digest(["src/p.cuh", "src/k.cu"]) != a
    _write_sources(tmp_path, text_k="kernel v1 ")
    assert bench.source_digest(["src/k.cu", "src/p.cuh"]) != a


def test_committed_summaries_are_well_formed():
    found = sorted(glob.glob(os.path.join(ROOT, "profiles", "*_traffic.txt")))
    assert found, "the bench's roofline traffic needs committed summaries"
    for path in found:
        vals = {}
        for line in open(path):
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
        files = [f.strip() for f in vals["source_files"].split(",")]
        assert files and all(os.path.exists(os.path.join(ROOT, f)) for f in files), path
        assert len(vals["source_sha256_16"]) == 16, path
        assert int(vals["traffic_bytes_per_launch"]) > 0, path
        assert "ncu " in open(path).read() and "--clock-control none" in open(path).read(), path
