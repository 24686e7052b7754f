"""Host-side bookkeeping of bench.py (no GPU): the DRAM-traffic records it
reports are keyed by a hash of each kernel's source and headers, and every
record names a kernel bench.py knows and a profile summary that exists."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


@pytest.fixture(scope="module")
def bench():
    argv = sys.argv
    sys.argv = ["bench.py"]
    try:
        import bench as b
    finally:
        sys.argv = argv
    return b


def test_source_hash_covers_included_headers(bench, tmp_path, monkeypatch):
    csrc = tmp_path / "invariant_bi_rmsnorm_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "include").mkdir()
    (csrc / "k.cu").write_text('#include "h.cuh"\nint k;\n')
    (csrc / "h.cuh").write_text("int h = 1;\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    a = bench.kernel_source_sha("k.cu")
    assert a == bench.kernel_source_sha("k.cu")  # deterministic
    (csrc / "h.cuh").write_text("int h = 2;\n")
    assert bench.kernel_source_sha("k.cu") != a  # a header edit changes the hash


def test_traffic_records_are_well_formed(bench):
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    seen = set()
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        kernel, sha, nbytes = line.split()[:3]
        assert kernel in bench.KERNEL_SOURCES, kernel
        assert len(sha) == 16 and int(sha, 16) >= 0
        assert int(nbytes) > 0
        for ref in (w.strip("(),;") for w in line.split() if w.strip("(),;").startswith("profiles/")):
            assert os.path.exists(os.path.join(ROOT, ref)), ref
        assert kernel not in seen, f"{kernel} recorded twice"
        seen.add(kernel)
    assert {"bi_gemm", "bi_decode_attention", "bi_rmsnorm"} <= seen


def test_traffic_record_only_for_matching_source(bench, monkeypatch):
    kernel = "bi_rmsnorm"
    current = bench.traffic_record(kernel)
    monkeypatch.setattr(bench, "kernel_source_sha", lambda src: "0" * 16)
    assert bench.traffic_record(kernel) is None  # a stale capture is not reported
    assert current is None or current > 0
