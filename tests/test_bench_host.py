"""Host-side pieces of the benchmark (no GPU): the per-launch DRAM traffic
table that fills roofline.traffic only while the captured kernel is unchanged."""

import hashlib
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench_workloads  # noqa: E402


def _table(tmp_path, src_rel, digest, rd, wr):
    (tmp_path / "profiles").mkdir(exist_ok=True)
    (tmp_path / "profiles" / "traffic.md").write_text(
        "| key | source | sha256 | read bytes | write bytes | launch captured |\n"
        "|---|---|---|---|---|---|\n"
        f"| k1 | {src_rel} | {digest} | {rd} | {wr} | test |\n")


def test_traffic_follows_the_source_hash(tmp_path):
    src = tmp_path / "kern.cu"
    src.write_bytes(b"__global__ void k() {}\n")
    _table(tmp_path, "kern.cu", hashlib.sha256(src.read_bytes()).hexdigest(), 1000, 24)
    assert bench_workloads.traffic(str(tmp_path), "k1") == 1024
    assert bench_workloads.traffic(str(tmp_path), "missing") is None
    src.write_bytes(b"__global__ void k() { }\n")  # any edit voids the capture
    assert bench_workloads.traffic(str(tmp_path), "k1") is None
    os.remove(src)
    assert bench_workloads.traffic(str(tmp_path), "k1") is None


def test_committed_traffic_rows_are_well_formed():
    path = os.path.join(ROOT, "profiles", "traffic.md")
    rows = [r.split("|")[1:-1] for r in open(path).read().splitlines() if r.startswith("| ")]
    rows = [[c.strip() for c in r] for r in rows if r[0].strip() not in ("key",)]
    assert rows
    for key, src, digest, rd, wr, _ in rows:
        assert os.path.exists(os.path.join(ROOT, src)), src
        assert len(digest) == 64 and int(digest, 16) >= 0
        assert int(rd) >= 0 and int(wr) >= 0
