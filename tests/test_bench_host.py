"""Host-side pieces of the benchmark (no GPU): the per-launch DRAM traffic
table that fills roofline.traffic only while the captured kernel is unchanged."""

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench_workloads  # noqa: E402


def _table(tmp_path, src_rel, digest, rd, wr):
    (tmp_path / "profiles").mkdir(exist_ok=True)
    row = {"key": "k1", "source": src_rel, "code_digest": digest, "read_bytes": rd, "write_bytes": wr,
           "launch": "test", "command": "none"}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"about": "test", "rows": [row]}))


def test_traffic_follows_the_code_digest(tmp_path):
    src = tmp_path / "kern.cu"
    src.write_text("// kernel\n__global__ void k(int* p) { p[0] = 1; }\n")
    _table(tmp_path, "kern.cu", bench_workloads.code_digest(src.read_text()), 1000, 24)
    assert bench_workloads.traffic(str(tmp_path), "k1") == 1024
    assert bench_workloads.traffic(str(tmp_path), "missing") is None
    # comments and layout do not change the code
    src.write_text("/* the kernel, one store */\n__global__ void k(int* p) {\n  p[0] = 1;  // one\n}\n")
    assert bench_workloads.traffic(str(tmp_path), "k1") == 1024
    src.write_text("__global__ void k(int* p) { p[0] = 2; }\n")  # a code edit voids the capture
    assert bench_workloads.traffic(str(tmp_path), "k1") is None
    os.remove(src)
    assert bench_workloads.traffic(str(tmp_path), "k1") is None


def test_code_digest_keeps_literals():
    d = bench_workloads.code_digest
    assert d('asm("a // b");') != d('asm("a");')  # a comment marker inside a literal is code
    assert d("x = '/'; // c\ny = 1;") == d("x = '/';\ny = 1;")
    assert d("a /* c */ + b") == d("a + b") and d("a + b") != d("a - b")


def test_committed_traffic_rows_are_well_formed():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rows = json.load(f)["rows"]
    assert rows
    keys = [r["key"] for r in rows]
    assert len(set(keys)) == len(keys)
    for r in rows:
        assert os.path.exists(os.path.join(ROOT, r["source"])), r["source"]
        assert len(r["code_digest"]) == 64 and int(r["code_digest"], 16) >= 0
        assert int(r["read_bytes"]) >= 0 and int(r["write_bytes"]) >= 0
        assert r["command"].startswith("ncu ") and "--clock-control none" in r["command"]


def test_reference_arm_prints_one_contract_line():
    """bench.py --impl reference: the oracle on the host cores, one JSON line
    with the contract's keys and the library arm's metric and workload."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    j = json.loads(lines[0])
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in j, k
    assert j["impl"] == "reference" and j["metric"] == "decode-attn HBM GB/s" and j["unit"] == "GB/s"
    assert j["higher_is_better"] is True and j["steps"] == 1 and j["warmup"] == 3 and j["value"] > 0
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["cores"] >= 1
    assert j["cpu_baseline"]["value"] == j["value"] and j["e2e"]["value"] == j["value"]
    assert j["e2e"]["h2d_bytes_per_step"] == 0 and j["e2e"]["d2h_bytes_per_step"] == 0
    assert j["config"]["workload"].startswith("decode attention, 1 layer, batch 1, 32 q / 8 kv heads, head_dim 128, "
                                              "seq 16384, K/V TurboQuant_MSE b=4")
