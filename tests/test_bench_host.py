"""Host-side logic of bench.py, without a GPU: the recorded DRAM traffic is tied
to the CUDA sources' hash, and the reference arm (the oracle on host cores)
prints one JSON line with the contract's keys."""

import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_recorded_traffic_follows_the_kernel_source_hash(monkeypatch):
    rows = [line for line in open(bench.TRAFFIC_FILE) if line.startswith("| ") and "`" in line]
    assert rows, "profiles/dram_traffic.md has no rows"
    name, digest = rows[0].split("|")[1].strip(), rows[0].split("`")[1]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: digest)
    got = bench.recorded_traffic(name, "decode")
    assert isinstance(got, int) and got > 0
    assert bench.recorded_traffic(name, "fused") is None  # only the decode call's partial pass is recorded
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)  # sources changed since the capture
    assert bench.recorded_traffic(name, "decode") is None


def test_kernel_source_hash_is_stable():
    a, b = bench.kernel_source_hash(), bench.kernel_source_hash()
    assert a == b and len(a) == 16 and int(a, 16) >= 0


def test_reference_arm_prints_one_contract_line():
    res = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                         cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [line for line in res.stdout.splitlines() if line.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["config"]["workload"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
