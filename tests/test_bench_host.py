"""Host-side logic of bench.py, without a GPU: the recorded DRAM traffic is tied
to the CUDA sources' hash and read from a machine-readable record, ncu CSV logs
are summed per step, and the reference arm (the oracle on host cores) prints one
JSON line with the contract's keys."""

import json
import os
import subprocess
import sys

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

NCU_CSV = """==PROF== Connected to process 1 (/usr/bin/python3)
"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size","Grid Size","Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"
"0","1","python3","h","void pkv_partial_kernel<4, 256, 256, 1, 1, 0, 0>(PartialParams, CUtensorMap_st, CUtensorMap_st)","1","7","(128, 1, 1)","(4, 8, 64)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","Mbyte","2,616.03"
"0","1","python3","h","void pkv_partial_kernel<4, 256, 256, 1, 1, 0, 0>(PartialParams, CUtensorMap_st, CUtensorMap_st)","1","7","(128, 1, 1)","(4, 8, 64)","0","10.3","Command line profiler metrics","dram__bytes_write.sum","byte","5222144"
"1","1","python3","h","pkv_merge_kernel(MergeParams)","1","7","(256, 1, 1)","(512, 1, 1)","0","10.3","Command line profiler metrics","dram__bytes_read.sum","byte","999"
"""


def test_recorded_traffic_follows_the_kernel_source_hash(monkeypatch):
    rows = json.load(open(bench.TRAFFIC_FILE))["rows"]
    assert rows, "profiles/dram_traffic.json has no rows"
    name, digest = rows[0]["workload"], rows[0]["kernel_sources"]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: digest)
    got = bench.recorded_traffic(name, "decode")
    assert got == rows[0]["dram_bytes"] and got > 0
    assert bench.recorded_traffic(name, "fused") is None  # only the decode call's partial pass is recorded
    assert bench.recorded_traffic("no_such_workload", "decode") is None
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: "0" * 16)  # sources changed since the capture
    assert bench.recorded_traffic(name, "decode") is None


def test_recorded_traffic_tolerates_a_missing_or_broken_record(tmp_path):
    assert bench.recorded_traffic("x", "decode", path=str(tmp_path / "none.json")) is None
    bad = tmp_path / "bad.json"
    bad.write_text("{not json")
    assert bench.recorded_traffic("x", "decode", path=str(bad)) is None
    bad.write_text('{"rows": [{"workload": "x", "kernel_sources": "y", "dram_bytes": "12"}]}')
    assert bench.recorded_traffic("x", "decode", path=str(bad)) is None


def test_ncu_csv_sums_the_partial_pass_only(tmp_path):
    p = tmp_path / "dram.csv"
    p.write_text(NCU_CSV)
    assert bench.ncu_dram_bytes([str(p)]) == 2616030000 + 5222144
    assert bench.ncu_dram_bytes([str(p), str(p)]) == 2 * (2616030000 + 5222144)


def test_record_traffic_writes_a_row_for_the_current_sources(tmp_path):
    p = tmp_path / "dram.csv"
    p.write_text(NCU_CSV)
    out = tmp_path / "traffic.json"
    row = bench.record_traffic("affine4_batch64_hq32_d256", [str(p)], path=str(out))
    assert row["kernel_sources"] == bench.kernel_source_hash() and row["dram_bytes"] == 2621252144
    assert row["algorithmic_bytes"] == 2612496384  # the seeded lengths x 8 KV heads x 2 x 144 B
    assert bench.recorded_traffic("affine4_batch64_hq32_d256", "decode", path=str(out)) == 2621252144
    bench.record_traffic("affine4_batch64_hq32_d256", [str(p), str(p)], path=str(out))  # replaces the row
    rows = json.load(open(out))["rows"]
    assert len(rows) == 1 and rows[0]["dram_bytes"] == 2 * 2621252144


def test_compute_dtype_names_the_products_of_each_page_format():
    assert "fp16" in bench.compute_dtype([4, 8]) and "bf16 tensor-core" not in bench.compute_dtype([4, 8])
    assert bench.compute_dtype([16]).startswith("bf16 pages: bf16 tensor-core products")


def test_default_workload_is_the_largest_configuration():
    from quantized_kv_decode_partial_gb300.workloads import draw_lengths, required_kv_bytes
    specs = bench.workload_specs(bench.DEFAULT_WORKLOAD)
    step = sum(required_kv_bytes(sp, draw_lengths(sp)) for sp in specs)
    assert len(specs) == 2 and step == 2612496384 + 4934715392


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
    assert d["impl"] == "reference" and d["value"] > 0 and d["config"]["workload"] == bench.DEFAULT_WORKLOAD
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_profiling_length_override_keeps_the_windowed_plan():
    # --seq-len lets the windowed workload's launch be captured from a smaller pool: with
    # lengths past the window the plan (and the rows read) are those of the full workload
    import ctypes

    from quantized_kv_decode_partial_gb300 import binding as B
    from quantized_kv_decode_partial_gb300.workloads import WORKLOADS
    sp = WORKLOADS["bf16_8x131072_n4_w8192_hq32_d128"]
    assert bench.parse_args(["--seq-len", "16384"]).seq_len == 16384
    lay = B.PoolLayout(1000, sp.num_kv_heads, sp.block_size, sp.head_dim, sp.bits, sp.group_size)
    plans = []
    for length in (sp.lengths[0], 16384):
        par = B.DecodeParams(sp.num_seqs, sp.num_q_heads, sp.n_query, length // sp.block_size, 0, sp.window)
        plan = B.Plan()
        assert B.load_library().pkv_make_plan(ctypes.byref(lay), ctypes.byref(par), 152, ctypes.byref(plan)) == 0
        plans.append((plan.partition_tokens, plan.max_partitions, plan.merge_in_cluster, plan.threads_per_cta,
                      plan.smem_bytes, plan.workspace_bytes))
    assert plans[0] == plans[1]
