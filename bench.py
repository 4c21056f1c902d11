"""Benchmark of paged decode attention on GB300: K/V GB/s, decode steps/s and the
fraction of the measured HBM roofline.

One step = one decode call (partial pass + merge pass) over every sequence of the
workload; a two-layer workload (4-bit + 8-bit pages) runs both layers per step.
Inputs are seeded synthetic data of the workload's shapes and length mix, already
resident in HBM when the timed region starts. Workloads whose inputs are smaller
than 3x the L2 cache rotate through enough independent input copies that every
timed step reads from HBM. Steps are recorded once into a CUDA graph and the
graph is replayed; time comes from CUDA events on the launching stream.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own instance of the workload (weak
scaling: sequences are independent, there is no exchange between GPUs); the time
is the maximum over ranks and the value counts every rank's bytes.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode attention K/V GB/s and steps/s; % of GB300 HBM roofline"
# The largest single-GPU configuration: 64 sequences of 1024-32768 rows, HQ=32 HK=8
# D=256, one 4-bit and one 8-bit affine layer per step (7.55 GB of K/V per step).
DEFAULT_WORKLOAD = "affine_batch64_hq32_d256"
FALLBACK_HBM_GBS = 6800.0


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the CPU oracle sample")
    ap.add_argument("--profile-calls", type=int, default=0,
                    help="profiling mode: make the workload, run this many eager decode calls, exit")
    ap.add_argument("--num-seqs", type=int, default=0,
                    help="profiling mode: keep only the first N sequences of the workload")
    ap.add_argument("--seq-len", type=int, default=0,
                    help="profiling mode: give every kept sequence this length (with a window shorter than it, "
                         "the kernels read the same rows from a smaller pool)")
    ap.add_argument("--partition-tokens", type=int, default=-2,
                    help="rows per partition instead of the workload's choice (0: the library's plan)")
    ap.add_argument("--print-kernel-hash", action="store_true",
                    help="print the hash of the CUDA sources that profiles/dram_traffic.json rows refer to, and exit")
    ap.add_argument("--record-traffic", nargs="+", metavar="NCU_CSV",
                    help="store the DRAM bytes of one step of --workload, summed over these ncu CSV logs, in "
                         "profiles/dram_traffic.json for the current kernel sources, and exit")
    ap.add_argument("--schedule", choices=["auto", "partitions", "balanced"], default="auto",
                    help="how rows are split over the CTAs: the library's choice, partitions of every (sequence, KV "
                         "head), or equal runs of the whole chunk list (pkv_decode_params.schedule)")
    ap.add_argument("--contraction", choices=["auto", "tensor", "cuda_core"], default="auto",
                    help="the contraction the kernels run: the library's choice, tensor-core MMA, or per-lane "
                         "f32 FMAs with warp-shuffle reductions (bf16 pages, at most 4 query rows per KV head)")
    ap.add_argument("--step", choices=["decode", "fused"], default="decode",
                    help="decode: the decode call; fused: the decode step with its write "
                         "(pkv_paged_decode_append_attention: append the N new K/V rows, then attend)")
    return ap.parse_args(argv)


CONTRACTIONS = {"auto": 0, "tensor": 1, "cuda_core": 2}
SCHEDULES = {"auto": 0, "partitions": 1, "balanced": 2}


def workload_specs(name):
    from quantized_kv_decode_partial_gb300.workloads import LAYER_GROUPS, WORKLOADS
    if name in LAYER_GROUPS:
        return [WORKLOADS[n] for n in LAYER_GROUPS[name]]
    if name not in WORKLOADS:
        raise SystemExit(f"unknown workload {name}; choose from {sorted(WORKLOADS) + sorted(LAYER_GROUPS)}")
    return [WORKLOADS[name]]


def kernel_source_hash():
    """Hash of the CUDA sources' code (comments and blank lines left out): DRAM traffic
    recorded for one version of the kernels applies to that version only."""
    import hashlib
    import re
    csrc = os.path.join(ROOT, "quantized_kv_decode_partial_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)  # the sources hold no "//" or "/*" in strings
            lines = [re.sub(r"//.*", "", line).rstrip() for line in text.splitlines()]
            code = "\n".join(line for line in lines if line)
            h.update(name.encode() + b"\0" + code.encode())
    return h.hexdigest()[:16]


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")


def recorded_traffic(workload, step, path=TRAFFIC_FILE):
    """DRAM bytes (read + write) of the partial-pass launches of one step, from the ncu
    capture recorded in profiles/dram_traffic.json for the current kernel sources, or None
    (no capture, or the kernels changed since)."""
    if step != "decode":
        return None
    try:
        with open(path) as f:
            rows = json.load(f)["rows"]
    except (OSError, ValueError, KeyError, TypeError):
        return None
    want = kernel_source_hash()
    for row in rows if isinstance(rows, list) else []:
        if isinstance(row, dict) and row.get("workload") == workload and row.get("kernel_sources") == want:
            value = row.get("dram_bytes")
            return int(value) if isinstance(value, int) and value > 0 else None
    return None


NCU_UNITS = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "Tbyte": 1e12}


def ncu_dram_bytes(csv_paths):
    """DRAM bytes read + written by the partial-pass launches in ncu CSV logs
    (``--metrics dram__bytes_read.sum,dram__bytes_write.sum --csv --log-file``)."""
    import csv
    total = 0.0
    for path in csv_paths:
        with open(path) as f:
            lines = [line for line in f if line.startswith('"')]
        for row in csv.DictReader(lines):
            if "pkv_partial" not in row.get("Kernel Name", ""):
                continue
            if row.get("Metric Name") in ("dram__bytes_read.sum", "dram__bytes_write.sum"):
                total += float(row["Metric Value"].replace(",", "")) * NCU_UNITS[row["Metric Unit"]]
    return int(round(total))


def record_traffic(workload, csv_paths, path=TRAFFIC_FILE):
    """Stores the DRAM bytes of one step of `workload` (the sum over the given ncu logs,
    one per layer) for the current kernel sources in profiles/dram_traffic.json."""
    from quantized_kv_decode_partial_gb300.workloads import draw_lengths, required_kv_bytes
    dram = ncu_dram_bytes(csv_paths)
    if dram <= 0:
        raise SystemExit(f"no pkv_partial DRAM metrics in {csv_paths}")
    algo = sum(required_kv_bytes(sp, draw_lengths(sp)) for sp in workload_specs(workload))
    try:
        with open(path) as f:
            doc = json.load(f)
    except (OSError, ValueError):
        doc = {}
    rows = [r for r in doc.get("rows", []) if r.get("workload") != workload]
    rows.append({"workload": workload, "kernel_sources": kernel_source_hash(), "dram_bytes": dram,
                 "algorithmic_bytes": algo, "ratio": round(dram / algo, 4)})
    doc = {"what": "DRAM bytes read + written by the partial-pass launches of one decode step (ncu "
                   "dram__bytes_read.sum + dram__bytes_write.sum, one capture per layer, each launch "
                   "profiled in one pass), for the CUDA sources whose hash is kernel_sources",
           "rows": sorted(rows, key=lambda r: r["workload"])}
    with open(path, "w") as f:
        json.dump(doc, f, indent=1)
        f.write("\n")
    return rows[-1]


def compute_dtype(bits_list, contractions=None):
    """The arithmetic the timed kernels run, per page format (and contraction) of the
    step's layers."""
    names = []
    for i, bits in enumerate(bits_list):
        cuda_cores = contractions is not None and contractions[i] == 2
        name = ("bf16 pages: f32 FMAs on CUDA cores (f32 products of bf16 values)" if cuda_cores else
                "bf16 pages: bf16 tensor-core products" if bits == 16 else
                f"{bits}-bit affine pages: fp16 tensor-core products on exact-subnormal codes")
        if name not in names:
            names.append(name)
    return "; ".join(names) + "; f32 softmax and accumulation; bf16 output"


def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class NvmlClockPoller:
    """Reads the SM clock and the clock-event reasons through NVML (the driver's
    libnvidia-ml, read-only calls) every few milliseconds in a thread, so that a timed
    region of a few tens of milliseconds still gets many samples."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, torch_device, period_s=0.002):
        import ctypes
        import threading
        self.samples = []
        self.period = period_s
        self._stop = threading.Event()
        self._thread = None
        self.handle = None
        self.max_mhz = None
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            handle = ctypes.c_void_p()
            uuid = None
            try:
                import torch
                uuid = str(torch.cuda.get_device_properties(torch_device).uuid)
            except Exception:
                uuid = None
            ok = False
            if uuid:
                ok = self.nvml.nvmlDeviceGetHandleByUUID(("GPU-" + uuid).encode(), ctypes.byref(handle)) == 0
            if not ok:
                ok = self.nvml.nvmlDeviceGetHandleByIndex_v2(int(torch_device.index or 0), ctypes.byref(handle)) == 0
            if not ok:
                return
            self.handle = handle
            mx = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
        except OSError:
            self.handle = None

    def _read(self):
        import ctypes
        clk = ctypes.c_uint()
        reasons = ctypes.c_ulonglong()
        if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(clk)) != 0:
            return None
        fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        if fn(self.handle, ctypes.byref(reasons)) != 0:
            reasons.value = 0
        return float(clk.value), int(reasons.value)

    def _run(self):
        while not self._stop.is_set():
            r = self._read()
            if r is not None:
                self.samples.append(r)
            self._stop.wait(self.period)

    def start(self):
        if self.handle is None:
            return
        import threading
        self._thread = threading.Thread(target=self._run, daemon=True)
        self._thread.start()

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)
        reasons = set()
        for _, bits in self.samples:
            for bit, name in self.REASONS.items():
                if bits & bit:
                    reasons.add(name)
        return [mhz for mhz, _ in self.samples], sorted(reasons)


class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, torch_device=None):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.poller = NvmlClockPoller(torch_device) if torch_device is not None else None

    def _once(self):
        try:
            out = subprocess.run(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                  "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=20)
            return out.stdout.strip().splitlines()
        except (OSError, subprocess.SubprocessError):
            return []

    def start(self):
        self.lines = self._once()
        if self.poller is not None:
            self.poller.start()
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100", "-f", self.path],
                                         stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        self.nvml = self.poller.stop() if self.poller is not None else ([], [])
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=10)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            try:
                with open(self.path) as f:
                    self.lines += f.read().strip().splitlines()
            except OSError:
                pass
        self.lines += self._once()
        if self.path and os.path.exists(self.path):
            os.unlink(self.path)
        return self.summary()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower() == "active":
                    reasons.add(name)
        nvml_mhz, nvml_reasons = getattr(self, "nvml", ([], []))
        reasons.update(nvml_reasons)
        if nvml_mhz:  # NVML polled every few ms during the timed region: the denser record
            mx_nvml = self.poller.max_mhz or (max(mx) if mx else None)
            return {"sm_mhz": statistics.median(nvml_mhz), "sm_max_mhz": mx_nvml, "reasons": sorted(reasons),
                    "samples": len(nvml_mhz), "sm_mhz_min": min(nvml_mhz),
                    "source": "NVML every 2 ms during the timed region (plus nvidia-smi every 100 ms: "
                              f"{len(sm)} samples, reasons included)"}
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "source": "nvidia-smi every 100 ms during the timed region"}


# ---------------------------------------------------------------------------
# the CPU oracle baseline (bounded sample, one thread, in a child process)
# ---------------------------------------------------------------------------

CPU_CHILD = r"""
import json, os, sys, time
from dataclasses import replace
sys.path.insert(0, {root!r})
import torch
torch.set_num_threads(1)
import oracle
from quantized_kv_decode_partial_gb300.workloads import WORKLOADS, draw_lengths, make_case, required_kv_bytes
# One (sequence, KV head) unit of each layer: the first sequence of the seeded
# length draw, with its REP query heads. Every unit of a workload costs the same
# per cached row, so the rate of one unit is the rate of the workload.
units = []
for name in {names!r}:
    spec = WORKLOADS[name]
    lens = draw_lengths(spec, {seed})
    unit = replace(spec, name=name + "_unit", num_seqs=1, num_kv_heads=1, num_q_heads=spec.rep,
                   lengths=(lens[0],), length_range=None, pool_factor=1.0)
    case = make_case(unit, device="cpu", seed={seed})
    f64 = lambda t: None if t is None else t.float().double().numpy()
    kw = dict(bits=unit.bits, group_size=unit.group_size)
    if unit.bits == 16:
        kp, vp = f64(case.k_pool), f64(case.v_pool)
    else:
        kp, vp = case.k_pool.numpy(), case.v_pool.numpy()
        kw.update(k_scales=f64(case.k_scales), k_biases=f64(case.k_biases), v_scales=f64(case.v_scales),
                  v_biases=f64(case.v_biases))
    args = (f64(case.q), kp, vp, case.block_tables.numpy(), case.seq_lens.numpy(), case.scale, unit.n_query)
    units.append((name, args, kw, required_kv_bytes(unit, case.lens_host), case.lens_host[0]))
steps = []
for _ in range({steps}):
    t_start = time.perf_counter()
    done, secs, count = 0, 0.0, 0
    while True:
        for name, args, kw, nbytes, L in units:
            t0 = time.perf_counter()
            oracle.paged_decode_attention(*args, **kw)
            secs += time.perf_counter() - t0
            done += nbytes
        count += 1
        if time.perf_counter() - t_start >= {budget}:
            break
    steps.append({{"bytes": done, "seconds": secs, "repeats": count}})
sample = "; ".join(f"{{n}}: 1 sequence x 1 KV head ({{L}} rows, {{nb}} K/V bytes)" for n, _, _, nb, L in units)
print(json.dumps({{"steps": steps, "sample": sample}}))
"""


def cpu_oracle_baseline(names, seed, budget_s, steps=1):
    """The oracle on a bounded sample of the workload, one thread, in a child
    process (started before or apart from any GPU work). Returns per-step rates."""
    code = CPU_CHILD.format(root=ROOT, budget=budget_s, names=list(names), seed=seed, steps=steps)
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                         timeout=max(900, 3 * steps * budget_s + 300))
    if res.returncode != 0:
        raise RuntimeError(f"CPU oracle failed:\n{res.stderr[-2000:]}")
    info = json.loads(res.stdout.strip().splitlines()[-1])
    tot_b = sum(s["bytes"] for s in info["steps"])
    tot_s = sum(s["seconds"] for s in info["steps"])
    return {"value": tot_b / tot_s / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": info["sample"] + f"; {tot_b} K/V bytes in {tot_s:.2f} s on one thread",
            "steps": info["steps"], "bytes": tot_b, "seconds": tot_s}


# ---------------------------------------------------------------------------
# reference arm: the oracle, timed on the host cores
# ---------------------------------------------------------------------------

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    specs = workload_specs(args.workload)
    names = [s.name for s in specs]
    per_step = min(2.0, max(0.05, 120.0 / max(1, args.steps + args.warmup)))
    r = cpu_oracle_baseline(names, specs[0].seed, per_step, steps=args.warmup + args.steps)
    timed = r["steps"][args.warmup:]
    tot_b = sum(s["bytes"] for s in timed)
    tot_s = sum(s["seconds"] for s in timed)
    value = tot_b / tot_s / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_s / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload,
                   "sample": f"each step repeats the oracle on the sample for about {per_step:.2f} s"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": r["sample"]},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args):
    from dataclasses import replace

    import torch
    import torch.distributed as dist

    from quantized_kv_decode_partial_gb300 import (DecodeParams, load_library, make_plan, paged_decode_attention,
                                                   paged_decode_append_attention, paged_decode_passes,
                                                   HostDecodeStep)
    from quantized_kv_decode_partial_gb300 import build as pkv_build
    from quantized_kv_decode_partial_gb300.binding import layout_for
    from quantized_kv_decode_partial_gb300.workloads import make_case, required_kv_bytes

    from quantized_kv_decode_partial_gb300.dist import max_over_ranks, rank_seed, weak_scaling_rate, world as env_world

    rank, world, local = env_world()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pkv_build.build()
    load_library()

    # CPU baseline first, in a child process, before this process does GPU work.
    specs = workload_specs(args.workload)
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_oracle_baseline([s.name for s in specs], specs[0].seed, args.cpu_seconds)

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    layers = []
    for sp in specs:
        if args.partition_tokens != -2:
            sp = replace(sp, partition_tokens=args.partition_tokens)
        base = make_case(sp, device=dev, seed=rank_seed(sp.seed, rank), poison=False)
        in_bytes = sum(t.numel() * t.element_size() for t in
                       (base.q, base.k_pool, base.v_pool, base.k_scales, base.k_biases, base.v_scales, base.v_biases,
                        base.block_tables, base.seq_lens) if t is not None)
        copies = max(1, math.ceil(3 * l2 / in_bytes))
        insts = [base] + [make_case(sp, device=dev, seed=rank_seed(sp.seed, rank) + 104729 * (c + 1), poison=False,
                                    lengths=base.lens_host) for c in range(copies - 1)]
        layout = layout_for(base.k_pool, sp.head_dim, sp.bits, sp.group_size, v_pool=base.v_pool)
        params = DecodeParams(sp.num_seqs, sp.num_q_heads, sp.n_query, base.block_tables.shape[1],
                              base.partition_tokens, sp.window, CONTRACTIONS[args.contraction],
                              SCHEDULES[args.schedule])
        plan = make_plan(layout, params)
        ws = torch.empty(max(1, plan.workspace_bytes), dtype=torch.uint8, device=dev)
        out = torch.empty(base.q.shape[:-1] + (sp.dv,), dtype=base.q.dtype, device=dev)
        if args.step == "fused":  # the step's new K/V rows (rows len-N .. len-1 of each sequence)
            gen = torch.Generator(device=dev).manual_seed(rank_seed(sp.seed, rank) + 7)
            for c in insts:
                shape = (sp.num_seqs, sp.num_kv_heads, sp.n_query)
                c.k_new = torch.randn(shape + (sp.head_dim,), generator=gen, device=dev).to(torch.bfloat16)
                c.v_new = torch.randn(shape + (sp.dv,), generator=gen, device=dev).to(torch.bfloat16)
        layers.append(dict(spec=sp, insts=insts, plan=plan, ws=ws, out=out, copies=copies, in_bytes=in_bytes,
                           kv_bytes=required_kv_bytes(sp, base.lens_host)))
    step_bytes = sum(L["kv_bytes"] for L in layers)
    n_copies = max(L["copies"] for L in layers)

    def call(L, i, passes=None):
        c = L["insts"][i % L["copies"]]
        sp = L["spec"]
        kw = dict(bits=sp.bits, group_size=sp.group_size, k_scales=c.k_scales, k_biases=c.k_biases,
                  v_scales=c.v_scales, v_biases=c.v_biases, partition_tokens=c.partition_tokens, window=sp.window,
                  out=L["out"], workspace=L["ws"], contraction=CONTRACTIONS[args.contraction],
                  schedule=SCHEDULES[args.schedule])
        if args.step == "fused":
            paged_decode_append_attention(c.q, c.k_new, c.v_new, c.k_pool, c.v_pool, c.block_tables, c.seq_lens,
                                          c.scale, **kw)
        elif passes is None:
            paged_decode_attention(c.q, c.k_pool, c.v_pool, c.block_tables, c.seq_lens, c.scale, **kw)
        else:
            paged_decode_passes(c.q, c.k_pool, c.v_pool, c.block_tables, c.seq_lens, c.scale, passes=passes, **kw)

    def step(i, passes=None, only=None):
        for L in layers if only is None else [only]:
            call(L, i, passes)

    stream = torch.cuda.Stream(device=dev)

    def capture(n, passes=None, offset=0, only=None):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                step(offset + i, passes, only)
        return g

    def replay_timed(graphs_reps):
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for g, reps in graphs_reps:
                for _ in range(reps):
                    g.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        ms = max_over_ranks(e0.elapsed_time(e1), dev)
        if world > 1:
            dist.barrier()
        return ms

    # warm-up: W eager steps on the launching stream
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    torch.cuda.synchronize(dev)

    # graphs of whole rotations of the input copies, replayed to make exactly K steps
    K = args.steps
    chunk = min(K, max(n_copies, 50 if n_copies == 1 else n_copies))
    g_full = capture(chunk)
    rest = K % chunk
    g_rest = capture(rest, offset=0) if rest else None
    g_full.replay()  # first replay outside the timed region (graph upload)
    if g_rest is not None:
        g_rest.replay()
    torch.cuda.synchronize(dev)

    clocks = ClockSampler(local, dev)
    clocks.start()
    ms = replay_timed([(g_full, K // chunk)] + ([(g_rest, 1)] if g_rest else []))
    clk = clocks.stop()

    # the partial pass alone (the dominant kernel), same inputs, same stream; the fused
    # step has no separate partial pass, so its roofline is the whole step's
    if args.step == "fused":
        ms_partial = ms
    else:
        g_part = capture(chunk, passes="partial")
        g_part_rest = capture(rest, passes="partial") if rest else None
        g_part.replay()
        torch.cuda.synchronize(dev)
        ms_partial = replay_timed([(g_part, K // chunk)] + ([(g_part_rest, 1)] if g_part_rest else []))
        del g_part, g_part_rest

    # each layer's partial pass alone, when a step has several layers
    layer_rows = []
    if len(layers) > 1 and args.step != "fused":
        for L in layers:
            g1 = capture(chunk, passes="partial", only=L)
            g1_rest = capture(rest, passes="partial", only=L) if rest else None
            g1.replay()
            torch.cuda.synchronize(dev)
            ms1 = replay_timed([(g1, K // chunk)] + ([(g1_rest, 1)] if g1_rest else [])) / K
            del g1, g1_rest
            layer_rows.append((L, ms1))

    # end to end through the public host-driven step (pkv_step_run): per step the
    # kernels read the step's inputs (q, block tables, lengths and, for the fused step,
    # the new K/V rows) from pinned host memory and write the output back into pinned
    # host memory, over NVLink-C2C
    host_steps = []  # [layer][input copy], rotated like the device-timed loop
    for L in layers:
        sp = L["spec"]
        host_steps.append([HostDecodeStep(
            c.q, c.block_tables, c.seq_lens, c.k_pool, c.v_pool, c.scale,
            k_new=c.k_new if args.step == "fused" else None, v_new=c.v_new if args.step == "fused" else None,
            bits=sp.bits, group_size=sp.group_size, k_scales=c.k_scales, k_biases=c.k_biases, v_scales=c.v_scales,
            v_biases=c.v_biases, partition_tokens=c.partition_tokens, window=sp.window, workspace=L["ws"],
            stream=stream, contraction=CONTRACTIONS[args.contraction], schedule=SCHEDULES[args.schedule])
            for c in L["insts"]])
    h2d = sum(hs[0].h2d_bytes for hs in host_steps)
    d2h = sum(hs[0].d2h_bytes for hs in host_steps)
    e2e_steps = min(K, max(50, n_copies))

    def e2e_once(i):
        for hs in host_steps:
            hs[i % len(hs)]()

    with torch.cuda.stream(stream):
        for i in range(3):
            e2e_once(i)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(e2e_steps):
            e2e_once(i)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, dev)

    ms_step = ms / K
    value = weak_scaling_rate(step_bytes, world, ms_step)
    part_ms = ms_partial / K
    peak, peak_kind = measured_hbm_peak()
    achieved = step_bytes / (part_ms * 1e-3) / 1e9
    # the merge kernel runs after a partial pass through the workspace: balanced (not for the
    # fused step, which runs partitions), or partitions that do not merge in a cluster
    launches_per_step = sum(1 + ((L["plan"].balanced and args.step == "decode") or
                                 (L["plan"].max_partitions > 1 and not L["plan"].merge_in_cluster)) for L in layers)
    if rank == 0:
        sp0 = layers[0]["spec"]
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": ms_step, "steps_per_s": 1e3 / ms_step * world, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": compute_dtype([L["spec"].bits for L in layers], [L["plan"].contraction for L in layers]),
            "data": "synthetic",
            "config": {
                "workload": args.workload,
                "layers": [L["spec"].description for L in layers],
                "kv_bytes_per_step": step_bytes, "partition_tokens": [L["plan"].partition_tokens for L in layers],
                "partitions_max": [L["plan"].max_partitions for L in layers],
                "l2": (f"inputs rotate over {n_copies} independent copies ({n_copies} x "
                       f"{layers[0]['in_bytes'] / 1e6:.1f} MB >= 3 x L2 {l2 / 1e6:.0f} MB)" if n_copies > 1 else
                       f"inputs ({layers[0]['in_bytes'] / 1e9:.2f} GB) larger than L2 ({l2 / 1e6:.0f} MB)"),
                "timing": "CUDA graph of the K steps replayed; CUDA events on the launching stream",
                "step": ("decode call (pkv_paged_decode_attention)" if args.step == "decode" else
                         "decode step with its write (pkv_paged_decode_append_attention): the N new K/V rows of "
                         "every (sequence, KV head) are written into their pages, then the grown cache is read"),
                "parallelism": f"dp{world} (independent instances)",
                "contraction": ["cuda cores" if L["plan"].contraction == 2 else "tensor cores" for L in layers],
                "schedule": ["balanced" if L["plan"].balanced and args.step == "decode" else "partitions"
                             for L in layers],
            },
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": recorded_traffic(args.workload, args.step),
                         "traffic_unit": "DRAM bytes read + written by the partial-pass launches of one step "
                                         "(ncu, profiles/dram_traffic.json); algorithmic bytes per step: "
                                         f"{step_bytes}",
                         "kernel": (f"pkv_partial_kernel (partial pass alone, {part_ms * 1e3:.2f} us per step)"
                                    if args.step == "decode" else
                                    f"the fused step (write + partial + merge, {part_ms * 1e3:.2f} us per step)"),
                         "peak_source": f"{peak_kind} hbm_gbs", "frac_of_nominal_7900": achieved / 7900.0},
            "e2e": {"value": weak_scaling_rate(step_bytes, world, e2e_ms), "unit": "GB/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "what": "host-driven step (pkv_step_run) per step: q, block tables, lengths"
                            + (" and the new K/V rows" if args.step == "fused" else "")
                            + " read from pinned host memory and the output written back to pinned host memory by "
                              "the kernels (over NVLink-C2C, counted in h2d/d2h bytes); the KV pool is "
                              "device-resident cache state; steps rotate over the same input copies as the "
                              "device-timed loop, launched one by one from the host"},
            "gpu_launches": launches_per_step * K,
            "clocks": clk,
        }
        if layer_rows:  # per layer: its partial pass alone, timed the same way
            line["roofline"]["layers"] = [
                {"workload": L["spec"].name, "kv_bytes": L["kv_bytes"], "us_partial": ms1 * 1e3,
                 "achieved": L["kv_bytes"] / (ms1 * 1e-3) / 1e9,
                 "frac": L["kv_bytes"] / (ms1 * 1e-3) / 1e9 / peak,
                 "traffic": recorded_traffic(L["spec"].name, args.step)} for L, ms1 in layer_rows]
        if cpu is not None:
            line["cpu_baseline"] = {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample")}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_profile_calls(args):
    """A plain sequence of eager decode calls on one instance (for ncu): no graphs,
    no timing, no CPU work."""
    from dataclasses import replace

    import torch

    from quantized_kv_decode_partial_gb300 import load_library, paged_decode_attention
    from quantized_kv_decode_partial_gb300 import build as pkv_build
    from quantized_kv_decode_partial_gb300.workloads import draw_lengths, make_case, required_kv_bytes

    pkv_build.build()
    load_library()
    dev = torch.device("cuda", 0)
    for sp in workload_specs(args.workload):
        if args.num_seqs:
            lens = draw_lengths(sp)[:args.num_seqs]
            sp = replace(sp, num_seqs=len(lens), lengths=tuple(lens), length_range=None)
        if args.seq_len:
            sp = replace(sp, lengths=(args.seq_len,) * sp.num_seqs, length_range=None)
        if args.partition_tokens != -2:
            sp = replace(sp, partition_tokens=args.partition_tokens)
        c = make_case(sp, device=dev, poison=False)
        for _ in range(args.profile_calls):
            paged_decode_attention(c.q, c.k_pool, c.v_pool, c.block_tables, c.seq_lens, c.scale, bits=sp.bits,
                                   group_size=sp.group_size, k_scales=c.k_scales, k_biases=c.k_biases,
                                   v_scales=c.v_scales, v_biases=c.v_biases, partition_tokens=c.partition_tokens,
                                   window=sp.window, contraction=CONTRACTIONS[args.contraction],
                                   schedule=SCHEDULES[args.schedule])
        torch.cuda.synchronize()
        print(json.dumps({"profile_calls": args.profile_calls, "workload": sp.name, "num_seqs": sp.num_seqs,
                          "kv_bytes_per_call": required_kv_bytes(sp, c.lens_host)}), flush=True)


def main(argv=None):
    args = parse_args(argv)
    if args.print_kernel_hash:
        print(kernel_source_hash())
    elif args.record_traffic:
        print(json.dumps(record_traffic(args.workload, args.record_traffic)))
    elif args.profile_calls:
        run_profile_calls(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
