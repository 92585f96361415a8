"""Benchmark of the fused grouped-query attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

One step = one sdp_fwd launch over the whole workload (every query head,
every query row, every key). The default workload is the pages' headline
shape: 32 query heads over 2 KV heads, head dim 256, Sq = Skv = 16384, fp16,
non-causal, scale 1/16. Prints one JSON line (rank 0).

Throughput counts 4 * Sq * Skv * D FLOPs per (batch, query head). Inputs are
synthetic and seeded (N(0,1) rounded to the I/O dtype). Q and O are 268 MB
each, larger than the 126 MB L2, so no explicit flush runs between steps.

--impl reference times the fp64 CPU oracle (the only other implementation
that exists for this path) on the host cores, on a bounded sample of query
rows of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gqa_flash_attention_gb300 import workloads  # noqa: E402

METRIC = "attention fwd TFLOP/s on 1 GB300 and % of dense fp16/bf16 tensor peak"
BENCH_WORKLOADS = {**workloads.ALL_WORKLOADS, **workloads.VARLEN_WORKLOADS}
FALLBACK_PEAK_TFLOPS = 1900.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=workloads.HEADLINE, choices=sorted(BENCH_WORKLOADS))
    ap.add_argument("--cpu-rows", type=int, default=0, help="query rows per head in the CPU sample (0: auto)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--op", choices=["attention", "merge", "host"], default="attention",
                    help="merge: time sdp_merge (HBM-bound) on a context-parallel-shaped case instead; host: "
                         "the host time of one sdp_fwd call (argument checks, tensor maps, launch) on the "
                         "smallest workload")
    ap.add_argument("--merge-parts", type=int, default=8)
    ap.add_argument("--override", nargs="*", default=[], metavar="FIELD=VALUE",
                    help="change fields of a dense workload (B, Hq, Hkv, Sq, Skv): a smaller case of the same "
                         "kernel, e.g. for a multi-pass ncu capture; the workload name gets the changes appended")
    ap.add_argument("--debug-flags", type=int, default=0,
                    help="the library's test hooks (sdp_set_debug_flags), e.g. 128 for the opt-in two-tile "
                         "kernel at head dim 128; 0 (the default) runs what sdp_fwd picks")
    ap.add_argument("--graph", choices=["auto", "on", "off"], default="auto",
                    help="replay each step from a CUDA graph (auto: for the split-KV decode workloads, whose "
                         "steps are shorter than the host's per-call work)")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, device) -> float:
    """The largest x over all ranks (the slowest replica sets the job's time); x itself at N=1."""
    if dist_env()[0] == 1:
        return float(x)
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, flops_per_replica: float, ms_per_step: float) -> float:
    """Whole-job TFLOP/s: every replica does the same work, timed by the slowest."""
    return world * flops_per_replica / (ms_per_step * 1e-3) / 1e12


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return float(pk["bf16_tflops"]), float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"])), "measured"
    return FALLBACK_PEAK_TFLOPS, 1700.0, "fallback"


def load_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def code_tokens(text: str) -> str:
    """C++ source without comments and with whitespace collapsed: what the compiler sees, so a
    comment edit does not count as a kernel change."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def source_hash():
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gqa_flash_attention_gb300", "csrc")
    # the kernel's own sources only (the host-side entry points do not change its traffic)
    for name in sorted(n for n in os.listdir(csrc) if n.startswith(("sdp_fwd", "ptx", "sdp_launch"))):
        with open(os.path.join(csrc, name)) as f:
            h.update(name.encode() + code_tokens(f.read()).encode())
    return h.hexdigest()[:16]


def merge_source_hash():
    import hashlib
    with open(os.path.join(ROOT, "gqa_flash_attention_gb300", "csrc", "sdp_merge.cu")) as f:
        return hashlib.sha256(code_tokens(f.read()).encode()).hexdigest()[:16]


def load_traffic(workload: str, prefix: str = "sdp_fwd_", current_hash=None):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", f"{prefix}{workload}_traffic.txt")
    if not os.path.exists(path):
        return None
    kv = {}
    with open(path) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
    if kv.get("source_hash") != (current_hash or source_hash()):
        return None
    try:
        return int(float(kv["traffic_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


class NvmlSampler:
    """Read-only NVML queries (SM clock, power, clock-event reasons) every ~10 ms in a
    background thread while the timed region runs, through ctypes on the driver's
    libnvidia-ml (no Python package needed). Nothing is set or reset."""

    # clock-event reason bits of nvmlDeviceGetCurrentClocksEventReasons
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, device_index: int, period_s: float = 0.01):
        import ctypes
        self.period = period_s
        self.rows = []
        self.thread = None
        self.stop_flag = False
        self.ok = False
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            h = ctypes.c_void_p()
            if nv.nvmlDeviceGetHandleByUUID(("GPU-" + uuid).encode(), ctypes.byref(h)) != 0:
                return
            self.nv, self.h, self.ct = nv, h, ctypes
            mx = ctypes.c_uint()
            self.sm_max = float(mx.value) if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0 else None
            self.reasons_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons", None)
            self.ok = self.sample() is not None
        except Exception:
            self.ok = False

    def sample(self):
        ct, nv, h = self.ct, self.nv, self.h
        clk, mw, rs = ct.c_uint(), ct.c_uint(), ct.c_ulonglong()
        if nv.nvmlDeviceGetClockInfo(h, 1, ct.byref(clk)) != 0:  # NVML_CLOCK_SM
            return None
        power = mw.value / 1000.0 if nv.nvmlDeviceGetPowerUsage(h, ct.byref(mw)) == 0 else None
        reasons = rs.value if self.reasons_fn is not None and self.reasons_fn(h, ct.byref(rs)) == 0 else 0
        return float(clk.value), power, reasons

    def _loop(self):
        while not self.stop_flag:
            r = self.sample()
            if r is not None:
                self.rows.append(r)
            time.sleep(self.period)

    def start(self):
        import threading
        self.rows = []
        self.stop_flag = False
        self.thread = threading.Thread(target=self._loop, daemon=True)
        self.thread.start()

    def stop(self):
        self.stop_flag = True
        self.thread.join(timeout=5)
        r = self.sample()  # at least one reading from the end of the region
        if r is not None:
            self.rows.append(r)
        sm = [x[0] for x in self.rows]
        pw = [x[1] for x in self.rows if x[1] is not None]
        reasons = sorted({name for x in self.rows for bit, name in self.REASONS.items() if x[2] & bit})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_mhz_min": min(sm) if sm else None,
                "sm_max_mhz": self.sm_max, "power_w_max": max(pw) if pw else None,
                "power_w_median": statistics.median(pw) if pw else None, "samples": len(sm),
                "period_ms": 1000 * self.period, "source": "NVML (read-only), in-process", "reasons": reasons}


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs (the
    fallback where NVML cannot be loaded in-process)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.uuid = None
        try:
            self.uuid = "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)
        except Exception:
            pass

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        if self.uuid:
            cmd += ["-i", self.uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        rows = [r.split(",") for r in self.out.read().strip().splitlines() if r.strip()]
        os.unlink(self.out.name)
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                pw.append(float(r[3]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "samples": len(sm), "reasons": sorted(reasons)}


def clock_sampler(device_index: int):
    """NVML sampling every 10 ms where it loads, else nvidia-smi every 50 ms."""
    nv = NvmlSampler(device_index)
    return nv if nv.ok else ClockSampler(device_index)


# The second roofline denominator: NVIDIA's nominal dense fp16/bf16 tensor rate of one
# GB300 (HGX B300 specifications: 36 PFLOPS FP16/BF16 per 8 GPUs, quoted with 2:4
# sparsity; dense is half of that, per GPU 2.25 PFLOPS).
DATASHEET_TFLOPS = 2250.0
DATASHEET_SOURCE = ("NVIDIA HGX B300 specifications: 36 PFLOPS FP16/BF16 per 8 GPUs with 2:4 sparsity "
                    "= 2.25 PFLOPS dense per GPU")


def is_varlen(w):
    return isinstance(w, workloads.VarlenWorkload)


def cpu_rows_auto(w):
    # about 10-20 s of oracle work on a 16-core host (the oracle runs near 60 fp64 GFLOP/s there)
    target = 8e11
    if is_varlen(w):
        per_row = 4.0 * w.D * w.Hq * sum(w.lens_k)  # one row per sequence and head
        return int(max(2, min(w.max_q, target / per_row)))
    per_row = 4.0 * w.Skv * w.D
    return int(max(2, min(w.Sq, target / (per_row * w.B * w.Hq))))


def host_inputs(w):
    return workloads.make_varlen_inputs(w) if is_varlen(w) else workloads.make_inputs(w)


def run_cpu_oracle(w, rows_per_head, q=None, k=None, v=None):
    """Time the oracle on a sample of query rows; returns (tflops, seconds, sample description, threads)."""
    import oracle
    if q is None:
        q, k, v = host_inputs(w)
    dt = oracle.FP16 if w.dtype == "fp16" else oracle.BF16
    if is_varlen(w):
        # rows_per_head rows of every (sequence, head), each sequence on its own through the dense oracle
        rng = np.random.default_rng(1234)
        sec, seen = 0.0, 0
        for b in range(w.nseq):
            lq, lk = w.lens_q[b], w.lens_k[b]
            if lq == 0 or lk == 0:
                continue
            m = min(rows_per_head, lq)
            rows = np.sort(np.stack([rng.choice(lq, size=m, replace=False) for _ in range(w.Hq)]))
            rows = rows.reshape(1, w.Hq, m).astype(np.int32)
            qs = q[w.cu_q[b]:w.cu_q[b + 1]].permute(1, 0, 2).unsqueeze(0).contiguous()
            ks = k[w.cu_k[b]:w.cu_k[b + 1]].permute(1, 0, 2).unsqueeze(0).contiguous()
            vs = v[w.cu_k[b]:w.cu_k[b + 1]].permute(1, 0, 2).unsqueeze(0).contiguous()
            t0 = time.perf_counter()
            oracle.sdp_fwd_rows(qs, ks, vs, dt, (1, w.Hq, w.Hkv, lq, lk, w.D), w.softmax_scale, rows,
                                causal=w.causal)
            sec += time.perf_counter() - t0
            seen += int((np.minimum(rows.astype(np.int64) + 1, lk) if w.causal else np.full(rows.shape, lk)).sum())
        desc = (f"{rows_per_head} query rows per (sequence, head) x {w.nseq} sequences x {w.Hq} heads of "
                f"{w.name}, all of each sequence's keys")
        return 4.0 * seen * w.D / sec / 1e12, sec, desc, oracle.num_threads()
    rows = workloads.sample_rows(w, rows_per_head, seed=1234)
    t0 = time.perf_counter()
    oracle.sdp_fwd_rows(q, k, v, dt, w.shape, w.softmax_scale, rows, causal=w.causal)
    sec = time.perf_counter() - t0
    seen = (np.minimum(rows.astype(np.int64) + 1, w.Skv) if w.causal else np.full(rows.shape, w.Skv)).sum()
    flops = 4.0 * float(seen) * w.D
    desc = f"{rows.shape[2]} query rows per (batch, head) x {w.B * w.Hq} heads of {w.name}, all {w.Skv} keys"
    return flops / sec / 1e12, sec, desc, oracle.num_threads()


# ------------------------------------------------------------------ arms

def reference_arm(args, w):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    rows = args.cpu_rows or max(2, cpu_rows_auto(w) // 4)
    q, k, v = host_inputs(w)
    for _ in range(args.warmup):
        run_cpu_oracle(w, max(2, rows // 8), q, k, v)
    vals, secs = [], []
    for _ in range(args.steps):
        tf, sec, desc, threads = run_cpu_oracle(w, rows, q, k, v)
        vals.append(tf)
        secs.append(sec)
    value = statistics.median(vals)
    sample = desc + ", per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * statistics.median(secs),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {**config_of(w, args.gpus), "cuda_graph": use_graph_for(args, w)},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample,
                         "extrapolated_full_workload_s": w.flops() / (value * 1e12)},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def use_graph_for(args, w):
    """Whether our arm replays each step from a CUDA graph (auto: the split-KV decode
    workloads, whose steps are shorter than the host's per-call work)."""
    return args.graph == "on" or (args.graph == "auto" and not is_varlen(w) and w.kv_splits != 1)


def launch_shape(w):
    """(Sq, G) of the launch: without a causal mask the G query heads of a KV
    group run as one head of G * Sq rows when Sq is not a multiple of 128."""
    G = w.Hq // w.Hkv
    if not w.causal and G > 1 and w.Sq % 128:
        return w.Sq * G, 1
    return w.Sq, G


def kernel_name(w, debug_flags=0, captured=False):
    """The kernel sdp_fwd launches for this workload: the CTA-pair kernel when
    the units of each (batch, KV head) pair up (and, causal, share the query
    tile), else the single-CTA kernel, each in its persistent form for dense
    launches with more units than SMs (debug bit 4 keeps one CTA or pair per
    unit; a launch captured into a graph keeps one CTA per unit on single CTAs);
    split-KV adds the merge kernel; variable-length batches pair up when the
    group size is even; head dim 128 runs on single CTAs."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 152
    if w.D == 128:
        # dense, non-causal launches whose two-tile units pair up and fill a wave of CTAs run the
        # two-tile CTA-pair kernel; the rest the single-CTA kernel
        name = "sdp_fwd_kernel"
        if (PAIR2_BY_DEFAULT or debug_flags & 128) and not is_varlen(w) and not w.causal:
            sq, G = launch_shape(w)
            n_qpairs = ((sq + 127) // 128 + 1) // 2
            splits = max(1, w.kv_splits)
            if (n_qpairs * G) % 2 == 0 and (w.B * w.Hkv * G * n_qpairs * splits >= sms or debug_flags & 128):
                name = "sdp_fwd_pair2_kernel"
        if getattr(w, "kv_splits", 1) != 1:
            return name + " + merge_kernel"
        if name == "sdp_fwd_kernel" and not is_varlen(w) and not w.causal and not debug_flags & 16 and not captured:
            sq, G = launch_shape(w)
            if w.B * w.Hkv * G * ((sq + 127) // 128) > sms:
                return "sdp_fwd_persist_kernel"
        return name
    if is_varlen(w):
        if (w.Hq // w.Hkv) % 2:
            return "sdp_fwd_kernel"
        # causal batches with more (compact-list) units than SMs run the persistent CTA pair
        n_units = w.Hq * sum((lq + 127) // 128 for lq in w.lens_q)
        if w.causal and n_units > sms and not debug_flags & 16:
            return "sdp_fwd_pair_persistent_kernel"
        return "sdp_fwd_pair_kernel"
    sq, G = launch_shape(w)
    n_qtiles = (sq + 127) // 128
    pair = (n_qtiles * G) % 2 == 0 and not (w.causal and G % 2)
    name = "sdp_fwd_pair_kernel" if pair else "sdp_fwd_kernel"
    if w.kv_splits != 1:
        return name + " + merge_kernel"
    # dense launches with more units than SMs run the persistent forms
    units = w.B * w.Hkv * G * n_qtiles
    if units > sms and not debug_flags & 16 and (pair or not w.causal):
        if pair:
            return "sdp_fwd_pair_persistent_kernel"
        if not captured:
            return "sdp_fwd_persist_kernel"
    return name


# whether the library runs dense D=128 launches on the two-tile CTA-pair kernel by default
PAIR2_BY_DEFAULT = False

L2_BYTES = 126 * 2 ** 20


def needs_flush(w):
    return w.hbm_bytes() < 2 * L2_BYTES


def config_of(w, n):
    if is_varlen(w):
        return {"workload": w.name, "nseq": w.nseq, "lens_q": list(w.lens_q), "lens_k": list(w.lens_k),
                "total_q": w.total_q, "total_k": w.total_k, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
                "io_dtype": w.dtype, "scale": w.softmax_scale, "causal": w.causal, "layout": "tokens, heads, D",
                "flops_per_step_per_gpu": w.flops(),
                "l2": ("L2 flushed (256 MB write) before every timed step; only the call is timed" if needs_flush(w)
                       else "inputs larger than L2; no flush"),
                "parallelism": "replicas" if n > 1 else "single GPU"}
    return {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq, "Skv": w.Skv, "D": w.D,
            "io_dtype": w.dtype, "scale": w.softmax_scale, "causal": w.causal, "peaky_k": w.peaky_k,
            "flops_per_step_per_gpu": w.flops(), "kv_splits": w.kv_splits,
            "l2": ("L2 flushed (256 MB write) before every timed step; only the call is timed" if needs_flush(w)
                   else "inputs larger than L2; no flush"),
            "parallelism": "replicas" if n > 1 else "single GPU"}


def ours_arm(args, w):
    import gqa_flash_attention_gb300 as sdp
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    sdp.lib()
    sdp.set_debug_flags(args.debug_flags)

    q_h, k_h, v_h = host_inputs(w)
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    o = torch.empty_like(q)
    if is_varlen(w):
        lse = torch.empty(w.Hq, w.total_q, dtype=torch.float32, device=dev)
        cu_h = [torch.from_numpy(w.cu_q), torch.from_numpy(w.cu_k)]
        cu_q, cu_k = (t.to(dev) for t in cu_h)
    else:
        lse = torch.empty(w.B, w.Hq, w.Sq, dtype=torch.float32, device=dev)
        cu_h = []
    stream = torch.cuda.current_stream(dev)

    launches_per_step = 1
    ws = None
    if is_varlen(w):
        pass
    elif w.kv_splits != 1:
        dt = sdp.SDP_BF16 if w.dtype == "bf16" else sdp.SDP_FP16
        splits = sdp.splitkv_count(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, dt, w.kv_splits)
        need = sdp.splitkv_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, dt, w.kv_splits)
        ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        launches_per_step = 2 if splits > 1 else 1

    def call():
        if is_varlen(w):
            sdp.sdp_fwd_varlen(q, k, v, cu_q, cu_k, w.max_q, scale=w.softmax_scale, causal=w.causal, out=o,
                               lse=lse)
        else:
            sdp.sdp_fwd(q, k, v, scale=w.softmax_scale, out=o, lse=lse, causal=w.causal, kv_splits=w.kv_splits,
                        workspace=ws)

    flush = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=dev) if needs_flush(w) else None
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize(dev)
    if sdp.poll_status() != sdp.SDP_OK:
        raise RuntimeError("kernel reported a timeout during warm-up")
    use_graph = use_graph_for(args, w)
    step = call
    if use_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            call()
        graph.replay()
        torch.cuda.synchronize(dev)
        step = graph.replay

    K = args.steps
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    clocks = clock_sampler(dev.index)
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    for i in range(K):
        if flush is not None:
            flush.zero_()
        ev0[i].record(stream)
        step()
        ev1[i].record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()
    per_launch_ms = [ev0[i].elapsed_time(ev1[i]) for i in range(K)]
    # back to back, the whole region is the time; with flushes between steps, the sum of the steps
    total_ms = sum(per_launch_ms) if flush is not None else ev0[0].elapsed_time(ev1[K - 1])
    if sdp.poll_status() != sdp.SDP_OK:
        raise RuntimeError("kernel reported a timeout in the timed region")

    ms_per_step = max_over_ranks(total_ms, dev) / K
    value = job_throughput(world, w.flops(), ms_per_step)

    # End to end through the public API: every step copies its inputs from pinned host memory and
    # reads O and LSE back to pinned host memory. Steps are pipelined as a serving loop would run
    # them: a copy-in stream, the compute stream and a copy-out stream, with two device buffer sets,
    # so step i+1's inputs and step i-1's outputs move while step i computes.
    e2e = None
    if not args.no_e2e:
        qp, kp, vp = q_h.pin_memory(), k_h.pin_memory(), v_h.pin_memory()
        cu_p = [t.pin_memory() for t in cu_h]
        op = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
        lp = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
        # enough steps that the pipeline's fill (the first step's copy-in) and drain (the last
        # step's copy-out) weigh little against the steady state a serving loop runs in
        n_e2e = max(10, K // 2)
        sets = [dict(q=q, k=k, v=v, o=o, lse=lse, cu=[cu_q, cu_k] if cu_h else [])]
        sets.append({key: (torch.empty_like(val) if isinstance(val, torch.Tensor) else [torch.empty_like(t_) for t_ in val])
                     for key, val in sets[0].items()})
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def compute(b, st):
            if is_varlen(w):
                sdp.sdp_fwd_varlen(b["q"], b["k"], b["v"], b["cu"][0], b["cu"][1], w.max_q, scale=w.softmax_scale,
                                   causal=w.causal, out=b["o"], lse=b["lse"], stream=st)
            else:
                sdp.sdp_fwd(b["q"], b["k"], b["v"], scale=w.softmax_scale, out=b["o"], lse=b["lse"], causal=w.causal,
                            kv_splits=w.kv_splits, workspace=ws, stream=st)

        def pipeline(n):
            done_c = [torch.cuda.Event() for _ in range(n)]
            done_o = [torch.cuda.Event() for _ in range(n)]
            for i in range(n):
                b = sets[i % 2]
                with torch.cuda.stream(s_in):
                    if i >= 2:
                        s_in.wait_event(done_c[i - 2])  # this set's inputs were consumed by step i-2
                    b["q"].copy_(qp, non_blocking=True)
                    b["k"].copy_(kp, non_blocking=True)
                    b["v"].copy_(vp, non_blocking=True)
                    for d_, h_ in zip(b["cu"], cu_p):
                        d_.copy_(h_, non_blocking=True)
                stream.wait_stream(s_in)
                if i >= 2:
                    stream.wait_event(done_o[i - 2])  # this set's outputs were read back
                compute(b, stream)
                done_c[i].record(stream)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(done_c[i])
                    op.copy_(b["o"], non_blocking=True)
                    lp.copy_(b["lse"], non_blocking=True)
                    done_o[i].record(s_out)
            stream.wait_stream(s_out)

        pipeline(2)
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        e0.record(stream)
        s_in.wait_stream(stream)
        pipeline(n_e2e)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        if sdp.poll_status() != sdp.SDP_OK:
            raise RuntimeError("kernel reported a timeout in the end-to-end leg")
        te = max_over_ranks(e0.elapsed_time(e1) / n_e2e, dev)
        h2d = sum(t_.numel() * t_.element_size() for t_ in (q_h, k_h, v_h, *cu_h))
        d2h = o.numel() * o.element_size() + lse.numel() * lse.element_size()
        e2e = {"value": job_throughput(world, w.flops(), te), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "pipelined": "copy-in, compute and copy-out streams, two device buffer sets"}

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    peak, peak_sus, peak_src = load_peaks()
    hbm_peak, hbm_src = load_hbm_peak()
    avg_launch_ms = statistics.mean(per_launch_ms)
    tflops = w.flops() / (avg_launch_ms * 1e-3) / 1e12
    intensity = w.flops() / w.hbm_bytes()  # FLOP per algorithmic HBM byte
    if intensity >= peak * 1e12 / (hbm_peak * 1e9):
        roofline = {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                    "frac": tflops / peak, "traffic": load_traffic(w.name),
                    "peak_source": f"{peak_src} bf16 dense (burst); fp16 runs at the same tensor rate",
                    "frac_of_sustained": tflops / peak_sus}
    else:
        gbs = w.hbm_bytes() / (avg_launch_ms * 1e-3) / 1e9
        roofline = {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
                    "traffic": load_traffic(w.name), "peak_source": f"{hbm_src} HBM copy bandwidth",
                    "algorithmic_bytes": w.hbm_bytes(), "tflops": tflops}
    roofline.update({"kernel": kernel_name(w, args.debug_flags, use_graph), "launch_ms_median": statistics.median(per_launch_ms),
                     "flop_per_byte": intensity})
    if roofline["bound"] == "tensor":
        roofline.update({"peak_datasheet": DATASHEET_TFLOPS, "frac_datasheet": tflops / DATASHEET_TFLOPS,
                         "peak_datasheet_source": DATASHEET_SOURCE})
    # FLOP per SM per clock at the sampled median SM clock: comparable across power states
    # (the tensor cores' nominal dense fp16/bf16 rate is 8192 per SM per clock)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    if clk.get("sm_mhz"):
        roofline["flop_per_sm_cycle"] = w.flops() / (avg_launch_ms * 1e-3 * clk["sm_mhz"] * 1e6 * sms)
    achieved = tflops

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        rows = args.cpu_rows or cpu_rows_auto(w)
        tf, sec, desc, threads = run_cpu_oracle(w, rows, q_h, k_h, v_h)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "extrapolated_full_workload_s": w.flops() / (tf * 1e12),
               "sample": f"{desc} ({sec:.1f} s)"}

    cfg = config_of(w, world)
    cfg["cuda_graph"] = use_graph
    if args.debug_flags:
        cfg["debug_flags"] = args.debug_flags
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "latency_us_per_step": 1000 * ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic", "config": cfg,
        "pct_of_peak": 100.0 * achieved / peak,
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clk,
        "gpu_launches": K * launches_per_step,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def merge_arm(args, w):
    """sdp_merge of P partial results per row (one per key shard, as in ring
    attention) for every (batch, head, query row) of the workload."""
    import gqa_flash_attention_gb300 as sdp
    dev = torch.device("cuda", 0)
    P, rows = args.merge_parts, w.B * w.Hq * w.Sq
    g = torch.Generator(device=dev).manual_seed(w.seed)
    o_parts = torch.randn(P, rows, w.D, device=dev, generator=g).to(w.torch_dtype)
    lse_parts = torch.randn(P, rows, device=dev, generator=g) * 3
    o = torch.empty(rows, w.D, dtype=w.torch_dtype, device=dev)
    lse = torch.empty(rows, dtype=torch.float32, device=dev)
    for _ in range(args.warmup):
        sdp.sdp_merge(o_parts, lse_parts, out=o, lse=lse)
    K = args.steps
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    clocks = clock_sampler(0)
    clocks.start()
    torch.cuda.synchronize(dev)
    ev[0].record()
    for i in range(K):
        sdp.sdp_merge(o_parts, lse_parts, out=o, lse=lse)
        ev[i + 1].record()
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    ms = statistics.mean(ev[i].elapsed_time(ev[i + 1]) for i in range(K))
    nbytes = P * rows * (w.D * 2 + 4) + rows * (w.D * 2 + 4)
    gbs = nbytes / (ms * 1e-3) / 1e9
    peak, _ = load_hbm_peak()
    print(json.dumps({
        "metric": "sdp_merge HBM GB/s", "value": gbs, "unit": "GB/s", "n_gpus": 1, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": f"merge of {P} parts over {w.name} rows", "parts": P, "rows": rows, "D": w.D,
                   "l2": "inputs larger than L2; no flush"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                     "traffic": load_traffic(f"{w.name}_p{P}", "sdp_merge_", merge_source_hash()),
                     "kernel": "merge_kernel", "bytes_per_launch": nbytes},
        "clocks": clk, "gpu_launches": K}), flush=True)


def host_arm(args):
    """Host-side cost of one call: back-to-back sdp_fwd calls on gqa4_s256_d128_fp16
    (whose kernel is shorter than the call, so the launch queue never fills), timed with
    the host clock; the ctypes cost of a trivial exported call is reported beside it."""
    import ctypes
    import gqa_flash_attention_gb300 as sdp
    w = workloads.ALL_WORKLOADS["gqa4_s256_d128_fp16"]
    dev = torch.device("cuda", 0)
    q, k, v = (t.to(dev) for t in workloads.make_inputs(w))
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.Hq, w.Sq, dtype=torch.float32, device=dev)
    st = torch.cuda.current_stream(dev).cuda_stream
    args_ptr = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), w.B, w.Hq, w.Hkv, w.Sq,
                w.Skv, w.D, w.softmax_scale, sdp.SDP_FP16, st)
    L = sdp.lib()
    raw = L.sdp_fwd
    c_args = [ctypes.c_void_p(a) for a in args_ptr[:5]] + list(args_ptr[5:11]) + \
        [ctypes.c_float(args_ptr[11]), args_ptr[12], ctypes.c_void_p(st)]
    n = max(args.steps, 200)

    def per_call_us(fn):
        for _ in range(args.warmup + 10):
            fn()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(n):
            fn()
        t1 = time.perf_counter()
        torch.cuda.synchronize(dev)
        return 1e6 * (t1 - t0) / n

    res = {
        "ctypes_trivial_call_us": per_call_us(lambda: L.sdp_version()),
        "c_abi_call_us": per_call_us(lambda: raw(*c_args)),
        "python_binding_call_us": per_call_us(lambda: sdp.sdp_fwd(q, k, v, scale=w.softmax_scale, out=o, lse=lse)),
    }
    if sdp.poll_status() != sdp.SDP_OK:
        raise RuntimeError("kernel reported a timeout")
    print(json.dumps({"metric": "host microseconds per sdp_fwd call", "value": res["c_abi_call_us"],
                      "unit": "us", "higher_is_better": False, "steps": n, "warmup": args.warmup,
                      "config": {"workload": w.name, "calls": n}, **res}), flush=True)


def main():
    args = parse()
    w = BENCH_WORKLOADS[args.workload]
    if args.override:
        if is_varlen(w):
            raise SystemExit("--override applies to dense workloads only")
        kw = {}
        for item in args.override:
            key, _, val = item.partition("=")
            if key not in ("B", "Hq", "Hkv", "Sq", "Skv"):
                raise SystemExit(f"cannot override {key!r}")
            kw[key] = int(val)
        w = w.with_(name=w.name + "_" + "_".join(f"{k}{v}" for k, v in kw.items()), **kw)
    if args.op == "host":
        host_arm(args)
    elif args.op == "merge":
        merge_arm(args, w)
    elif args.impl == "reference":
        reference_arm(args, w)
    else:
        ours_arm(args, w)


if __name__ == "__main__":
    main()
