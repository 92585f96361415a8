"""The committed DRAM-traffic summaries that bench.py reads: every one parses,
names a positive byte count and a source hash in the form bench.py compares,
and records the full command it came from, for every workload bench.py can
time. (Whether a summary matches the current kernel sources is decided by
bench.py at run time: a stale one reports `traffic: null`.)"""
import os
import re
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from gqa_flash_attention_gb300 import workloads  # noqa: E402

PROFILES = os.path.join(ROOT, "profiles")
TRAFFIC = sorted(f for f in os.listdir(PROFILES) if f.endswith("_traffic.txt"))


def _fields(path):
    kv = {}
    with open(path) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
    return kv


@pytest.mark.parametrize("name", TRAFFIC)
def test_traffic_summary_is_well_formed(name):
    path = os.path.join(PROFILES, name)
    kv = _fields(path)
    assert int(kv["traffic_bytes_per_launch"]) > 0
    assert re.fullmatch(r"[0-9a-f]{16}", kv["source_hash"]), kv["source_hash"]
    text = open(path).read()
    assert "ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum" in text
    assert "--clock-control none" in text


def test_every_bench_workload_has_a_traffic_summary():
    names = set(workloads.ALL_WORKLOADS) | set(workloads.VARLEN_WORKLOADS)
    names.discard("gqa4_s256_d128_fp16")  # eight CTAs, latency-bound: timed in us, no DRAM roofline
    missing = sorted(n for n in names if f"sdp_fwd_{n}_traffic.txt" not in TRAFFIC)
    assert not missing, missing


def test_bench_reads_a_summary_only_for_its_own_sources():
    name = "gqa16_s16k_d256_fp16"
    kv = _fields(os.path.join(PROFILES, f"sdp_fwd_{name}_traffic.txt"))
    assert bench.load_traffic(name, current_hash=kv["source_hash"]) == int(kv["traffic_bytes_per_launch"])
    assert bench.load_traffic(name, current_hash="0" * 16) is None
