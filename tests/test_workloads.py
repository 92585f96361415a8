"""The seeded input generator: reproducible, correctly shaped, and the
peaky-K recipe scales exactly ceil(1% of Skv) K rows per (batch, KV head) by 8."""
import math
import os

import numpy as np
import torch

import oracle
from gqa_flash_attention_gb300 import workloads
from gqa_flash_attention_gb300.workloads import Workload

HERE = os.path.dirname(os.path.abspath(__file__))


def test_shapes_dtypes_and_reproducibility():
    w = Workload("t", 2, 4, 2, 33, 17, 16, "bf16", seed=5)
    q, k, v = workloads.make_inputs(w)
    assert q.shape == (2, 4, 33, 16) and k.shape == v.shape == (2, 2, 17, 16)
    assert q.dtype == k.dtype == v.dtype == torch.bfloat16
    q2, k2, v2 = workloads.make_inputs(w)
    assert torch.equal(q, q2) and torch.equal(k, k2) and torch.equal(v, v2)


def test_peaky_keys():
    base = Workload("t", 2, 4, 2, 8, 300, 16, "bf16", seed=9)
    peaky = base.with_(peaky_k=True)
    _, k0, v0 = workloads.make_inputs(base)
    _, k1, v1 = workloads.make_inputs(peaky)
    assert torch.equal(v0, v1)
    n_peak = math.ceil(0.01 * 300)
    for b in range(2):
        for g in range(2):
            diff = (k0[b, g] != k1[b, g]).any(dim=1)
            assert int(diff.sum()) == n_peak
            assert torch.equal(k1[b, g][diff].float(), 8 * k0[b, g][diff].float())


def test_sample_rows_cover_ends_and_are_distinct():
    w = workloads.WORKLOADS["gqa16_s4k_d256_fp16"]
    rows = workloads.sample_rows(w, 256)
    assert rows.shape == (1, 32, 256)
    for h in range(32):
        r = rows[0, h]
        assert r[0] == 0 and r[-1] == w.Sq - 1 and len(np.unique(r)) == 256


def test_golden_fixture_is_reproduced():
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(HERE, "golden", "make_golden.py"))
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    o, lse = mg.compute()
    with open(os.path.join(HERE, "golden", "oracle_gqa_small.txt")) as f:
        for line in f:
            if line.startswith("#"):
                continue
            parts = line.split()
            b, h, i = (int(x) for x in parts[1:4])
            vals = np.array([float(x) for x in parts[4:]])
            ref = lse[b, h, i:i + 1] if parts[0] == "lse" else o[b, h, i]
            assert np.abs(vals - ref).max() <= 1e-13


def test_flop_and_byte_counts():
    w = workloads.WORKLOADS["gqa16_s16k_d256_fp16"]
    assert w.flops() == 4 * 32 * 16384 * 16384 * 256
    assert w.hbm_bytes() == 2 * (2 * 32 * 16384 * 256) + 2 * (2 * 2 * 16384 * 256) + 32 * 16384 * 4


def test_causal_flop_count():
    """Row i sees min(i + 1, Skv) keys; 4 * D FLOPs per (row, key)."""
    w = Workload("c", 1, 1, 1, 5, 3, 128, causal=True)
    assert w.flops() == 4 * 128 * (1 + 2 + 3 + 3 + 3)
    w2 = Workload("c2", 2, 4, 2, 300, 300, 64, causal=True)
    assert w2.flops() == 4 * 64 * 2 * 4 * (300 * 301 // 2)


def test_varlen_workloads_offsets_and_flops():
    for w in workloads.VARLEN_WORKLOADS.values():
        assert w.cu_q[0] == 0 and w.cu_q[-1] == w.total_q and np.all(np.diff(w.cu_q) == np.array(w.lens_q))
        assert w.cu_k[-1] == w.total_k and len(w.lens_k) == w.nseq
        seen = 0
        for lq, lk in zip(w.lens_q, w.lens_k):
            if w.causal:
                seen += sum(min(i + 1, lk) for i in range(lq))
            else:
                seen += lq * lk
        assert w.flops() == 4 * w.Hq * w.D * seen


def test_varlen_inputs_are_seeded_and_shaped():
    w = workloads.VarlenWorkload("t", (3, 130), (5, 1), 4, 2, 128, "bf16", seed=9)
    q, k, v = workloads.make_varlen_inputs(w)
    assert q.shape == (133, 4, 128) and k.shape == (6, 2, 128) and v.shape == k.shape
    assert q.dtype == torch.bfloat16
    q2, _, _ = workloads.make_varlen_inputs(w)
    assert torch.equal(q, q2)
