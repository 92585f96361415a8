"""A seeded sweep of shapes nobody picked by hand: batch, query and KV head
counts (odd group sizes included, so pairing and head packing take their
fallbacks), ragged query and key lengths, both head dims and dtypes, the causal
mask and split-KV counts; and variable-length batches of random sequence
counts and lengths (empty queries and key-less sequences included). Every row
of every case is checked against the fp64 oracle, and every output buffer has a
canary-filled guard tail."""
import numpy as np
import pytest
import torch

import gqa_flash_attention_gb300 as sdp
import oracle
from gqa_flash_attention_gb300 import workloads
from gqa_flash_attention_gb300.workloads import VarlenWorkload, Workload
from parity import ORACLE_DTYPE, assert_within, compare
from test_varlen import check_every_row

pytestmark = pytest.mark.gpu


def _cases(n=24, seed=2026):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        D = int(rng.choice([128, 256]))
        dt = str(rng.choice(["fp16", "bf16"]))
        Hkv = int(rng.integers(1, 4))
        G = int(rng.choice([1, 2, 3, 4, 5, 8]))
        B = int(rng.integers(1, 3))
        Sq = int(rng.integers(1, 600))
        Skv = int(rng.integers(1, 700))
        causal = bool(rng.random() < 0.35)
        splits = 1 if causal else int(rng.choice([1, 1, 0, 2, 3]))
        name = f"r{i}_b{B}_h{Hkv * G}x{Hkv}_q{Sq}_k{Skv}_d{D}_{dt}{'_causal' if causal else ''}_s{splits}"
        cases.append((Workload(name, B, Hkv * G, Hkv, Sq, Skv, D, dt, seed=1000 + i, causal=causal), splits))
    return cases


CASES = _cases()


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gqa_flash_attention_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    sdp.lib()


@pytest.mark.parametrize("w,splits", CASES, ids=[w.name for w, _ in CASES])
def test_random_shape_every_row(w, splits, guard=4096):
    q, k, v = workloads.make_inputs(w)
    dev = torch.device("cuda")
    B, Hq, Sq = w.B, w.Hq, w.Sq
    o_buf = torch.full((q.numel() + guard,), float("nan"), dtype=q.dtype, device=dev)
    l_buf = torch.full((B * Hq * Sq + guard,), float("nan"), dtype=torch.float32, device=dev)
    o = o_buf[:q.numel()].view(q.shape)
    lse = l_buf[:B * Hq * Sq].view(B, Hq, Sq)
    sdp.sdp_fwd(q.to(dev), k.to(dev), v.to(dev), scale=w.softmax_scale, out=o, lse=lse, causal=w.causal,
                kv_splits=splits)
    assert sdp.poll_status() == sdp.SDP_OK
    assert torch.isnan(o_buf[q.numel():]).all(), "write past the end of O"
    assert torch.isnan(l_buf[B * Hq * Sq:]).all(), "write past the end of LSE"
    ref_o, ref_l = oracle.sdp_fwd(q, k, v, ORACLE_DTYPE[w.dtype], w.shape, w.softmax_scale, causal=w.causal)
    assert_within(compare(o, lse, ref_o, ref_l, w.dtype), w.dtype)


def _varlen_cases(n=16, seed=2027):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        nseq = int(rng.integers(1, 8))
        lq = tuple(0 if rng.random() < 0.1 else int(rng.integers(1, 400)) for _ in range(nseq))
        lk = tuple(0 if rng.random() < 0.1 else int(rng.integers(1, 500)) for _ in range(nseq))
        if sum(lq) == 0:
            lq = (1,) + lq[1:]
        D = int(rng.choice([128, 256]))
        dt = str(rng.choice(["fp16", "bf16"]))
        Hkv = int(rng.integers(1, 4))
        G = int(rng.choice([1, 2, 3, 4]))
        causal = bool(rng.random() < 0.4)
        name = f"v{i}_n{nseq}_h{Hkv * G}x{Hkv}_d{D}_{dt}{'_causal' if causal else ''}"
        cases.append(VarlenWorkload(name, lq, lk, Hkv * G, Hkv, D, dt, seed=2000 + i, causal=causal))
    return cases


VARLEN_CASES = _varlen_cases()


@pytest.mark.parametrize("w", VARLEN_CASES, ids=[w.name for w in VARLEN_CASES])
def test_random_varlen_batch_every_row(w):
    check_every_row(w)
