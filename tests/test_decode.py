"""Small-Sq / decode grouped-query attention against the fp64 oracle.

Two launch-shape changes serve problems with few query rows:
- head packing: without a causal mask, the G query heads of a KV group are
  run as one head of G * Sq rows when Sq is not a multiple of 128 (the same
  buffer viewed as [B, Hkv, G*Sq, D]);
- split-KV: the keys are cut into runs of 128-key tiles; each run writes a
  partial O / LSE into the caller's workspace and sdp_merge combines them.
Both must give sdp_fwd's function: every case is checked on every row against
the oracle, with canary-filled guard tails after O, LSE and the workspace.
"""
import numpy as np
import pytest
import torch

import gqa_flash_attention_gb300 as sdp
import oracle
from gqa_flash_attention_gb300 import workloads
from gqa_flash_attention_gb300.workloads import Workload
from parity import ORACLE_DTYPE, assert_within, compare

pytestmark = pytest.mark.gpu

DEBUG_SINGLE_CTA = 2
DEBUG_NO_PACK = 4


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gqa_flash_attention_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    sdp.lib()


def run(q, k, v, scale, kv_splits=1, guard=4096):
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    B, Hq, Sq, D = q.shape
    _, Hkv, Skv, _ = k.shape
    o_buf = torch.full((q.numel() + guard,), float("nan"), dtype=q.dtype, device=dev)
    l_buf = torch.full((B * Hq * Sq + guard,), float("nan"), dtype=torch.float32, device=dev)
    o = o_buf[:q.numel()].view(q.shape)
    lse = l_buf[:B * Hq * Sq].view(B, Hq, Sq)
    ws = None
    need = 0
    if kv_splits != 1:
        dt = sdp.SDP_BF16 if q.dtype == torch.bfloat16 else sdp.SDP_FP16
        need = sdp.splitkv_workspace_bytes(B, Hq, Hkv, Sq, Skv, D, dt, kv_splits)
        ws_buf = torch.full((need + guard,), 0x7F, dtype=torch.uint8, device=dev)
        ws = ws_buf[:max(need, 16)]
    sdp.sdp_fwd(qd, kd, vd, scale=scale, out=o, lse=lse, kv_splits=kv_splits, workspace=ws)
    assert sdp.poll_status() == sdp.SDP_OK
    assert torch.isnan(o_buf[q.numel():]).all(), "write past the end of O"
    assert torch.isnan(l_buf[B * Hq * Sq:]).all(), "write past the end of LSE"
    if ws is not None:
        assert (ws_buf[max(need, 16):] == 0x7F).all(), "write past the end of the workspace"
    return o, lse


def check(w: Workload, kv_splits=1):
    q, k, v = workloads.make_inputs(w)
    o, lse = run(q, k, v, w.softmax_scale, kv_splits=kv_splits)
    ref_o, ref_l = oracle.sdp_fwd(q, k, v, ORACLE_DTYPE[w.dtype], w.shape, w.softmax_scale)
    st = compare(o, lse, ref_o, ref_l, w.dtype)
    assert_within(st, w.dtype)
    return o, lse


# Packed shapes: G * Sq rows per KV head, Sq not a multiple of 128; ragged keys.
PACKED = [
    Workload("decode_g16_d256_fp16", 2, 32, 2, 1, 1000, 256, "fp16", seed=61),
    Workload("decode_g4_d128_bf16", 3, 16, 4, 1, 777, 128, "bf16", seed=62),
    Workload("sq5_g8_d128_fp16", 1, 8, 1, 5, 300, 128, "fp16", seed=63),
    Workload("sq16_g16_d256_bf16", 1, 32, 2, 16, 513, 256, "bf16", seed=64),
    Workload("sq200_g4_d128_fp16", 1, 8, 2, 200, 129, 128, "fp16", seed=65),
    Workload("sq33_g2_d256_fp16", 2, 4, 2, 33, 1, 256, "fp16", seed=66),
    Workload("sq1_g64_d128_fp16", 1, 64, 1, 1, 257, 128, "fp16", seed=67),
]


@pytest.mark.parametrize("w", PACKED, ids=lambda w: w.name)
def test_packed_heads_every_row(w):
    check(w)


@pytest.mark.parametrize("w", PACKED[:4], ids=lambda w: w.name)
def test_packing_matches_the_unpacked_launch(w):
    """Each output row's arithmetic does not depend on which rows share its
    tile, so the packed and unpacked launches (single-CTA kernel in both)
    agree bit for bit."""
    q, k, v = workloads.make_inputs(w)
    old = sdp.set_debug_flags(DEBUG_SINGLE_CTA)
    try:
        o1, l1 = run(q, k, v, w.softmax_scale)
        sdp.set_debug_flags(DEBUG_SINGLE_CTA | DEBUG_NO_PACK)
        o2, l2 = run(q, k, v, w.softmax_scale)
    finally:
        sdp.set_debug_flags(old)
    assert torch.equal(o1, o2)
    assert torch.equal(l1, l2)


SPLIT = [
    (Workload("split_decode_g16_d256_fp16", 1, 32, 2, 1, 4000, 256, "fp16", seed=71), 0),
    (Workload("split_decode_g4_d128_bf16", 2, 16, 4, 1, 3000, 128, "bf16", seed=72), 0),
    (Workload("split_decode_g4_d128_fp16_s3", 2, 16, 4, 1, 3000, 128, "fp16", seed=72), 3),
    (Workload("split_sq7_g8_d128_fp16_s5", 1, 8, 1, 7, 1300, 128, "fp16", seed=73), 5),
    (Workload("split_mha_d128_fp16_s4", 1, 2, 2, 256, 1025, 128, "fp16", seed=74), 4),
    (Workload("split_gqa2_d256_bf16_s2", 1, 4, 2, 300, 700, 256, "bf16", seed=75), 2),
    (Workload("split_one_tile_fp16", 1, 4, 1, 1, 100, 128, "fp16", seed=76), 8),
    (Workload("split_many_fp16", 1, 8, 2, 2, 2049, 128, "fp16", seed=77), 1000),
    (Workload("split_peaky_bf16", 1, 16, 2, 1, 5000, 128, "bf16", seed=78, peaky_k=True), 0),
]


@pytest.mark.parametrize("w,splits", SPLIT, ids=lambda x: x.name if isinstance(x, Workload) else str(x))
def test_split_kv_every_row(w, splits):
    check(w, kv_splits=splits)


@pytest.mark.parametrize("w,splits", SPLIT[:5], ids=lambda x: x.name if isinstance(x, Workload) else str(x))
def test_split_kv_single_cta(w, splits):
    old = sdp.set_debug_flags(DEBUG_SINGLE_CTA)
    try:
        check(w, kv_splits=splits)
    finally:
        sdp.set_debug_flags(old)


def test_split_counts_and_workspace_sizes():
    fp16 = sdp.SDP_FP16
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # decode, 32 heads over 2 KV heads: packed into 2 units, auto fills one wave
    n_kv = (16384 + 127) // 128
    s = sdp.splitkv_count(1, 32, 2, 1, 16384, 256, fp16, 0)
    tps = -(-n_kv // (sms // 2))
    assert s == -(-n_kv // tps)
    assert 2 * s <= sms
    assert sdp.splitkv_workspace_bytes(1, 32, 2, 1, 16384, 256, fp16, 0) == \
        -(-(s * 32 * 256 * 2) // 256) * 256 + s * 32 * 4
    # requests clamp to the KV tile count and even out
    assert sdp.splitkv_count(1, 4, 1, 1, 300, 128, fp16, 100) == 3
    assert sdp.splitkv_count(1, 4, 1, 1, 1000, 128, fp16, 5) == 4  # 8 tiles: 2 per split
    assert sdp.splitkv_count(1, 4, 1, 1, 1000, 128, fp16, 1) == 1
    assert sdp.splitkv_workspace_bytes(1, 4, 1, 1, 1000, 128, fp16, 1) == 0
    # enough units already: no split
    assert sdp.splitkv_count(8, 32, 8, 4096, 4096, 128, fp16, 0) == 1
    with pytest.raises(sdp.SdpError):
        sdp.splitkv_count(1, 4, 1, 1, 1000, 128, fp16, -1)


def test_split_kv_rejects_bad_workspace():
    dev = torch.device("cuda")
    q = torch.randn(1, 8, 1, 128, device=dev).half()
    k = torch.randn(1, 2, 2000, 128, device=dev).half()
    v = torch.randn(1, 2, 2000, 128, device=dev).half()
    o = torch.empty_like(q)
    need = sdp.splitkv_workspace_bytes(1, 8, 2, 1, 2000, 128, sdp.SDP_FP16, 4)
    assert need > 0
    ws = torch.empty(need + 64, dtype=torch.uint8, device=dev)

    def call(ws_ptr, ws_bytes, splits=4, o_ptr=None):
        return sdp.sdp_fwd_splitkv_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                       o.data_ptr() if o_ptr is None else o_ptr, 0, 1, 8, 2, 1, 2000, 128,
                                       0.088, sdp.SDP_FP16, splits, ws_ptr, ws_bytes,
                                       torch.cuda.current_stream().cuda_stream)

    assert call(ws.data_ptr(), need - 1) == sdp.SDP_ERR_INVALID_ARG
    assert call(0, need) == sdp.SDP_ERR_INVALID_ARG
    assert call(ws.data_ptr() + 8, need) == sdp.SDP_ERR_ALIGNMENT
    assert call(ws.data_ptr(), need, splits=-1) == sdp.SDP_ERR_INVALID_ARG
    assert call(ws.data_ptr(), need, o_ptr=ws.data_ptr() + 256) == sdp.SDP_ERR_INVALID_ARG
    assert call(ws.data_ptr(), need) == sdp.SDP_OK
    assert sdp.poll_status() == sdp.SDP_OK
    with pytest.raises(ValueError):
        sdp.sdp_fwd(q, k, v, causal=True, kv_splits=0)


def test_split_kv_is_deterministic_and_stream_ordered():
    w = SPLIT[0][0]
    q, k, v = workloads.make_inputs(w)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o1, l1 = sdp.sdp_fwd(qd, kd, vd, kv_splits=0, stream=s)
        o2, l2 = sdp.sdp_fwd(qd, kd, vd, kv_splits=0, stream=s)
    s.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("name", list(workloads.DECODE_WORKLOADS))
def test_full_size_decode_workloads(name):
    """The decode workloads in the benchmark's launch configuration (their
    split count), checked on every output row."""
    w = workloads.DECODE_WORKLOADS[name]
    check(w, kv_splits=w.kv_splits)


def test_split_kv_replays_from_a_cuda_graph():
    """Both launches of a split-KV call (attention into the workspace, then the
    merge) are capturable: a graph replay gives the eager call's result bit for bit."""
    w = SPLIT[0][0]
    q, k, v = (t.cuda() for t in workloads.make_inputs(w))
    dt = sdp.SDP_FP16
    need = sdp.splitkv_workspace_bytes(w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, dt, 0)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o_eager, l_eager = sdp.sdp_fwd(q, k, v, kv_splits=0, workspace=ws)
    o = torch.empty_like(q)
    lse = torch.empty_like(l_eager)
    sdp.sdp_fwd(q, k, v, out=o, lse=lse, kv_splits=0, workspace=ws)  # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        sdp.sdp_fwd(q, k, v, out=o, lse=lse, kv_splits=0, workspace=ws)
    o.zero_()
    lse.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert sdp.poll_status() == sdp.SDP_OK
    assert torch.equal(o, o_eager) and torch.equal(lse, l_eager)
