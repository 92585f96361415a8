"""CUDA path vs the fp64 oracle, through the C ABI, on the same seeded inputs.

Small cases are checked element by element on every output row; they span
several 128-row query tiles and 128-key KV tiles, ragged tails on both, and
the degenerate one-row / one-key cases. The five full-size workloads are run
in the same launch configuration the benchmark times and checked on a seeded
sample of 256 query rows per (batch, head), rows 0 and Sq-1 included.
"""
import math

import numpy as np
import pytest
import torch

import gqa_flash_attention_gb300 as sdp
import oracle
from gqa_flash_attention_gb300 import workloads
from gqa_flash_attention_gb300.workloads import Workload
from parity import ORACLE_DTYPE, assert_within, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gqa_flash_attention_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    sdp.lib()


def gpu_run(q, k, v, scale, guard=4096, causal=False):
    """Run through the C ABI into canary-filled buffers with guard tails."""
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    B, Hq, Sq, D = q.shape
    o_buf = torch.full((q.numel() + guard,), float("nan"), dtype=q.dtype, device=dev)
    l_buf = torch.full((B * Hq * Sq + guard,), float("nan"), dtype=torch.float32, device=dev)
    o = o_buf[:q.numel()].view(q.shape)
    lse = l_buf[:B * Hq * Sq].view(B, Hq, Sq)
    sdp.sdp_fwd(qd, kd, vd, scale=scale, out=o, lse=lse, causal=causal)
    assert sdp.poll_status() == sdp.SDP_OK
    assert torch.isnan(o_buf[q.numel():]).all(), "write past the end of O"
    assert torch.isnan(l_buf[B * Hq * Sq:]).all(), "write past the end of LSE"
    return o, lse


def check_full(w: Workload):
    q, k, v = workloads.make_inputs(w)
    o, lse = gpu_run(q, k, v, w.softmax_scale, causal=w.causal)
    ref_o, ref_l = oracle.sdp_fwd(q, k, v, ORACLE_DTYPE[w.dtype], w.shape, w.softmax_scale, causal=w.causal)
    st = compare(o, lse, ref_o, ref_l, w.dtype)
    assert_within(st, w.dtype)
    return st


SMALL = []
for D in (128, 256):
    for dt in ("fp16", "bf16"):
        SMALL += [
            Workload(f"one_{D}_{dt}", 1, 2, 1, 1, 1, D, dt, seed=31),
            Workload(f"tails_{D}_{dt}", 1, 2, 2, 127, 129, D, dt, seed=32),
            Workload(f"gqa2_{D}_{dt}", 1, 4, 2, 129, 300, D, dt, seed=33),
            Workload(f"gqa4_b2_{D}_{dt}", 2, 4, 1, 300, 1000, D, dt, seed=34),
            Workload(f"gqa16_{D}_{dt}", 1, 16, 1, 64, 127, D, dt, seed=35),
            Workload(f"mha_{D}_{dt}", 1, 4, 4, 200, 128, D, dt, seed=36),
            Workload(f"kv1_{D}_{dt}", 1, 2, 1, 130, 1, D, dt, seed=37),
        ]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_small_cases_every_row(w):
    # CTA-pair kernel wherever units pair within a KV group, else the single-CTA kernel
    check_full(w)


DEBUG_SINGLE_CTA = 2


@pytest.mark.parametrize("w", [w for w in SMALL if not w.name.startswith("one_")], ids=lambda w: w.name)
def test_single_cta_kernel_every_row(w):
    """The single-CTA kernel (used when units cannot pair) on the same cases."""
    old = sdp.set_debug_flags(DEBUG_SINGLE_CTA)
    try:
        check_full(w)
    finally:
        sdp.set_debug_flags(old)


DEBUG_PAIR_D128 = 8


@pytest.mark.parametrize("w", [w for w in SMALL if w.D == 128 and not w.name.startswith("one_")],
                         ids=lambda w: w.name)
def test_pair_kernel_at_d128_every_row(w):
    """Head dim 128 runs on single CTAs by default; the CTA-pair kernel, kept
    for it behind a flag, must give the same function."""
    old = sdp.set_debug_flags(DEBUG_PAIR_D128)
    try:
        check_full(w)
    finally:
        sdp.set_debug_flags(old)


@pytest.mark.parametrize("name", ["gqa4_b2_s8k_d128_bf16_peaky", "mha_b4_s16k_d128_fp16"])
def test_pair_kernel_at_d128_full_size_sampled(name):
    old = sdp.set_debug_flags(DEBUG_PAIR_D128)
    try:
        test_full_size_workload_sampled_rows(name)
    finally:
        sdp.set_debug_flags(old)


def test_smallest_workload_every_row():
    check_full(workloads.WORKLOADS["gqa4_s256_d128_fp16"])


@pytest.mark.parametrize("scale", [0.0, -0.0625, 0.5])
def test_scale_sign_and_zero(scale):
    check_full(Workload("scale", 1, 4, 2, 150, 260, 128, "fp16", seed=41, scale=scale))


@pytest.mark.parametrize("scale", [0.0, -0.0625])
@pytest.mark.parametrize("causal", [False, True])
def test_scale_sign_and_zero_on_cta_pairs(scale, causal):
    """256 query rows of two heads per group at D=256 (no head packing): CTA
    pairs, whose row extreme is a minimum when the scale is negative."""
    check_full(Workload("scale_pair", 1, 4, 2, 256, 260, 256, "bf16", seed=46, scale=scale, causal=causal))


def test_peaky_keys_small():
    check_full(Workload("peaky", 1, 8, 2, 256, 1024, 128, "bf16", seed=42, peaky_k=True))


@pytest.mark.parametrize("name", [n for n in workloads.ALL_WORKLOADS if n != "gqa4_s256_d128_fp16"])
def test_full_size_workload_sampled_rows(name):
    w = workloads.ALL_WORKLOADS[name]
    q, k, v = workloads.make_inputs(w)
    o, lse = gpu_run(q, k, v, w.softmax_scale, causal=w.causal)
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    rows = workloads.sample_rows(w, 256)
    ref_o, ref_l = oracle.sdp_fwd_rows(q, k, v, ORACLE_DTYPE[w.dtype], w.shape, w.softmax_scale, rows, causal=w.causal)
    idx = torch.from_numpy(rows.astype(np.int64)).to(o.device)
    o_s = torch.gather(o, 2, idx[..., None].expand(-1, -1, -1, w.D))
    l_s = torch.gather(lse, 2, idx)
    st = compare(o_s, l_s, ref_o, ref_l, w.dtype)
    assert_within(st, w.dtype)


def test_deterministic_and_stream_aware():
    w = Workload("det", 1, 8, 2, 300, 700, 256, "bf16", seed=43)
    q, k, v = (t.cuda() for t in workloads.make_inputs(w))
    o1, l1 = sdp.sdp_fwd(q, k, v)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        o2, l2 = sdp.sdp_fwd(q, k, v)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_without_lse():
    w = Workload("nolse", 1, 4, 1, 128, 256, 128, "fp16", seed=44)
    q, k, v = workloads.make_inputs(w)
    o, lse = sdp.sdp_fwd(q.cuda(), k.cuda(), v.cuda(), return_lse=False)
    assert lse is None
    ref_o, _ = oracle.sdp_fwd(q, k, v, oracle.FP16, w.shape, w.softmax_scale)
    st = compare(o, None, ref_o, None, "fp16")
    assert_within(st, "fp16")


def test_default_scale_is_inverse_sqrt_d():
    w = Workload("defscale", 1, 2, 1, 64, 64, 256, "fp16", seed=45)
    q, k, v = (t.cuda() for t in workloads.make_inputs(w))
    o1, _ = sdp.sdp_fwd(q, k, v)
    o2, _ = sdp.sdp_fwd(q, k, v, scale=1.0 / math.sqrt(256))
    assert torch.equal(o1, o2)


# ------------------------------------------------------------------- causal

CAUSAL = []
for D in (128, 256):
    for dt in ("fp16", "bf16"):
        CAUSAL += [
            Workload(f"causal_sq_eq_skv_gqa2_{D}_{dt}", 1, 4, 2, 300, 300, D, dt, seed=71, causal=True),
            Workload(f"causal_mha_{D}_{dt}", 2, 2, 2, 257, 257, D, dt, seed=72, causal=True),
            Workload(f"causal_sq_lt_skv_{D}_{dt}", 1, 4, 1, 129, 400, D, dt, seed=73, causal=True),
            Workload(f"causal_sq_gt_skv_{D}_{dt}", 1, 2, 1, 300, 130, D, dt, seed=74, causal=True),
            Workload(f"causal_one_key_{D}_{dt}", 1, 2, 1, 5, 1, D, dt, seed=75, causal=True),
        ]


@pytest.mark.parametrize("w", CAUSAL, ids=lambda w: w.name)
def test_causal_every_row(w):
    check_full(w)


@pytest.mark.parametrize("w", [w for w in CAUSAL if w.D == 256 and w.dtype == "bf16"], ids=lambda w: w.name)
def test_causal_single_cta_kernel_every_row(w):
    old = sdp.set_debug_flags(DEBUG_SINGLE_CTA)
    try:
        check_full(w)
    finally:
        sdp.set_debug_flags(old)


# Dense causal single-CTA launches order their units by query tile (longest first) inside blocks of
# ceil(4 / G) KV groups; these shapes leave a partial last block or a single short one.
CAUSAL_BLOCKS = [
    # MHA, five heads: blocks of four KV groups and of one; six query tiles, the last ragged
    Workload("causal_blk_mha5_d128_fp16", 1, 5, 5, 700, 700, 128, "fp16", seed=76, causal=True),
    # three heads per group (blocks of two groups), two batches, fewer queries than keys
    Workload("causal_blk_g3_b2_d128_bf16", 2, 6, 2, 450, 500, 128, "bf16", seed=77, causal=True),
    # three KV groups, fewer than a block
    Workload("causal_blk_mha_b3_d128_bf16", 3, 1, 1, 600, 600, 128, "bf16", seed=78, causal=True),
    # two heads per group, seven groups: blocks of two, two, two and one
    Workload("causal_blk_g2_d128_fp16", 1, 14, 7, 300, 300, 128, "fp16", seed=79, causal=True),
    # more queries than keys: the last query tiles see every key
    Workload("causal_blk_mha6_d128_bf16", 1, 6, 6, 520, 260, 128, "bf16", seed=80, causal=True),
]


@pytest.mark.parametrize("w", CAUSAL_BLOCKS, ids=lambda w: w.name)
def test_causal_unit_blocks_every_row(w):
    check_full(w)


def test_causal_unit_blocks_single_cta_at_d256_every_row():
    """Debug flag 2 at head dim 256, five MHA heads: the same block order on the single-CTA kernel."""
    old = sdp.set_debug_flags(DEBUG_SINGLE_CTA)
    try:
        check_full(Workload("causal_blk_mha5_d256_fp16", 1, 5, 5, 400, 400, 256, "fp16", seed=81, causal=True))
    finally:
        sdp.set_debug_flags(old)



def test_dense_call_replays_from_a_cuda_graph():
    w = workloads.WORKLOADS["gqa4_s256_d128_fp16"]
    q, k, v = (t.cuda() for t in workloads.make_inputs(w))
    o_eager, l_eager = sdp.sdp_fwd(q, k, v)
    o = torch.empty_like(q)
    lse = torch.empty_like(l_eager)
    sdp.sdp_fwd(q, k, v, out=o, lse=lse)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        sdp.sdp_fwd(q, k, v, out=o, lse=lse)
    o.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert sdp.poll_status() == sdp.SDP_OK
    assert torch.equal(o, o_eager) and torch.equal(lse, l_eager)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_large_scores_saturate_cleanly(dtype):
    """Inputs scaled by 24 so the scaled scores reach the thousands: almost every weight
    underflows to exactly 0 and each row copies (nearly) one V row; nothing
    overflows in the fp32 scaling, exponentials or sums."""
    w = Workload(f"large_{dtype}", 1, 4, 2, 200, 700, 128, dtype, seed=97)
    q, k, v = workloads.make_inputs(w)
    q, k = (q.float() * 24).to(q.dtype), (k.float() * 24).to(k.dtype)
    o, lse = gpu_run(q, k, v, w.softmax_scale)
    ref_o, ref_l = oracle.sdp_fwd(q, k, v, ORACLE_DTYPE[dtype], w.shape, w.softmax_scale)
    st = compare(o, lse, ref_o, ref_l, dtype)
    assert st["nan_o"] == 0 and st["nan_lse"] == 0
    assert st["max_abs"] <= (2e-2 if dtype == "fp16" else 4e-2), st
    assert st["lse_max_abs"] <= 1e-6 * max(1.0, float(np.abs(ref_l).max())) * 8, st


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_peaky_keys_on_cta_pairs(dtype):
    """1 % of the key rows scaled by 8 at D=256 with two heads per group and whole query tiles (CTA
    pairs): a row's maximum jumps when a scaled key arrives in a later tile, so O is rescaled before
    the first part of P is handed to the PV MMAs."""
    check_full(Workload(f"peaky_pair_{dtype}", 1, 4, 2, 256, 2048, 256, dtype, seed=47, peaky_k=True))


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_large_scores_on_cta_pairs(dtype):
    """The saturating case above at D=256 on CTA pairs (whole query tiles, two heads per group)."""
    w = Workload(f"large_pair_{dtype}", 1, 4, 2, 256, 700, 256, dtype, seed=98)
    q, k, v = workloads.make_inputs(w)
    q, k = (q.float() * 24).to(q.dtype), (k.float() * 24).to(k.dtype)
    o, lse = gpu_run(q, k, v, w.softmax_scale)
    ref_o, ref_l = oracle.sdp_fwd(q, k, v, ORACLE_DTYPE[dtype], w.shape, w.softmax_scale)
    st = compare(o, lse, ref_o, ref_l, dtype)
    assert st["nan_o"] == 0 and st["nan_lse"] == 0
    assert st["max_abs"] <= (2e-2 if dtype == "fp16" else 4e-2), st
    assert st["lse_max_abs"] <= 1e-6 * max(1.0, float(np.abs(ref_l).max())) * 8, st


DEBUG_NO_PERSIST = 16


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_persistent_pair_kernel_every_row(dtype):
    """160 units (more than the SMs) of a dense, non-causal D=256 launch run on the persistent CTA-pair
    kernel: each cluster takes several unit pairs, so tile counters, ring positions and barrier phases
    carry over unit boundaries; the last KV tile is ragged."""
    check_full(Workload(f"persist_{dtype}", 1, 8, 2, 2560, 700, 256, dtype, seed=48))


def test_persistent_pair_kernel_matches_the_per_unit_launch_bit_for_bit():
    """The persistent form changes the schedule, not the arithmetic: same O and LSE bits as one unit
    pair per cluster."""
    w = Workload("persist_eq", 1, 8, 2, 2560, 1000, 256, "fp16", seed=49)
    q, k, v = (t.cuda() for t in workloads.make_inputs(w))
    o1, l1 = sdp.sdp_fwd(q, k, v)
    assert sdp.poll_status() == sdp.SDP_OK
    old = sdp.set_debug_flags(DEBUG_NO_PERSIST)
    try:
        o2, l2 = sdp.sdp_fwd(q, k, v)
        assert sdp.poll_status() == sdp.SDP_OK
    finally:
        sdp.set_debug_flags(old)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)



@pytest.mark.parametrize("w", [
    # 160 causal units at D=256, two heads per group: the persistent CTA-pair kernel, units of 1 to 20 KV tiles
    Workload("persist_causal_fp16", 1, 8, 2, 2560, 2560, 256, "fp16", seed=87, causal=True),
    # more query rows than keys: the late units all read the 8 KV tiles, ragged last tile
    Workload("persist_causal_sq_gt_skv_bf16", 1, 8, 2, 2560, 1000, 256, "bf16", seed=88, causal=True),
], ids=lambda w: w.name)
def test_persistent_pair_kernel_causal_every_row(w):
    """Causal launches with more units than SMs run the persistent CTA-pair kernel: unit pairs of
    different lengths, longest first, walked in alternating directions; the diagonal tile of every
    unit is masked per row."""
    check_full(w)


def test_persistent_pair_kernel_causal_matches_the_per_unit_launch_bit_for_bit():
    w = Workload("persist_causal_eq", 1, 8, 2, 2560, 3000, 256, "fp16", seed=89, causal=True)
    q, k, v = (t.cuda() for t in workloads.make_inputs(w))
    o1, l1 = sdp.sdp_fwd(q, k, v, causal=True)
    assert sdp.poll_status() == sdp.SDP_OK
    old = sdp.set_debug_flags(DEBUG_NO_PERSIST)
    try:
        o2, l2 = sdp.sdp_fwd(q, k, v, causal=True)
        assert sdp.poll_status() == sdp.SDP_OK
    finally:
        sdp.set_debug_flags(old)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)

