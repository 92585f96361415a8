"""Variable-length batches (sdp_fwd_varlen) against the fp64 oracle.

Sequences of different lengths are packed back to back in (token, head, dim)
layout; every query row must attend to its own sequence's keys only. Small
batches are checked on every row, with ragged tails, one-row and empty
sequences, sequences without keys, more keys than queries and the reverse,
causal and not. The long-tailed full-size batches run in the benchmark's
launch configuration and are checked on a seeded sample of rows per
(sequence, head) against the dense oracle on that sequence alone.
"""
import numpy as np
import pytest
import torch

import gqa_flash_attention_gb300 as sdp
import oracle
from gqa_flash_attention_gb300 import workloads
from gqa_flash_attention_gb300.workloads import VarlenWorkload
from parity import ORACLE_DTYPE, assert_within, compare

pytestmark = pytest.mark.gpu

DEBUG_SINGLE_CTA = 2
DEBUG_PAIR_D128 = 8
DEBUG_FULL_VARLEN_GRID = 32


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gqa_flash_attention_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    sdp.lib()


def run(w: VarlenWorkload, q, k, v, guard=4096):
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    cq = torch.from_numpy(w.cu_q).to(dev)
    ck = torch.from_numpy(w.cu_k).to(dev)
    o_buf = torch.full((q.numel() + guard,), float("nan"), dtype=q.dtype, device=dev)
    l_buf = torch.full((w.Hq * w.total_q + guard,), float("nan"), dtype=torch.float32, device=dev)
    o = o_buf[:q.numel()].view(q.shape)
    lse = l_buf[:w.Hq * w.total_q].view(w.Hq, w.total_q)
    sdp.sdp_fwd_varlen(qd, kd, vd, cq, ck, w.max_q, scale=w.softmax_scale, causal=w.causal, out=o, lse=lse)
    assert sdp.poll_status() == sdp.SDP_OK
    assert torch.isnan(o_buf[q.numel():]).all(), "write past the end of O"
    assert torch.isnan(l_buf[w.Hq * w.total_q:]).all(), "write past the end of LSE"
    return o, lse


def check_every_row(w: VarlenWorkload):
    q, k, v = workloads.make_varlen_inputs(w)
    o, lse = run(w, q, k, v)
    ref_o, ref_l = oracle.sdp_fwd_varlen(q, k, v, ORACLE_DTYPE[w.dtype], w.cu_q, w.cu_k, w.softmax_scale,
                                         causal=w.causal)
    o_c, l_c = o.double().cpu().numpy(), lse.double().cpu().numpy()
    # rows that see no key: exactly 0 and -inf
    seen_none = np.zeros(w.total_q, dtype=bool)
    for b in range(w.nseq):
        if w.lens_k[b] == 0:
            seen_none[w.cu_q[b]:w.cu_q[b + 1]] = True
    assert np.all(o_c[seen_none] == 0.0)
    assert np.all(np.isneginf(l_c[:, seen_none]))
    keep = ~seen_none
    st = compare(o_c[keep], l_c[:, keep], ref_o[keep], ref_l[:, keep], w.dtype)
    assert_within(st, w.dtype)
    return o, lse


SMALL = []
for D in (128, 256):
    for dt in ("fp16", "bf16"):
        SMALL += [
            VarlenWorkload(f"mixed_{D}_{dt}", (1, 127, 128, 129, 300), (5, 127, 128, 260, 300), 4, 2, D, dt,
                           seed=81),
            VarlenWorkload(f"empty_{D}_{dt}", (0, 40, 0, 200, 7), (10, 0, 0, 150, 33), 8, 2, D, dt, seed=82),
            VarlenWorkload(f"causal_{D}_{dt}", (50, 257, 3, 140), (50, 257, 90, 100), 4, 1, D, dt, seed=83,
                           causal=True),
        ]
SMALL += [
    VarlenWorkload("mha_many_128_fp16", tuple(range(1, 40, 3)), tuple(range(40, 1, -3)), 2, 2, 128, "fp16",
                   seed=84),
    VarlenWorkload("gqa16_long_256_bf16", (700, 1), (1300, 2), 16, 1, 256, "bf16", seed=85),
    VarlenWorkload("causal_more_keys_128_bf16", (33, 500), (400, 129), 4, 4, 128, "bf16", seed=86, causal=True),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_small_batches_every_row(w):
    check_every_row(w)


@pytest.mark.parametrize("flags", [DEBUG_SINGLE_CTA, DEBUG_PAIR_D128], ids=["single_cta", "pair_at_d128"])
@pytest.mark.parametrize("w", [w for w in SMALL if w.Hq // w.Hkv % 2 == 0], ids=lambda w: w.name)
def test_small_batches_other_kernel(w, flags):
    """Batches whose groups pair up run on CTA pairs by default at D=256 and on
    single CTAs at D=128; the other kernel must give the same function."""
    old = sdp.set_debug_flags(flags)
    try:
        check_every_row(w)
    finally:
        sdp.set_debug_flags(old)


@pytest.mark.parametrize("causal", [False, True])
def test_one_sequence_equals_the_dense_call(causal):
    """A batch of one sequence is sdp_fwd on the transposed layout: with both
    on the single-CTA kernel the per-row arithmetic is the same, so bit for bit."""
    w = VarlenWorkload("one", (300,), (420,), 8, 2, 128, "fp16", seed=87, causal=causal)
    q, k, v = workloads.make_varlen_inputs(w)
    dev = torch.device("cuda")
    qd, kd, vd = (t.permute(1, 0, 2).unsqueeze(0).contiguous().to(dev) for t in (q, k, v))
    old = sdp.set_debug_flags(DEBUG_SINGLE_CTA)
    try:
        o, lse = run(w, q, k, v)
        od, ld = sdp.sdp_fwd(qd, kd, vd, scale=w.softmax_scale, causal=causal)
        assert sdp.poll_status() == sdp.SDP_OK
    finally:
        sdp.set_debug_flags(old)
    assert torch.equal(o, od[0].permute(1, 0, 2))
    assert torch.equal(lse, ld[0])


@pytest.mark.parametrize("flags", [0, DEBUG_FULL_VARLEN_GRID], ids=["compact_grid", "full_grid"])
def test_bad_offsets_are_reported_and_skipped(flags):
    old = sdp.set_debug_flags(flags)
    try:
        _bad_offsets()
    finally:
        sdp.set_debug_flags(old)


def _bad_offsets():
    dev = torch.device("cuda")
    w = VarlenWorkload("bad", (100, 200), (100, 200), 4, 1, 128, "fp16", seed=88)
    q, k, v = (t.to(dev) for t in workloads.make_varlen_inputs(w))
    good_q = torch.from_numpy(w.cu_q).to(dev)
    good_k = torch.from_numpy(w.cu_k).to(dev)
    cases = [
        (torch.tensor([0, 150, 120], dtype=torch.int32, device=dev), good_k, 200),  # decreasing, past total
        (good_q, torch.tensor([0, 100, 999], dtype=torch.int32, device=dev), 200),  # past total_k
        (good_q, good_k, 100),                                # 200 rows > max_seqlen_q rounded up to 128
    ]
    for cq, ck, mx in cases:
        o = torch.zeros_like(q)
        sdp.sdp_fwd_varlen(q, k, v, cq, ck, mx, out=o)
        assert sdp.poll_status() == sdp.SDP_ERR_BAD_SEQLENS
        assert sdp.last_status_detail() & 0xFF == 7
    # the status word was cleared: a good call afterwards reports OK
    sdp.sdp_fwd_varlen(q, k, v, good_q, good_k, 200)
    assert sdp.poll_status() == sdp.SDP_OK


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_compact_grid_matches_the_full_grid_bit_for_bit(w):
    """The compact grid (only the query tiles that exist, each CTA finding its
    tile from the offsets) and the full grid (the longest sequence's tiles for
    every sequence) run the same per-tile arithmetic: identical outputs."""
    q, k, v = workloads.make_varlen_inputs(w)
    o, lse = run(w, q, k, v)
    old = sdp.set_debug_flags(DEBUG_FULL_VARLEN_GRID)
    try:
        of, lf = run(w, q, k, v)
    finally:
        sdp.set_debug_flags(old)
    assert torch.equal(o, of)
    assert torch.equal(lse, lf)


def _many(n, causal, seed):
    rng = np.random.default_rng(seed)
    lq = tuple(int(x) for x in rng.integers(0, 300, size=n))
    lk = tuple(int(x) for x in rng.integers(0, 300, size=n))
    return VarlenWorkload(f"many{n}_{'causal' if causal else 'full'}", lq, lk, 4, 2, 128, "bf16", seed=seed,
                          causal=causal)


# Sequence counts on both sides of the limits up to which the compact grid is used
# (512 sequences without the causal mask, 64 with it), plus one long sequence after
# many short ones.
MANY = [_many(64, True, 91), _many(65, True, 92), _many(100, False, 93), _many(513, False, 94),
        VarlenWorkload("short_then_long", (1,) * 40 + (1000,), (1,) * 40 + (1000,), 4, 1, 256, "fp16", seed=95,
                       causal=True)]


@pytest.mark.parametrize("w", MANY, ids=lambda w: w.name)
def test_many_sequences_every_row(w):
    check_every_row(w)


def test_zero_query_rows_is_a_no_op():
    dev = torch.device("cuda")
    q = torch.empty(0, 4, 128, dtype=torch.float16, device=dev)
    k = torch.randn(10, 2, 128, device=dev).half()
    cu = torch.tensor([0, 0], dtype=torch.int32, device=dev)
    ck = torch.tensor([0, 10], dtype=torch.int32, device=dev)
    o, lse = sdp.sdp_fwd_varlen(q, k, k.clone(), cu, ck, 0)
    assert o.shape == (0, 4, 128) and lse.shape == (4, 0)
    assert sdp.poll_status() == sdp.SDP_OK


@pytest.mark.parametrize("name", list(workloads.VARLEN_WORKLOADS))
def test_full_size_batches_sampled(name):
    """The benchmark's batches, checked on 8 seeded rows per (sequence, head)
    (first and last row included) against the dense oracle on that sequence."""
    w = workloads.VARLEN_WORKLOADS[name]
    q, k, v = workloads.make_varlen_inputs(w)
    o, lse = run(w, q, k, v)
    o_c, l_c = o.cpu(), lse.cpu()
    rng = np.random.default_rng(w.seed + 1000)
    got_o, got_l, ref_o, ref_l = [], [], [], []
    for b in range(w.nseq):
        lq, lk = w.lens_q[b], w.lens_k[b]
        if lq == 0 or lk == 0:
            continue
        qs = q[w.cu_q[b]:w.cu_q[b + 1]].permute(1, 0, 2).unsqueeze(0).contiguous()
        ks = k[w.cu_k[b]:w.cu_k[b + 1]].permute(1, 0, 2).unsqueeze(0).contiguous()
        vs = v[w.cu_k[b]:w.cu_k[b + 1]].permute(1, 0, 2).unsqueeze(0).contiguous()
        m = min(8, lq)
        rows = np.empty((1, w.Hq, m), dtype=np.int32)
        for h in range(w.Hq):
            mid = rng.choice(np.arange(1, lq - 1), size=m - 2, replace=False) if m > 2 else []
            rows[0, h] = np.sort(np.concatenate([[0], mid, [lq - 1]])[:m]).astype(np.int32)
        ro, rl = oracle.sdp_fwd_rows(qs, ks, vs, ORACLE_DTYPE[w.dtype], (1, w.Hq, w.Hkv, lq, lk, w.D),
                                     w.softmax_scale, rows, causal=w.causal)
        for h in range(w.Hq):
            tok = w.cu_q[b] + rows[0, h]
            got_o.append(o_c[tok, h].double().numpy())
            got_l.append(l_c[h, tok].double().numpy())
            ref_o.append(ro[0, h])
            ref_l.append(rl[0, h])
    st = compare(np.concatenate(got_o), np.concatenate(got_l), np.concatenate(ref_o), np.concatenate(ref_l),
                 w.dtype)
    assert_within(st, w.dtype)


DEBUG_NO_PERSIST = 16

# Causal batches at D=256 with an even group size and more units than SMs: the persistent
# CTA-pair kernel (unit pairs longest first, walked in alternating directions), with empty and
# key-less sequences, ragged tails, more keys than queries and the reverse. (The same batches
# without the causal mask run on the per-unit CTA-pair kernel.)
PAIRED = [VarlenWorkload(f"pairs_{'causal' if causal else 'full'}_{dt}", (0, 700, 3, 1100, 129, 40, 1),
                         (10, 650, 0, 1200, 260, 40, 0), 16, 4, 256, dt, seed=96 + causal, causal=causal)
          for dt in ("fp16", "bf16") for causal in (False, True)]
PERSIST = [w for w in PAIRED if w.causal]


@pytest.mark.parametrize("w", PAIRED, ids=lambda w: w.name)
def test_batches_with_many_units_every_row(w):
    check_every_row(w)


@pytest.mark.parametrize("flags", [DEBUG_NO_PERSIST, DEBUG_FULL_VARLEN_GRID], ids=["per_unit", "full_grid"])
@pytest.mark.parametrize("w", PERSIST, ids=lambda w: w.name)
def test_persistent_pair_kernel_matches_other_launches_bit_for_bit(w, flags):
    """The persistent walk changes the schedule, not the arithmetic: the same bits as one unit pair
    per cluster (flag 16), and on the full grid of the longest sequence's tiles (flag 32)."""
    q, k, v = workloads.make_varlen_inputs(w)
    o, lse = run(w, q, k, v)
    old = sdp.set_debug_flags(flags)
    try:
        o2, l2 = run(w, q, k, v)
    finally:
        sdp.set_debug_flags(old)
    assert torch.equal(o, o2) and torch.equal(lse, l2)


def test_bad_offsets_on_the_persistent_kernel():
    dev = torch.device("cuda")
    w = VarlenWorkload("bad256", (1000, 1200), (1000, 1200), 16, 2, 256, "fp16", seed=98, causal=True)
    q, k, v = (t.to(dev) for t in workloads.make_varlen_inputs(w))
    good_q = torch.from_numpy(w.cu_q).to(dev)
    good_k = torch.from_numpy(w.cu_k).to(dev)
    bad_k = torch.tensor([0, 1000, 9999], dtype=torch.int32, device=dev)  # past total_k
    o = torch.zeros_like(q)
    sdp.sdp_fwd_varlen(q, k, v, good_q, bad_k, 1200, out=o, causal=True)
    assert sdp.poll_status() == sdp.SDP_ERR_BAD_SEQLENS
    assert sdp.last_status_detail() & 0xFF == 7
    o, lse = sdp.sdp_fwd_varlen(q, k, v, good_q, good_k, 1200, causal=True)
    assert sdp.poll_status() == sdp.SDP_OK
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
