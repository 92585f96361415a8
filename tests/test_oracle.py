"""Pins of the fp64 oracle against things other than itself.

Each test fixes the oracle to a closed form, an invariant of softmax
attention, an arbitrary-precision brute force, or PyTorch's float64 CPU
attention, so that a dropped term, a wrong sign or index, a wrong head
mapping or a transposed operand fails at least one of them.

The method: single-pass softmax attention with grouped-query heads, as on the
"xe2-sdp-hd256" page (sections "HD=256 Architecture Differences" and
"Performance Testing") and the "xe2-sdp-bf16" page (sections "Data flow
diagram" and "CPU reference must match input type").
"""
import math

import mpmath
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from gqa_flash_attention_gb300 import workloads

FP16, BF16 = oracle.FP16, oracle.BF16
TD = {FP16: torch.float16, BF16: torch.bfloat16}


def rand_qkv(B, Hq, Hkv, Sq, Skv, D, dtype, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(B, Hq, Sq, D, generator=g) * std).to(TD[dtype])
    k = (torch.randn(B, Hkv, Skv, D, generator=g) * std).to(TD[dtype])
    v = torch.randn(B, Hkv, Skv, D, generator=g).to(TD[dtype])
    return q, k, v


def run(q, k, v, dtype, scale):
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    return oracle.sdp_fwd(q, k, v, dtype, (B, Hq, Hkv, Sq, Skv, D), scale)


# ---------------------------------------------------------------- decoders

def test_fp16_decoder_matches_numpy_on_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.fp16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_bf16_decoder_matches_float32_prefix_on_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32)
    with np.errstate(invalid="ignore"):  # signalling-NaN patterns widen quietly to NaN
        ref = (bits << 16).view(np.float32).astype(np.float64)  # bf16 is the top half of fp32
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


# ------------------------------------------------------- library reference

@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,D", [
    (1, 4, 1, 5, 7, 16),
    (2, 4, 2, 9, 3, 32),
    (1, 6, 6, 4, 33, 8),
    (1, 8, 2, 17, 65, 64),
    (2, 3, 1, 1, 1, 16),
])
def test_matches_torch_float64_sdpa(dtype, B, Hq, Hkv, Sq, Skv, D):
    q, k, v = rand_qkv(B, Hq, Hkv, Sq, Skv, D, dtype, seed=Sq * 131 + Skv)
    scale = 0.7 / math.sqrt(D)
    o, lse = run(q, k, v, dtype, scale)
    qd, kd, vd = q.double(), k.double(), v.double()
    ref = F.scaled_dot_product_attention(qd, kd, vd, scale=scale, enable_gqa=(Hq != Hkv))
    G = Hq // Hkv
    s = qd @ kd.repeat_interleave(G, dim=1).transpose(-1, -2) * scale
    ref_lse = torch.logsumexp(s, dim=-1)
    assert np.abs(o - ref.numpy()).max() <= 1e-12
    assert np.abs(lse - ref_lse.numpy()).max() <= 1e-12


# ------------------------------------------------------------- brute force

def test_brute_force_arbitrary_precision():
    """exp(s_j) / sum exp(s) with 50 significant digits and no max shift."""
    B, Hq, Hkv, Sq, Skv, D = 1, 4, 2, 3, 5, 4
    q, k, v = rand_qkv(B, Hq, Hkv, Sq, Skv, D, FP16, seed=7)
    scale = 0.5
    o, lse = run(q, k, v, FP16, scale)
    mpmath.mp.dps = 50
    qd, kd, vd = q.double().numpy(), k.double().numpy(), v.double().numpy()
    for h in range(Hq):
        g = h // (Hq // Hkv)
        for i in range(Sq):
            s = [mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(float(qd[0, h, i, d])) * mpmath.mpf(float(kd[0, g, j, d]))
                                                 for d in range(D)) for j in range(Skv)]
            e = [mpmath.exp(x) for x in s]
            z = mpmath.fsum(e)
            for d in range(D):
                exact = mpmath.fsum(e[j] * mpmath.mpf(float(vd[0, g, j, d])) for j in range(Skv)) / z
                assert abs(float(exact) - o[0, h, i, d]) <= 1e-13 * max(1.0, abs(float(exact)))
            assert abs(float(mpmath.log(z)) - lse[0, h, i]) <= 1e-13


# ------------------------------------------------------------ closed forms

@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_single_key_returns_its_value_row(dtype):
    q, k, v = rand_qkv(1, 4, 2, 6, 1, 16, dtype, seed=3)
    scale = 0.3
    o, lse = run(q, k, v, dtype, scale)
    vd, qd, kd = v.double().numpy(), q.double().numpy(), k.double().numpy()
    for h in range(4):
        g = h // 2
        assert np.array_equal(o[0, h], np.broadcast_to(vd[0, g, 0], (6, 16)))
        s0 = np.array([math.fsum(qd[0, h, i] * kd[0, g, 0]) * scale for i in range(6)])
        assert np.abs(lse[0, h] - s0).max() <= 1e-12


def test_zero_scale_gives_column_mean_and_log_count():
    q, k, v = rand_qkv(1, 2, 1, 3, 37, 8, FP16, seed=4)
    o, lse = run(q, k, v, FP16, 0.0)
    mean = v.double().numpy()[0, 0].mean(axis=0)
    assert np.abs(o[0] - mean).max() <= 1e-13
    assert np.abs(lse - math.log(37)).max() <= 1e-13


def test_two_keys_is_a_logistic_mix():
    q, k, v = rand_qkv(1, 1, 1, 4, 2, 16, FP16, seed=5)
    scale = 0.25
    o, lse = run(q, k, v, FP16, scale)
    qd, kd, vd = q.double().numpy()[0, 0], k.double().numpy()[0, 0], v.double().numpy()[0, 0]
    for i in range(4):
        s1 = scale * math.fsum(qd[i] * kd[0])
        s2 = scale * math.fsum(qd[i] * kd[1])
        w1 = 1.0 / (1.0 + math.exp(s2 - s1))
        w2 = 1.0 / (1.0 + math.exp(s1 - s2))
        assert np.abs(o[0, 0, i] - (w1 * vd[0] + w2 * vd[1])).max() <= 1e-13
        assert abs(lse[0, 0, i] - (max(s1, s2) + math.log1p(math.exp(-abs(s1 - s2))))) <= 1e-13


def test_constant_values_give_that_constant():
    q, k, _ = rand_qkv(1, 4, 2, 7, 29, 32, BF16, seed=6)
    row = torch.linspace(-3, 3, 32).to(torch.bfloat16)
    v = row.expand(1, 2, 29, 32).contiguous()
    o, _ = run(q, k, v, BF16, 1.0 / math.sqrt(32))
    assert np.abs(o - row.double().numpy()).max() <= 1e-13


# -------------------------------------------------------------- invariants

def test_softmax_row_sums_to_one():
    shape = (1, 4, 2, 9, 50, 16)
    q, k, v = rand_qkv(*shape, FP16, seed=8, std=2.0)
    for h in range(4):
        for i in (0, 4, 8):
            p, _, _ = oracle.row_probs(q, k, v, FP16, shape, 0.5, 0, h, i)
            assert (p >= 0).all()
            assert abs(p.sum() - 1.0) <= 1e-12


def test_row_weights_match_torch_softmax():
    """The weights themselves, on a grouped case where h // G differs from h % Hkv."""
    shape = (2, 6, 3, 5, 21, 16)
    q, k, v = rand_qkv(*shape, BF16, seed=18)
    o_all, l_all = oracle.sdp_fwd(q, k, v, BF16, shape, 0.35)
    for b, h, i in [(0, 1, 0), (1, 3, 4), (0, 5, 2), (1, 4, 3)]:
        p, o, lse = oracle.row_probs(q, k, v, BF16, shape, 0.35, b, h, i)
        s = k.double()[b, h // 2] @ q.double()[b, h, i] * 0.35
        assert np.abs(p - torch.softmax(s, dim=0).numpy()).max() <= 1e-14
        assert np.array_equal(o, o_all[b, h, i]) and lse == l_all[b, h, i]


def test_dominant_key_selects_its_value_row():
    D, Skv = 16, 40
    q = torch.zeros(1, 1, 1, D)
    q[..., 0] = 4.0
    g = torch.Generator().manual_seed(9)
    k = torch.rand(1, 1, Skv, D, generator=g) * 2 - 1
    k[0, 0, 23, 0] = 64.0  # score 256 against at most 4 for every other key
    v = torch.randn(1, 1, Skv, D, generator=g)
    q, k, v = q.half(), k.half(), v.half()
    o, _ = run(q, k, v, FP16, 1.0)
    assert np.abs(o[0, 0, 0] - v.double().numpy()[0, 0, 23]).max() <= 1e-12


def test_large_scores_stay_finite():
    """Scores near 1e4: the maximum shift keeps every exponential finite."""
    D, Skv = 8, 16
    g = torch.Generator().manual_seed(10)
    q = (torch.rand(1, 1, 2, D, generator=g) * 100).half()
    k = (torch.rand(1, 1, Skv, D, generator=g) * 100).half()
    v = torch.randn(1, 1, Skv, D, generator=g).half()
    o, lse = run(q, k, v, FP16, 1.0)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    s = q.double()[0, 0] @ k.double()[0, 0].T
    top = s.argmax(dim=1)
    for i in range(2):
        srt = torch.sort(s[i], descending=True).values
        if srt[0] - srt[1] > 50:
            assert np.abs(o[0, 0, i] - v.double().numpy()[0, 0, top[i]]).max() <= 1e-12


def test_joint_key_value_permutation_is_invisible():
    shape = (2, 4, 2, 11, 31, 16)
    q, k, v = rand_qkv(*shape, BF16, seed=11)
    perm = torch.randperm(31, generator=torch.Generator().manual_seed(12))
    o1, l1 = run(q, k, v, BF16, 0.4)
    o2, l2 = run(q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous(), BF16, 0.4)
    assert np.abs(o1 - o2).max() <= 1e-13
    assert np.abs(l1 - l2).max() <= 1e-13


def test_common_key_shift_moves_only_the_lse():
    """K_j -> K_j + w shifts every score of row i by scale * q_i.w: O is
    unchanged and LSE moves by exactly that amount. Integer-valued entries
    keep both inputs exact in fp16."""
    B, Hq, Hkv, Sq, Skv, D = 1, 2, 1, 5, 13, 8
    g = torch.Generator().manual_seed(13)
    q = torch.randint(-3, 4, (B, Hq, Sq, D), generator=g).half()
    k = torch.randint(-8, 9, (B, Hkv, Skv, D), generator=g).half()
    w = torch.randint(-4, 5, (D,), generator=g).half()
    v = torch.randn(B, Hkv, Skv, D, generator=g).half()
    scale = 0.125
    o1, l1 = run(q, k, v, FP16, scale)
    o2, l2 = run(q, (k + w).contiguous(), v, FP16, scale)
    shift = scale * (q.double() @ w.double()).numpy()  # [B, Hq, Sq]
    assert np.abs(o1 - o2).max() <= 1e-12
    assert np.abs((l2 - l1) - shift).max() <= 1e-12


@pytest.mark.parametrize("G", [2, 4, 16])
def test_grouped_heads_equal_multi_head_on_repeated_kv(G):
    """Query head h reads KV head h // G: the same as MHA on K, V repeated G
    times per head (repeat_interleave order)."""
    Hkv = 2
    shape = (1, G * Hkv, Hkv, 6, 19, 16)
    q, k, v = rand_qkv(*shape, FP16, seed=14 + G)
    o1, l1 = run(q, k, v, FP16, 0.3)
    o2, l2 = run(q, k.repeat_interleave(G, dim=1).contiguous(), v.repeat_interleave(G, dim=1).contiguous(),
                 FP16, 0.3)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # and not the modulo mapping: head 1 reads KV head 0, not KV head 1
    o3, _ = run(q[:, :Hkv].contiguous(), k, v, FP16, 0.3)  # MHA over the first Hkv heads
    assert not np.allclose(o1[:, 1], o3[:, 1])


def test_row_subset_equals_full_evaluation():
    w = workloads.Workload("t", 1, 4, 2, 70, 45, 32, "bf16", seed=21)
    q, k, v = workloads.make_inputs(w)
    full_o, full_l = oracle.sdp_fwd(q, k, v, BF16, w.shape, w.softmax_scale)
    rows = workloads.sample_rows(w, n=9)
    o, l = oracle.sdp_fwd_rows(q, k, v, BF16, w.shape, w.softmax_scale, rows)
    for h in range(4):
        assert np.array_equal(o[0, h], full_o[0, h, rows[0, h]])
        assert np.array_equal(l[0, h], full_l[0, h, rows[0, h]])


def test_rejects_bad_shapes():
    q, k, v = rand_qkv(1, 3, 2, 2, 2, 8, FP16, seed=1)
    with pytest.raises(ValueError):
        oracle.sdp_fwd(q, k, v, FP16, (1, 3, 2, 2, 2, 8), 1.0)
    rows = np.full((1, 3, 1), 5, dtype=np.int32)
    q, k, v = rand_qkv(1, 3, 1, 2, 2, 8, FP16, seed=1)
    with pytest.raises(ValueError):
        oracle.sdp_fwd_rows(q, k, v, FP16, (1, 3, 1, 2, 2, 8), 1.0, rows)


# ------------------------------------------------------------------- causal

@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,D", [
    (1, 4, 1, 9, 9, 16),
    (2, 4, 2, 13, 7, 32),   # more queries than keys: late rows see every key
    (1, 2, 2, 5, 23, 8),    # more keys than queries: row i still sees keys 0..i only
])
def test_causal_matches_torch_float64_sdpa(dtype, B, Hq, Hkv, Sq, Skv, D):
    """Top-left alignment: row i sees keys 0..i (torch's is_causal convention)."""
    q, k, v = rand_qkv(B, Hq, Hkv, Sq, Skv, D, dtype, seed=Sq * 31 + Skv)
    scale = 0.6 / math.sqrt(D)
    o, lse = oracle.sdp_fwd(q, k, v, dtype, (B, Hq, Hkv, Sq, Skv, D), scale, causal=True)
    G = Hq // Hkv
    qd, kd, vd = q.double(), k.double().repeat_interleave(G, dim=1), v.double().repeat_interleave(G, dim=1)
    ref = F.scaled_dot_product_attention(qd, kd, vd, scale=scale, is_causal=True)
    s = qd @ kd.transpose(-1, -2) * scale
    mask = torch.ones(Sq, Skv, dtype=torch.bool).tril()
    ref_lse = torch.logsumexp(s.masked_fill(~mask, float("-inf")), dim=-1)
    assert np.abs(o - ref.numpy()).max() <= 1e-12
    assert np.abs(lse - ref_lse.numpy()).max() <= 1e-12


def test_causal_first_row_is_first_value_row():
    q, k, v = rand_qkv(1, 2, 1, 6, 40, 16, FP16, seed=61)
    o, lse = oracle.sdp_fwd(q, k, v, FP16, (1, 2, 1, 6, 40, 16), 0.5, causal=True)
    vd, qd, kd = v.double().numpy(), q.double().numpy(), k.double().numpy()
    for h in range(2):
        assert np.array_equal(o[0, h, 0], vd[0, 0, 0])
        assert abs(lse[0, h, 0] - 0.5 * math.fsum(qd[0, h, 0] * kd[0, 0, 0])) <= 1e-12


def test_causal_row_equals_full_attention_on_its_prefix():
    shape = (1, 4, 2, 12, 12, 16)
    q, k, v = rand_qkv(*shape, BF16, seed=62)
    o, lse = oracle.sdp_fwd(q, k, v, BF16, shape, 0.3, causal=True)
    for i in (0, 3, 11):
        qi = q[:, :, i:i + 1].contiguous()
        kp, vp = k[:, :, :i + 1].contiguous(), v[:, :, :i + 1].contiguous()
        o2, l2 = oracle.sdp_fwd(qi, kp, vp, BF16, (1, 4, 2, 1, i + 1, 16), 0.3)
        assert np.abs(o[:, :, i] - o2[:, :, 0]).max() <= 1e-13
        assert np.abs(lse[:, :, i] - l2[:, :, 0]).max() <= 1e-13


def test_causal_weights_vanish_past_the_diagonal():
    shape = (1, 2, 1, 8, 8, 16)
    q, k, v = rand_qkv(*shape, FP16, seed=63)
    for i in range(8):
        p, _, _ = oracle.row_probs(q, k, v, FP16, shape, 0.4, 0, 1, i, causal=True)
        assert (p[i + 1:] == 0).all() and (p[:i + 1] > 0).all()
        assert abs(p.sum() - 1.0) <= 1e-12


# -------------------------------------------------------------------- merge

@pytest.mark.parametrize("splits", [[7], [3, 4], [1, 5, 9, 2], [10, 0, 7]])
def test_merge_of_key_splits_equals_full_attention(splits):
    """Attention over disjoint key sets, merged through the log-sum-exps, is
    attention over their union (empty sets enter with LSE = -inf)."""
    Skv = sum(splits)
    shape = (1, 4, 2, 6, Skv, 16)
    q, k, v = rand_qkv(*shape, FP16, seed=81 + Skv)
    full_o, full_l = oracle.sdp_fwd(q, k, v, FP16, shape, 0.4)
    parts_o, parts_l, start = [], [], 0
    for n in splits:
        if n == 0:
            parts_o.append(np.zeros_like(full_o))
            parts_l.append(np.full(full_l.shape, -np.inf))
            continue
        ks, vs = k[:, :, start:start + n].contiguous(), v[:, :, start:start + n].contiguous()
        o_s, l_s = oracle.sdp_fwd(q, ks, vs, FP16, (1, 4, 2, 6, n, 16), 0.4)
        parts_o.append(o_s)
        parts_l.append(l_s)
        start += n
    P = len(splits)
    o, lse = oracle.sdp_merge(np.stack(parts_o).reshape(P, -1, 16), np.stack(parts_l).reshape(P, -1))
    assert np.abs(o - full_o.reshape(-1, 16)).max() <= 1e-12
    assert np.abs(lse - full_l.reshape(-1)).max() <= 1e-12


def test_merge_closed_forms():
    rng = np.random.default_rng(5)
    o1 = rng.standard_normal((1, 9, 8))
    l1 = rng.standard_normal((1, 9))
    o, lse = oracle.sdp_merge(o1, l1)  # one part: identity
    assert np.array_equal(o, o1[0]) and np.abs(lse - l1[0]).max() <= 1e-15
    parts = rng.standard_normal((4, 9, 8))
    same = np.broadcast_to(l1, (4, 9)).copy()
    o, lse = oracle.sdp_merge(parts, same)  # equal weights: the mean, LSE + ln 4
    assert np.abs(o - parts.mean(axis=0)).max() <= 1e-14
    assert np.abs(lse - (l1[0] + math.log(4))).max() <= 1e-14
    two_l = np.stack([np.zeros(9), np.full(9, math.log(3.0))])  # weights 1/4 and 3/4
    o, lse = oracle.sdp_merge(parts[:2], two_l)
    assert np.abs(o - (0.25 * parts[0] + 0.75 * parts[1])).max() <= 1e-14
    assert np.abs(lse - math.log(4.0)).max() <= 1e-14


# ------------------------------------------------------- variable length

def rand_thd(lens_q, lens_k, Hq, Hkv, D, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(sum(lens_q), Hq, D, generator=g).to(TD[dtype])
    k = torch.randn(sum(lens_k), Hkv, D, generator=g).to(TD[dtype])
    v = torch.randn(sum(lens_k), Hkv, D, generator=g).to(TD[dtype])
    cu = lambda ls: np.concatenate([[0], np.cumsum(ls)]).astype(np.int32)  # noqa: E731
    return q, k, v, cu(lens_q), cu(lens_k)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_single_sequence_equals_dense_layout(causal):
    """One sequence in (token, head, dim) layout is the dense [1, H, S, D] case transposed."""
    q, k, v, cq, ck = rand_thd([37], [53], 4, 2, 16, FP16, seed=71)
    o, lse = oracle.sdp_fwd_varlen(q, k, v, FP16, cq, ck, 0.3, causal=causal)
    qd, kd, vd = (t.permute(1, 0, 2).unsqueeze(0).contiguous() for t in (q, k, v))
    od, lsed = oracle.sdp_fwd(qd, kd, vd, FP16, (1, 4, 2, 37, 53, 16), 0.3, causal=causal)
    assert np.array_equal(o, od[0].transpose(1, 0, 2))
    assert np.array_equal(lse, lsed[0])


@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_matches_torch_float64_per_sequence(dtype, causal):
    lens_q, lens_k = [5, 1, 17, 9], [12, 3, 17, 2]
    Hq, Hkv, D = 4, 2, 16
    q, k, v, cq, ck = rand_thd(lens_q, lens_k, Hq, Hkv, D, dtype, seed=72 + causal)
    scale = 0.7 / math.sqrt(D)
    o, lse = oracle.sdp_fwd_varlen(q, k, v, dtype, cq, ck, scale, causal=causal)
    G = Hq // Hkv
    for b in range(len(lens_q)):
        qs = q[cq[b]:cq[b + 1]].double().permute(1, 0, 2)
        ks = k[ck[b]:ck[b + 1]].double().permute(1, 0, 2).repeat_interleave(G, dim=0)
        vs = v[ck[b]:ck[b + 1]].double().permute(1, 0, 2).repeat_interleave(G, dim=0)
        ref = F.scaled_dot_product_attention(qs, ks, vs, scale=scale, is_causal=causal)
        s = qs @ ks.transpose(-1, -2) * scale
        if causal:
            s = s.masked_fill(~torch.ones(lens_q[b], lens_k[b], dtype=torch.bool).tril(), float("-inf"))
        ref_lse = torch.logsumexp(s, dim=-1)
        assert np.abs(o[cq[b]:cq[b + 1]] - ref.permute(1, 0, 2).numpy()).max() <= 1e-12
        assert np.abs(lse[:, cq[b]:cq[b + 1]] - ref_lse.numpy()).max() <= 1e-12


def test_varlen_sequence_without_keys_gives_zero_and_minus_inf():
    q, k, v, cq, ck = rand_thd([3, 4, 2], [6, 0, 5], 2, 1, 8, FP16, seed=74)
    o, lse = oracle.sdp_fwd_varlen(q, k, v, FP16, cq, ck, 0.5)
    assert np.array_equal(o[3:7], np.zeros((4, 2, 8)))
    assert np.all(np.isneginf(lse[:, 3:7]))
    assert np.all(np.isfinite(lse[:, :3])) and np.all(np.isfinite(lse[:, 7:]))


def test_varlen_sequences_do_not_see_each_other():
    """Changing one sequence's keys and values leaves every other sequence's rows as they were,
    and a sequence with no query rows contributes nothing."""
    q, k, v, cq, ck = rand_thd([4, 6, 3], [5, 7, 4], 4, 1, 8, BF16, seed=75)
    o1, l1 = oracle.sdp_fwd_varlen(q, k, v, BF16, cq, ck, 0.4)
    k2, v2 = k.clone(), v.clone()
    k2[5:12] = torch.randn(7, 1, 8).to(torch.bfloat16)
    v2[5:12] = torch.randn(7, 1, 8).to(torch.bfloat16)
    o2, l2 = oracle.sdp_fwd_varlen(q, k2, v2, BF16, cq, ck, 0.4)
    keep = np.r_[0:4, 10:13]
    assert np.array_equal(o1[keep], o2[keep]) and np.array_equal(l1[:, keep], l2[:, keep])
    assert not np.array_equal(o1[4:10], o2[4:10])
    # insert an empty-query sequence with its own keys between sequences 0 and 1
    kx = torch.cat([k[:5], torch.randn(3, 1, 8).to(torch.bfloat16), k[5:]])
    vx = torch.cat([v[:5], torch.randn(3, 1, 8).to(torch.bfloat16), v[5:]])
    o3, l3 = oracle.sdp_fwd_varlen(q, kx, vx, BF16, np.array([0, 4, 4, 10, 13], np.int32),
                                   np.array([0, 5, 8, 15, 19], np.int32), 0.4)
    assert np.array_equal(o1, o3) and np.array_equal(l1, l3)


def test_varlen_rejects_bad_offsets():
    q, k, v, cq, ck = rand_thd([3, 4], [3, 4], 2, 1, 8, FP16, seed=76)
    for bad_q, bad_k in [([1, 3, 7], ck), ([0, 5, 4], ck), ([0, 3, 6], ck), (cq, [0, 3, 8])]:
        with pytest.raises(ValueError):
            oracle.sdp_fwd_varlen(q, k, v, FP16, np.array(bad_q, np.int32), np.array(bad_k, np.int32), 0.5)
