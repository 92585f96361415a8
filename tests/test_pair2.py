"""The two-tile CTA-pair kernel at head dim 128 (two 128-row query tiles per CTA,
64-key softmax steps) against the fp64 oracle, through the C ABI.

Debug flag 128 selects it (for dense, non-causal D=128 launches whose units
pair up); the cases here span one to many 64-key
steps, a last step of 1 to 64 keys, a second query tile that is partly or
wholly past the last row, and both dtypes.
"""
import numpy as np
import pytest
import torch

import gqa_flash_attention_gb300 as sdp
import oracle
from gqa_flash_attention_gb300 import workloads
from gqa_flash_attention_gb300.workloads import Workload
from parity import ORACLE_DTYPE, assert_within, compare
from test_parity import check_full, gpu_run, test_full_size_workload_sampled_rows

pytestmark = pytest.mark.gpu

FORCE_PAIR2 = 128
NO_PAIR2 = 64


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gqa_flash_attention_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    sdp.lib()


class flags:
    def __init__(self, f):
        self.f = f

    def __enter__(self):
        self.old = sdp.set_debug_flags(self.f)

    def __exit__(self, *a):
        sdp.set_debug_flags(self.old)


def pairs_up(B, Hq, Hkv, Sq, Skv):
    """The launch rule for this kernel's clusters, after the head packing that sdp_fwd applies
    when Sq is not a multiple of 128: two-tile units of one (batch, KV head) come in even number."""
    G = Hq // Hkv
    if G > 1 and Sq % 128:
        Sq, G = G * Sq, 1
    n_qpairs = ((Sq + 127) // 128 + 1) // 2
    return (n_qpairs * G) % 2 == 0


# (B, Hq, Hkv, Sq, Skv)
SHAPES = [
    (1, 2, 1, 256, 256),    # two whole tiles, four steps
    (1, 2, 1, 128, 64),     # one step; tile B wholly past the last row
    (1, 2, 2, 300, 65),     # two steps, the last of one key; rows 256-299 in a tile A, its tile B empty
    (1, 4, 2, 130, 129),    # packed heads (260 rows); three steps, the last of one key
    (1, 2, 2, 384, 200),    # MHA: a cluster takes two tile pairs of one head
    (2, 8, 2, 1000, 777),   # packed heads; 13 steps, the last of 9 keys
    (1, 2, 1, 512, 192),    # three steps, an odd count ending on a whole step
    (1, 4, 1, 256, 1),      # a single key
    (1, 2, 1, 200, 2048),   # packed heads; 32 steps: the K/V ring wraps several times
]
assert all(pairs_up(*s) for s in SHAPES)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_every_row(shape, dtype):
    B, Hq, Hkv, Sq, Skv = shape
    with flags(FORCE_PAIR2):
        check_full(Workload("pair2", B, Hq, Hkv, Sq, Skv, 128, dtype, seed=61 + Sq + Skv))


@pytest.mark.parametrize("scale", [0.0, -0.0884])
def test_scale_zero_and_negative(scale):
    with flags(FORCE_PAIR2):
        check_full(Workload("pair2_scale", 1, 4, 2, 256, 300, 128, "bf16", seed=62, scale=scale))


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_peaky_keys(dtype):
    """1 % of the key rows scaled by 8: a row's maximum jumps in a later step, so O is rescaled
    (after P is stored, before it is handed over)."""
    with flags(FORCE_PAIR2):
        check_full(Workload(f"pair2_peaky_{dtype}", 1, 8, 2, 512, 3000, 128, dtype, seed=63, peaky_k=True))


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_large_scores_saturate_cleanly(dtype):
    w = Workload(f"pair2_large_{dtype}", 1, 4, 2, 256, 700, 128, dtype, seed=64)
    q, k, v = workloads.make_inputs(w)
    q, k = (q.float() * 24).to(q.dtype), (k.float() * 24).to(k.dtype)
    with flags(FORCE_PAIR2):
        o, lse = gpu_run(q, k, v, w.softmax_scale)
    ref_o, ref_l = oracle.sdp_fwd(q, k, v, ORACLE_DTYPE[dtype], w.shape, w.softmax_scale)
    st = compare(o, lse, ref_o, ref_l, dtype)
    assert st["nan_o"] == 0 and st["nan_lse"] == 0
    assert st["max_abs"] <= (2e-2 if dtype == "fp16" else 4e-2), st
    assert st["lse_max_abs"] <= 1e-6 * max(1.0, float(np.abs(ref_l).max())) * 8, st


@pytest.mark.parametrize("splits", [2, 5])
def test_split_kv(splits):
    """Partial results per KV split (the split index outermost in the grid), merged by sdp_merge."""
    w = Workload("pair2_split", 1, 4, 2, 256, 1500, 128, "fp16", seed=65)
    q, k, v = workloads.make_inputs(w)
    with flags(FORCE_PAIR2):
        o, lse = sdp.sdp_fwd(q.cuda(), k.cuda(), v.cuda(), scale=w.softmax_scale, kv_splits=splits)
        assert sdp.poll_status() == sdp.SDP_OK
    ref_o, ref_l = oracle.sdp_fwd(q, k, v, oracle.FP16, w.shape, w.softmax_scale)
    assert_within(compare(o, lse, ref_o, ref_l, "fp16"), "fp16")


def test_deterministic():
    w = Workload("pair2_det", 1, 8, 2, 768, 900, 128, "bf16", seed=66)
    q, k, v = (t.cuda() for t in workloads.make_inputs(w))
    with flags(FORCE_PAIR2):
        o1, l1 = sdp.sdp_fwd(q, k, v)
        o2, l2 = sdp.sdp_fwd(q, k, v)
        assert sdp.poll_status() == sdp.SDP_OK
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("name", ["gqa4_b2_s8k_d128_bf16_peaky", "mha_b4_s16k_d128_fp16"])
def test_full_size_sampled(name):
    """The D=128 workloads at full size on this kernel, on sampled rows."""
    with flags(FORCE_PAIR2):
        test_full_size_workload_sampled_rows(name)
