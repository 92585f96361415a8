"""sdp_fwd_noalloc: the entry point for callers that cannot allocate device
memory (their memory belongs to their own pool or host application), checked
through the C ABI against sdp_fwd on the same inputs, on two calls in a row.

This file is collected last on purpose, so that a run stopping at the first
failure has run every other test first. It also passes on its own in a fresh
process, where its first call performs the per-device set-up.
"""
import math

import pytest
import torch

import gqa_flash_attention_gb300 as sdp
from gqa_flash_attention_gb300 import workloads
from gqa_flash_attention_gb300.workloads import Workload
from parity import assert_within, compare

pytestmark = pytest.mark.gpu

CODE = {"fp16": sdp.SDP_FP16, "bf16": sdp.SDP_BF16}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gqa_flash_attention_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    sdp.lib()


def _inputs(w):
    q, k, v = (t.cuda() for t in workloads.make_inputs(w))
    return q, k, v


def _noalloc(q, k, v, w):
    o = torch.full_like(q, float("nan"))
    lse = torch.full((w.B, w.Hq, w.Sq), float("nan"), dtype=torch.float32, device=q.device)
    rc = sdp.sdp_fwd_noalloc_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                 w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, w.softmax_scale, CODE[w.dtype],
                                 torch.cuda.current_stream().cuda_stream)
    assert rc == sdp.SDP_OK, sdp.strerror(rc)
    return o, lse


CASES = [
    Workload("noalloc_d256_fp16", 1, 8, 2, 300, 700, 256, "fp16", seed=51),
    Workload("noalloc_d128_bf16", 2, 4, 1, 129, 1000, 128, "bf16", seed=52),
]


def test_two_calls_in_a_row_match_sdp_fwd():
    inputs = [_inputs(w) for w in CASES]
    refs = []
    for w, (q, k, v) in zip(CASES, inputs):
        o_ref, l_ref = sdp.sdp_fwd(q, k, v, scale=w.softmax_scale)
        refs.append((o_ref, l_ref))
    torch.cuda.synchronize()
    # two calls in a row, back to back on one stream, different problems
    outs = [_noalloc(q, k, v, w) for w, (q, k, v) in zip(CASES, inputs)]
    torch.cuda.synchronize()
    for w, (o, lse), (o_ref, l_ref) in zip(CASES, outs, refs):
        st = compare(o, lse, o_ref.double().cpu().numpy(), l_ref.double().cpu().numpy(), w.dtype)
        assert_within(st, w.dtype)
    # and the same problem twice: the shared scratch from the first call does not leak into the second
    w = CASES[0]
    q, k, v = inputs[0]
    o1, l1 = _noalloc(q, k, v, w)
    o2, l2 = _noalloc(q, k, v, w)
    torch.cuda.synchronize()
    for o, lse in ((o1, l1), (o2, l2)):
        st = compare(o, lse, refs[0][0].double().cpu().numpy(), refs[0][1].double().cpu().numpy(), w.dtype)
        assert_within(st, w.dtype)


def test_rejects_bad_arguments_without_launching():
    q = torch.zeros(1, 4, 8, 128, dtype=torch.float16, device="cuda")
    args = dict(q=q.data_ptr(), k=q.data_ptr(), v=q.data_ptr(), o=q.data_ptr() + 4096, lse=0, B=1, Hq=4, Hkv=1,
                Sq=8, Skv=8, D=64, scale=1 / math.sqrt(128), dtype=sdp.SDP_FP16)
    assert sdp.sdp_fwd_noalloc_ptr(**args) == sdp.SDP_ERR_UNSUPPORTED
    args.update(D=128, Hq=6, Hkv=4)
    assert sdp.sdp_fwd_noalloc_ptr(**args) == sdp.SDP_ERR_INVALID_ARG
