"""sdp_fwd_noalloc: the entry point for callers that cannot allocate device
memory (their memory belongs to their own pool or host application), checked
through the C ABI against sdp_fwd on the same inputs, on two calls in a row.
It takes sdp_fwd's own launch, so its outputs are bit for bit sdp_fwd's,
including where that launch packs heads (decode) or runs the persistent
kernel; its timeouts are read back with sdp_fwd_noalloc_status.

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


def _noalloc(q, k, v, w, with_lse=True):
    o = torch.full_like(q, float("nan"))
    lse = torch.full((w.B, w.Hq, w.Sq), float("nan"), dtype=torch.float32, device=q.device) if with_lse else None
    rc = sdp.sdp_fwd_noalloc_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                 lse.data_ptr() if with_lse else 0,
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
    # same launch as sdp_fwd: bit for bit
    for (o, lse), (o_ref, l_ref) in zip(outs, refs):
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
    assert sdp.noalloc_status() == sdp.SDP_OK


@pytest.mark.parametrize("w", [
    # 160 units of a dense D=256 launch: sdp_fwd runs the persistent CTA-pair kernel here
    Workload("noalloc_persistent", 1, 8, 2, 2560, 384, 256, "fp16", seed=53),
    # 160 units of a dense D=128 launch: the persistent single-CTA kernel and its claim counter
    Workload("noalloc_persist_single", 1, 8, 2, 2560, 384, 128, "fp16", seed=56),
    # decode: one query row, 16 heads per KV head, packed into one 16-row tile
    Workload("noalloc_decode", 1, 16, 1, 1, 1000, 256, "fp16", seed=54),
    Workload("noalloc_decode_bf16", 2, 8, 2, 3, 777, 128, "bf16", seed=55),
], ids=lambda w: w.name)
def test_same_launch_as_sdp_fwd_bit_for_bit(w):
    q, k, v = _inputs(w)
    o_ref, l_ref = sdp.sdp_fwd(q, k, v, scale=w.softmax_scale)
    o, lse = _noalloc(q, k, v, w)
    o_nl, _ = _noalloc(q, k, v, w, with_lse=False)  # LSE is optional, as for sdp_fwd
    torch.cuda.synchronize()
    assert sdp.noalloc_status() == sdp.SDP_OK
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
    assert torch.equal(o_nl, o_ref)


def test_timeout_is_read_back_and_the_next_call_is_right():
    # Debug flag 1: the load warp issues no copies, so every wait runs out after the 50 ms
    # limit (a bounded wait on a barrier nothing completes; no fault). The timeout lands in
    # this entry point's own status word, which sdp_fwd_noalloc_status reads and clears.
    w = CASES[0]
    q, k, v = _inputs(w)
    assert sdp.noalloc_status() == sdp.SDP_OK
    assert sdp.poll_status() == sdp.SDP_OK
    old_ms = sdp.set_wait_timeout_ms(50)
    old_flags = sdp.set_debug_flags(1)
    try:
        _noalloc(q, k, v, w)
        assert sdp.noalloc_status() == sdp.SDP_ERR_DEVICE_TIMEOUT
        assert 1 <= (sdp.last_status_detail() & 0xFF) <= 6, hex(sdp.last_status_detail())
    finally:
        sdp.set_debug_flags(old_flags)
        sdp.set_wait_timeout_ms(old_ms)
    assert sdp.noalloc_status() == sdp.SDP_OK  # cleared
    assert sdp.poll_status() == sdp.SDP_OK     # sdp_fwd's word was not touched
    o_ref, l_ref = sdp.sdp_fwd(q, k, v, scale=w.softmax_scale)
    o, lse = _noalloc(q, k, v, w)
    assert sdp.noalloc_status() == sdp.SDP_OK
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


def test_rejects_bad_arguments_without_launching():
    q = torch.zeros(1, 4, 8, 128, dtype=torch.float16, device="cuda")
    args = dict(q=q.data_ptr(), k=q.data_ptr(), v=q.data_ptr(), o=q.data_ptr() + 4096, lse=0, B=1, Hq=4, Hkv=1,
                Sq=8, Skv=8, D=64, scale=1 / math.sqrt(128), dtype=sdp.SDP_FP16)
    assert sdp.sdp_fwd_noalloc_ptr(**args) == sdp.SDP_ERR_UNSUPPORTED
    args.update(D=128, Hq=6, Hkv=4)
    assert sdp.sdp_fwd_noalloc_ptr(**args) == sdp.SDP_ERR_INVALID_ARG
