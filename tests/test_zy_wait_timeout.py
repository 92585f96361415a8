"""Failure detection without a GPU fault: every mbarrier wait in the kernels
is bounded. With the load warp told to issue no copies (debug flag 1),
nothing ever completes the waits of the MMA issuers and the softmax warps;
each gives up after the configured limit, records a site code in the status
word, and the kernel drains, frees tensor memory and returns. The host reads
SDP_ERR_DEVICE_TIMEOUT from sdp_poll_status, and the context stays usable:
the next call computes the right result."""
import pytest
import torch

import gqa_flash_attention_gb300 as sdp
import oracle
from gqa_flash_attention_gb300 import workloads
from gqa_flash_attention_gb300.workloads import Workload
from parity import ORACLE_DTYPE, assert_within, compare

pytestmark = pytest.mark.gpu

DEBUG_NO_LOADS = 1
DEBUG_SINGLE_CTA = 2


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gqa_flash_attention_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    sdp.lib()


@pytest.mark.parametrize("flags,w", [
    (DEBUG_NO_LOADS, Workload("timeout", 1, 4, 2, 256, 384, 128, "fp16", seed=91)),  # two heads per group: CTA pairs
    (DEBUG_NO_LOADS | DEBUG_SINGLE_CTA, Workload("timeout", 1, 4, 2, 256, 384, 128, "fp16", seed=91)),
    # 160 units of a dense D=256 launch: the persistent CTA-pair kernel
    (DEBUG_NO_LOADS, Workload("timeout_persist", 1, 8, 2, 2560, 384, 256, "fp16", seed=92)),
    # the two-tile CTA-pair kernel at D=128 (debug flag 128 forces it below one wave)
    (DEBUG_NO_LOADS | 128, Workload("timeout_pair2", 1, 4, 2, 256, 384, 128, "bf16", seed=93)),
    # 160 causal units of a dense D=256 launch: the persistent CTA-pair kernel's causal walk
    (DEBUG_NO_LOADS, Workload("timeout_persist_causal", 1, 8, 2, 2560, 2560, 256, "fp16", seed=94, causal=True)),
    # 160 units of a dense D=128 launch: the persistent single-CTA kernel (no unit is ever announced)
    (DEBUG_NO_LOADS, Workload("timeout_persist_single", 1, 8, 2, 2560, 384, 128, "fp16", seed=97)),
], ids=["cta_pair", "single_cta", "persistent_pair", "two_tile_pair", "persistent_causal", "persistent_single"])
def test_wait_timeout_is_reported_and_the_context_survives(flags, w):
    q, k, v = (t.cuda() for t in workloads.make_inputs(w))
    assert sdp.poll_status() == sdp.SDP_OK
    old_ms = sdp.set_wait_timeout_ms(50)
    old_flags = sdp.set_debug_flags(flags)
    try:
        sdp.sdp_fwd(q, k, v, scale=w.softmax_scale, causal=w.causal)
        assert sdp.poll_status() == sdp.SDP_ERR_DEVICE_TIMEOUT
        site = sdp.last_status_detail() & 0xFF
        assert 1 <= site <= 6, hex(sdp.last_status_detail())
    finally:
        sdp.set_debug_flags(old_flags)
        sdp.set_wait_timeout_ms(old_ms)
    # the status word was cleared and the device still computes correctly
    assert sdp.poll_status() == sdp.SDP_OK
    o, lse = sdp.sdp_fwd(q, k, v, scale=w.softmax_scale, causal=w.causal)
    assert sdp.poll_status() == sdp.SDP_OK
    ref_o, ref_l = oracle.sdp_fwd(q.cpu(), k.cpu(), v.cpu(), ORACLE_DTYPE[w.dtype], w.shape, w.softmax_scale,
                                  causal=w.causal)
    assert_within(compare(o, lse, ref_o, ref_l, w.dtype), w.dtype)


def test_varlen_persistent_wait_timeout_is_reported():
    """The persistent CTA-pair kernel on a causal variable-length batch (16 heads over 4 KV heads at
    D=256, 304 units): every wait runs out, the status says so, and the next call is right."""
    from gqa_flash_attention_gb300.workloads import VarlenWorkload
    w = VarlenWorkload("timeout_varlen", (1000, 1200), (1000, 1200), 16, 4, 256, "fp16", seed=95, causal=True)
    q, k, v = (t.cuda() for t in workloads.make_varlen_inputs(w))
    cq, ck = torch.from_numpy(w.cu_q).cuda(), torch.from_numpy(w.cu_k).cuda()
    assert sdp.poll_status() == sdp.SDP_OK
    old_ms = sdp.set_wait_timeout_ms(50)
    old_flags = sdp.set_debug_flags(DEBUG_NO_LOADS)
    try:
        sdp.sdp_fwd_varlen(q, k, v, cq, ck, w.max_q, scale=w.softmax_scale, causal=True)
        assert sdp.poll_status() == sdp.SDP_ERR_DEVICE_TIMEOUT
    finally:
        sdp.set_debug_flags(old_flags)
        sdp.set_wait_timeout_ms(old_ms)
    o, lse = sdp.sdp_fwd_varlen(q, k, v, cq, ck, w.max_q, scale=w.softmax_scale, causal=True)
    assert sdp.poll_status() == sdp.SDP_OK
    ref_o, ref_l = oracle.sdp_fwd_varlen(q.cpu(), k.cpu(), v.cpu(), ORACLE_DTYPE[w.dtype], w.cu_q, w.cu_k,
                                         w.softmax_scale, causal=True)
    assert_within(compare(o, lse, ref_o, ref_l, w.dtype), w.dtype)
