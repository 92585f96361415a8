"""sdp_merge on the GPU: the merge of partial results over disjoint key sets
(the ring / context-parallel state exchange, "SyclKittens" summary section
I.2), against the oracle merge on the same inputs, and end to end: attention
over key shards with sdp_fwd, merged with sdp_merge, against the oracle's
attention over all keys."""
import numpy as np
import pytest
import torch

import gqa_flash_attention_gb300 as sdp
import oracle
from gqa_flash_attention_gb300 import workloads
from gqa_flash_attention_gb300.workloads import Workload
from parity import ORACLE_DTYPE, assert_within, compare

pytestmark = pytest.mark.gpu
TD = {"fp16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gqa_flash_attention_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    sdp.lib()


def random_parts(P, rows, D, dtype, seed, neg_inf_part=None):
    g = torch.Generator().manual_seed(seed)
    o = torch.randn(P, rows, D, generator=g).to(TD[dtype])
    lse = (torch.randn(P, rows, generator=g) * 3.0).float()
    if neg_inf_part is not None:
        lse[neg_inf_part] = float("-inf")
    return o, lse


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
# part counts on both sides of each all-in-flight bound of the merge kernels (8, 16, 32; more: batches of 8)
@pytest.mark.parametrize("P,rows", [(2, 1000), (5, 37), (8, 45), (9, 61), (16, 77), (17, 50), (32, 40), (33, 29),
                                    (37, 131), (1, 64)])
def test_merge_matches_oracle(D, dtype, P, rows):
    o_parts, lse_parts = random_parts(P, rows, D, dtype, seed=P * 1000 + rows)
    o, lse = sdp.sdp_merge(o_parts.cuda(), lse_parts.cuda())
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.sdp_merge(o_parts, lse_parts)
    st = compare(o, lse, ref_o, ref_l, dtype)
    assert_within(st, dtype)
    if P == 1:  # one part: the row itself, bit for bit
        assert torch.equal(o.cpu(), o_parts[0]) and torch.equal(lse.cpu(), lse_parts[0])


def test_merge_ignores_parts_without_keys():
    o_parts, lse_parts = random_parts(4, 300, 128, "fp16", seed=9, neg_inf_part=2)
    o, lse = sdp.sdp_merge(o_parts.cuda(), lse_parts.cuda())
    keep = [0, 1, 3]
    o2, l2 = sdp.sdp_merge(o_parts[keep].contiguous().cuda(), lse_parts[keep].contiguous().cuda())
    torch.cuda.synchronize()
    # same terms, summed in another lane order: equal up to the last bits
    assert torch.allclose(lse, l2, rtol=0, atol=1e-5)
    assert torch.allclose(o.float(), o2.float(), rtol=0, atol=2e-3)


def test_merge_rejects_bad_arguments():
    o_parts, lse_parts = random_parts(2, 8, 64, "fp16", seed=1)
    with pytest.raises(sdp.SdpError):
        sdp.sdp_merge(o_parts.cuda(), lse_parts.cuda())  # D = 64 unsupported


@pytest.mark.parametrize("w,splits", [
    (Workload("cp_d256_fp16", 1, 8, 2, 300, 700, 256, "fp16", seed=91), [128, 300, 272]),
    (Workload("cp_d128_bf16", 2, 4, 1, 129, 500, 128, "bf16", seed=92), [100, 1, 399]),
])
def test_context_parallel_shards_then_merge(w, splits):
    """Three key shards attended separately (as three ring steps would), then merged."""
    q, k, v = workloads.make_inputs(w)
    qd = q.cuda()
    parts_o, parts_l, start = [], [], 0
    for n in splits:
        ks = k[:, :, start:start + n].contiguous().cuda()
        vs = v[:, :, start:start + n].contiguous().cuda()
        o_s, l_s = sdp.sdp_fwd(qd, ks, vs, scale=w.softmax_scale)
        parts_o.append(o_s)
        parts_l.append(l_s)
        start += n
    assert start == w.Skv
    o, lse = sdp.sdp_merge(torch.stack(parts_o), torch.stack(parts_l))
    torch.cuda.synchronize()
    assert sdp.poll_status() == sdp.SDP_OK
    ref_o, ref_l = oracle.sdp_fwd(q, k, v, ORACLE_DTYPE[w.dtype], w.shape, w.softmax_scale)
    st = compare(o, lse, ref_o, ref_l, w.dtype)
    assert_within(st, w.dtype)
