"""The persistent single-CTA kernel. Dense launches without the causal mask
that run on single CTAs (head dim 128; an odd group size whose units do not
pair; debug flag 2) with more units than SMs run one CTA per SM, each claiming
units in launch order from a per-launch counter. Checked here: every row
against the oracle (ragged tiles, MHA, odd group sizes, packed heads, head dim
256), bit-equality with the per-unit launch (debug flag 16: each unit's
arithmetic does not depend on which CTA runs it), launches in flight on two
streams at once (different claim counters), two host threads on one stream (one counter), and
graph replay (captured launches run the per-unit grid). Causal launches
keep the per-unit grid (they are covered by the parity suite)."""
import pytest
import torch

import gqa_flash_attention_gb300 as sdp
from gqa_flash_attention_gb300 import workloads
from gqa_flash_attention_gb300.workloads import Workload
from test_parity import check_full

pytestmark = pytest.mark.gpu

DEBUG_SINGLE_CTA = 2
DEBUG_NO_PERSIST = 16

CASES = [
    # 160 units of six KV tiles, the last ragged
    Workload("ps_d128_fp16", 1, 8, 2, 2560, 700, 128, "fp16", seed=301),
    # MHA, bf16: 192 units of three KV tiles, ragged query tile
    Workload("ps_d128_mha_bf16", 2, 12, 12, 1000, 300, 128, "bf16", seed=302),
    # three query heads per KV head: 168 units
    Workload("ps_d128_g3", 1, 12, 4, 1700, 900, 128, "fp16", seed=303),
    # head dim 256, three heads per KV head over 21 query tiles: units that do not pair, 189 of them
    Workload("ps_d256_g3", 1, 9, 3, 2600, 700, 256, "bf16", seed=304),
    # Sq not a multiple of 128: eight heads packed into 2400 rows per KV head, 190 units
    Workload("ps_d128_packed", 5, 16, 2, 300, 900, 128, "fp16", seed=305),
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gqa_flash_attention_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    sdp.lib()


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_persistent_single_cta_every_row(w):
    check_full(w)


def _run(w, flags=0, stream=None):
    q, k, v = (t.cuda() for t in workloads.make_inputs(w))
    old = sdp.set_debug_flags(flags)
    try:
        o, lse = sdp.sdp_fwd(q, k, v, scale=w.softmax_scale, causal=w.causal, stream=stream)
        assert sdp.poll_status() == sdp.SDP_OK
    finally:
        sdp.set_debug_flags(old)
    return o, lse


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_persistent_single_cta_matches_the_per_unit_launch_bit_for_bit(w):
    o1, l1 = _run(w)
    o2, l2 = _run(w, DEBUG_NO_PERSIST)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_forced_single_cta_at_d256_runs_persistent_and_matches_per_unit():
    """Debug flag 2 (single CTAs) on a dense D=256 launch of 160 units: the persistent single-CTA
    kernel, bit for bit the per-unit single-CTA launch."""
    w = Workload("ps_d256_forced", 1, 8, 2, 2560, 500, 256, "fp16", seed=306)
    o1, l1 = _run(w, DEBUG_SINGLE_CTA)
    o2, l2 = _run(w, DEBUG_SINGLE_CTA | DEBUG_NO_PERSIST)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_two_streams_at_once_take_different_claim_counters():
    """Two persistent launches in flight together on unordered streams must not share a counter."""
    wa, wb = CASES[0], CASES[1]
    ref_a, ref_b = _run(wa), _run(wb)
    qa, ka, va = (t.cuda() for t in workloads.make_inputs(wa))
    qb, kb, vb = (t.cuda() for t in workloads.make_inputs(wb))
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    outs = []
    torch.cuda.synchronize()
    for _ in range(4):
        with torch.cuda.stream(sa):
            oa = sdp.sdp_fwd(qa, ka, va, scale=wa.softmax_scale, causal=wa.causal)
        with torch.cuda.stream(sb):
            ob = sdp.sdp_fwd(qb, kb, vb, scale=wb.softmax_scale, causal=wb.causal)
        outs.append((oa, ob))
    torch.cuda.synchronize()
    assert sdp.poll_status() == sdp.SDP_OK
    for (o_a, l_a), (o_b, l_b) in outs:
        assert torch.equal(o_a, ref_a[0]) and torch.equal(l_a, ref_a[1])
        assert torch.equal(o_b, ref_b[0]) and torch.equal(l_b, ref_b[1])


def test_two_host_threads_on_one_stream():
    """Two host threads enqueue persistent launches on the same stream at once. They share the
    stream's claim counter, so each launch's counter reset and kernel must stay together in
    stream order."""
    import threading
    ws = CASES[0], CASES[1]
    refs = [_run(w) for w in ws]
    ins = [tuple(t.cuda() for t in workloads.make_inputs(w)) for w in ws]
    s = torch.cuda.Stream()
    outs, errs = [[], []], []
    torch.cuda.synchronize()

    def worker(i):
        try:
            q, k, v = ins[i]
            with torch.cuda.stream(s):
                for _ in range(6):
                    outs[i].append(sdp.sdp_fwd(q, k, v, scale=ws[i].softmax_scale, causal=ws[i].causal))
        except Exception as e:  # reported below, on the test's thread
            errs.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errs, errs
    assert sdp.poll_status() == sdp.SDP_OK
    for i in range(2):
        assert len(outs[i]) == 6
        for o, l in outs[i]:
            assert torch.equal(o, refs[i][0]) and torch.equal(l, refs[i][1])


def test_per_thread_default_streams_of_two_host_threads():
    """Two host threads launch on cudaStreamPerThread (handle 2): the same handle names a different
    stream in each thread, and each stream's unique id gives it its own claim counter."""
    import threading
    per_thread_stream = 2
    ws = CASES[0], CASES[1]
    refs = [_run(w) for w in ws]
    ins = [tuple(t.cuda() for t in workloads.make_inputs(w)) for w in ws]
    outs = [[(torch.empty_like(ins[i][0]), torch.empty_like(refs[i][1])) for _ in range(6)] for i in range(2)]
    errs = []
    torch.cuda.synchronize()

    def worker(i):
        try:
            q, k, v = ins[i]
            for o, l in outs[i]:
                sdp.sdp_fwd(q, k, v, scale=ws[i].softmax_scale, out=o, lse=l, stream=per_thread_stream)
        except Exception as e:  # reported below, on the test's thread
            errs.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errs, errs
    assert sdp.poll_status() == sdp.SDP_OK
    for i in range(2):
        for o, l in outs[i]:
            assert torch.equal(o, refs[i][0]) and torch.equal(l, refs[i][1])


def test_captured_launch_replays_from_a_cuda_graph():
    """A launch under stream capture takes no claim counter (a graph may be replayed on any stream,
    beside eager launches on the capturing stream) and runs the per-unit grid: bit for bit the eager
    persistent result."""
    w = CASES[1]
    q, k, v = (t.cuda() for t in workloads.make_inputs(w))
    o_eager, l_eager = sdp.sdp_fwd(q, k, v, scale=w.softmax_scale)
    o = torch.empty_like(q)
    lse = torch.empty_like(l_eager)
    sdp.sdp_fwd(q, k, v, scale=w.softmax_scale, out=o, lse=lse)  # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        sdp.sdp_fwd(q, k, v, scale=w.softmax_scale, out=o, lse=lse)
    o.zero_()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert sdp.poll_status() == sdp.SDP_OK
    assert torch.equal(o, o_eager) and torch.equal(lse, l_eager)


def test_calls_after_shutdown_set_up_again():
    """sdp_shutdown frees the status region and forgets the streams' claim counters; the next call
    allocates the region again and gives the same result."""
    w = CASES[0]
    o1, l1 = _run(w)
    torch.cuda.synchronize()
    sdp.lib().sdp_shutdown()
    o2, l2 = _run(w)
    o3, l3 = _run(w)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(o1, o3) and torch.equal(l1, l3)
