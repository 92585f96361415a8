"""The Python binding's argument checks on a GPU: every malformed call raises
ValueError before anything is launched, and a well-formed call gives the same
result with or without caller-provided output buffers, on the current stream
or on an explicit one, and from a host thread whose first CUDA work is the call."""
import math

import pytest
import torch

import gqa_flash_attention_gb300 as sdp

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gqa_flash_attention_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    sdp.lib()


def tensors(dtype=torch.float16, B=1, Hq=4, Hkv=2, Sq=200, Skv=300, D=128):
    g = torch.Generator(device="cuda").manual_seed(5)
    q = torch.randn(B, Hq, Sq, D, device="cuda", generator=g).to(dtype)
    k = torch.randn(B, Hkv, Skv, D, device="cuda", generator=g).to(dtype)
    v = torch.randn(B, Hkv, Skv, D, device="cuda", generator=g).to(dtype)
    return q, k, v


def test_malformed_calls_raise_before_any_launch():
    q, k, v = tensors()
    bad = [
        dict(q=q.float(), k=k, v=v),                                   # fp32
        dict(q=q, k=k.to(torch.bfloat16), v=v),                        # mixed dtypes
        dict(q=q.transpose(2, 3), k=k, v=v),                           # not contiguous
        dict(q=q, k=k[:, :, :, :64].contiguous(), v=v),                # head dims differ
        dict(q=q, k=k, v=v[:, :, :299].contiguous()),                  # K and V differ
        dict(q=q, k=k[:1, :1].repeat(2, 1, 1, 1), v=v[:1, :1].repeat(2, 1, 1, 1)),  # batch differs
        dict(q=q, k=k, v=v, out=torch.empty_like(q)[:, :, :100]),      # out shaped wrong
        dict(q=q, k=k, v=v, out=torch.empty_like(q).to(torch.bfloat16)),
        dict(q=q, k=k, v=v, lse=torch.empty(1, 4, 200, device="cuda", dtype=torch.float16)),
        dict(q=q, k=k, v=v, lse=torch.empty(1, 4, 199, device="cuda")),
        dict(q=q, k=k, v=v, lse=torch.empty(1, 4, 200)),               # lse on the host
        dict(q=q, k=k.cpu(), v=v),                                     # k on the host
    ]
    for kw in bad:
        with pytest.raises(ValueError):
            sdp.sdp_fwd(**kw)
    torch.cuda.synchronize()
    assert sdp.poll_status() == sdp.SDP_OK


def test_results_do_not_depend_on_buffers_or_stream():
    q, k, v = tensors()
    o1, l1 = sdp.sdp_fwd(q, k, v)
    o2 = torch.full_like(q, float("nan"))
    l2 = torch.full((1, 4, 200), float("nan"), device="cuda")
    sdp.sdp_fwd(q, k, v, out=o2, lse=l2)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        o3, l3 = sdp.sdp_fwd(q, k, v)          # the current stream inside the context
    o4, l4 = sdp.sdp_fwd(q, k, v, stream=s)    # an explicit stream object
    o5, _ = sdp.sdp_fwd(q, k, v, return_lse=False)
    torch.cuda.synchronize()
    assert sdp.poll_status() == sdp.SDP_OK
    for o, l in ((o2, l2), (o3, l3), (o4, l4)):
        assert torch.equal(o, o1) and torch.equal(l, l1)
    assert torch.equal(o5, o1)


def test_first_call_from_a_fresh_host_thread():
    """The C call is the first CUDA work of a new host thread, with output buffers whose tensor maps
    are not cached: the library binds the device's primary context itself (the runtime binds it to a
    thread only on that thread's first call that needs it)."""
    import threading
    q, k, v = tensors()
    o_ref, l_ref = sdp.sdp_fwd(q, k, v)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((1, 4, 200), float("nan"), device="cuda")
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    rc = []

    def worker():
        rc.append(sdp.sdp_fwd_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                  1, 4, 2, 200, 300, 128, 1.0 / math.sqrt(128), sdp.SDP_FP16, s.cuda_stream))

    t = threading.Thread(target=worker)
    t.start()
    t.join()
    torch.cuda.synchronize()
    assert rc == [sdp.SDP_OK]
    assert sdp.poll_status() == sdp.SDP_OK
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
