"""The C ABI without a GPU: the library loads, exports every symbol that
include/sdp.h declares, and rejects bad arguments before any CUDA call."""
import math
import os
import re

import pytest

import gqa_flash_attention_gb300 as sdp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sdp.h")


@pytest.fixture(scope="module")
def L():
    from gqa_flash_attention_gb300 import build
    build.build()
    return sdp.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sdp_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("sdp_fwd", "sdp_poll_status", "sdp_strerror", "sdp_version"):
        assert required in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name


def test_version_and_messages(L):
    assert L.sdp_version() == 107
    for code in range(-7, 1):
        assert len(sdp.strerror(code)) > 0
    assert sdp.strerror(-99) == "unknown status code"


def test_setters_round_trip(L):
    old = sdp.set_wait_timeout_ms(123)
    assert sdp.set_wait_timeout_ms(old) == 123
    assert sdp.set_debug_flags(0) == 0


A = 0x10000  # 16-byte aligned stand-in addresses: never dereferenced, validation returns first


def call(**kw):
    args = dict(q=A, k=2 * A, v=3 * A, o=4 * A, lse=5 * A, B=1, Hq=4, Hkv=1, Sq=256, Skv=256, D=128,
                scale=0.088, dtype=sdp.SDP_FP16)
    args.update(kw)
    return sdp.sdp_fwd_ptr(**args)


DENSE_BAD = [
    (dict(D=64), sdp.SDP_ERR_UNSUPPORTED),
    (dict(D=192), sdp.SDP_ERR_UNSUPPORTED),
    (dict(dtype=2), sdp.SDP_ERR_UNSUPPORTED),
    (dict(q=0), sdp.SDP_ERR_INVALID_ARG),
    (dict(k=0), sdp.SDP_ERR_INVALID_ARG),
    (dict(v=0), sdp.SDP_ERR_INVALID_ARG),
    (dict(o=0), sdp.SDP_ERR_INVALID_ARG),
    (dict(B=0), sdp.SDP_ERR_INVALID_ARG),
    (dict(Hq=-1), sdp.SDP_ERR_INVALID_ARG),
    (dict(Sq=0), sdp.SDP_ERR_INVALID_ARG),
    (dict(Skv=0), sdp.SDP_ERR_INVALID_ARG),
    (dict(Hq=6, Hkv=4), sdp.SDP_ERR_INVALID_ARG),
    (dict(scale=math.inf), sdp.SDP_ERR_INVALID_ARG),
    (dict(scale=math.nan), sdp.SDP_ERR_INVALID_ARG),
    (dict(o=A), sdp.SDP_ERR_INVALID_ARG),
    (dict(q=A + 8), sdp.SDP_ERR_ALIGNMENT),
    (dict(v=3 * A + 2), sdp.SDP_ERR_ALIGNMENT),
    (dict(lse=5 * A + 2), sdp.SDP_ERR_ALIGNMENT),
    (dict(B=1 << 16, Hq=1 << 16, Hkv=1), sdp.SDP_ERR_OVERFLOW),
    (dict(B=1 << 10, Hq=1 << 12, Hkv=1, Sq=1 << 20), sdp.SDP_ERR_OVERFLOW),
]


@pytest.mark.parametrize("kw,code", DENSE_BAD)
def test_validation_errors_launch_nothing(L, kw, code):
    assert call(**kw) == code


@pytest.mark.parametrize("kw,code", DENSE_BAD)
def test_noalloc_validates_like_sdp_fwd(L, kw, code):
    # the allocation-free entry point runs sdp_fwd's own checks, before any CUDA call
    args = dict(q=A, k=2 * A, v=3 * A, o=4 * A, lse=5 * A, B=1, Hq=4, Hkv=1, Sq=256, Skv=256, D=128,
                scale=0.088, dtype=sdp.SDP_FP16)
    args.update(kw)
    assert sdp.sdp_fwd_noalloc_ptr(**args) == code


def test_python_binding_rejects_bad_tensors():
    import torch
    q = torch.zeros(1, 4, 8, 128, dtype=torch.float16)
    with pytest.raises(ValueError):
        sdp.sdp_fwd(q, q, q)  # CPU tensors
    with pytest.raises(ValueError):
        sdp.sdp_fwd(q[0], q, q)  # not 4-D


def split_call(**kw):
    args = dict(q=A, k=2 * A, v=3 * A, o=4 * A, lse=5 * A, B=1, Hq=4, Hkv=1, Sq=1, Skv=1000, D=128,
                scale=0.088, dtype=sdp.SDP_FP16, n_splits=0, workspace=6 * A, workspace_bytes=1 << 20)
    args.update(kw)
    return sdp.sdp_fwd_splitkv_ptr(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(D=64), sdp.SDP_ERR_UNSUPPORTED),
    (dict(dtype=2), sdp.SDP_ERR_UNSUPPORTED),
    (dict(q=0), sdp.SDP_ERR_INVALID_ARG),
    (dict(Hq=6, Hkv=4), sdp.SDP_ERR_INVALID_ARG),
    (dict(Skv=0), sdp.SDP_ERR_INVALID_ARG),
    (dict(scale=math.nan), sdp.SDP_ERR_INVALID_ARG),
    (dict(o=A), sdp.SDP_ERR_INVALID_ARG),
    (dict(n_splits=-1), sdp.SDP_ERR_INVALID_ARG),
    (dict(k=2 * A + 4), sdp.SDP_ERR_ALIGNMENT),
])
def test_split_kv_validation_errors_launch_nothing(L, kw, code):
    assert split_call(**kw) == code


@pytest.mark.parametrize("args,code", [
    ((1, 4, 1, 1, 1000, 64, 0, 0), sdp.SDP_ERR_UNSUPPORTED),
    ((1, 4, 1, 1, 1000, 128, 5, 0), sdp.SDP_ERR_UNSUPPORTED),
    ((0, 4, 1, 1, 1000, 128, 0, 0), sdp.SDP_ERR_INVALID_ARG),
    ((1, 6, 4, 1, 1000, 128, 0, 0), sdp.SDP_ERR_INVALID_ARG),
    ((1, 4, 1, 1, 1000, 128, 0, -2), sdp.SDP_ERR_INVALID_ARG),
])
def test_split_kv_planning_rejects_bad_sizes(L, args, code):
    assert L.sdp_fwd_splitkv_count(*args) == code
    assert L.sdp_fwd_splitkv_workspace_bytes(*args) == code


def varlen_call(**kw):
    args = dict(q=A, k=2 * A, v=3 * A, o=4 * A, lse=5 * A, cu_q=6 * A, cu_k=7 * A, nseq=2, Hq=4, Hkv=2,
                total_q=300, total_k=300, max_seqlen_q=200, D=128, scale=0.088, dtype=sdp.SDP_FP16)
    args.update(kw)
    return sdp.sdp_fwd_varlen_ptr(**args)


@pytest.mark.parametrize("kw,code", [
    (dict(D=64), sdp.SDP_ERR_UNSUPPORTED),
    (dict(dtype=2), sdp.SDP_ERR_UNSUPPORTED),
    (dict(cu_q=0), sdp.SDP_ERR_INVALID_ARG),
    (dict(cu_k=0), sdp.SDP_ERR_INVALID_ARG),
    (dict(max_seqlen_q=0), sdp.SDP_ERR_INVALID_ARG),
    (dict(nseq=0), sdp.SDP_ERR_INVALID_ARG),
    (dict(Hq=6, Hkv=4), sdp.SDP_ERR_INVALID_ARG),
    (dict(total_k=-1), sdp.SDP_ERR_INVALID_ARG),
    (dict(max_seqlen_q=-1), sdp.SDP_ERR_INVALID_ARG),
    (dict(o=2 * A), sdp.SDP_ERR_INVALID_ARG),
    (dict(scale=math.inf), sdp.SDP_ERR_INVALID_ARG),
    (dict(cu_q=6 * A + 2), sdp.SDP_ERR_ALIGNMENT),
    (dict(q=A + 4), sdp.SDP_ERR_ALIGNMENT),
    (dict(total_q=0), sdp.SDP_OK),
    (dict(total_q=0, q=0, o=0), sdp.SDP_OK),
    (dict(nseq=1 << 20, Hq=1 << 12, Hkv=1, max_seqlen_q=1 << 10), sdp.SDP_ERR_OVERFLOW),
])
def test_varlen_validation_errors_launch_nothing(L, kw, code):
    assert varlen_call(**kw) == code
