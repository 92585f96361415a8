"""GB300-native fused grouped-query attention forward.

``sdp_fwd(q, k, v)`` computes O = softmax(Q K^T * scale) V and the natural
log-sum-exp of every score row for query heads that share KV heads in
groups of Hq / Hkv. The work runs in ``libsdp.so`` (hand-written CUDA for
sm_103a: TMA, mbarriers, tcgen05 MMAs with TMEM accumulators); this module
only checks and marshals arguments through the C ABI of ``include/sdp.h``.
PyTorch supplies device memory and streams. There is no fallback: if the
library is missing or the device is not sm_103, calls raise.
"""
from __future__ import annotations

import contextlib
import ctypes
import math
import os

import torch

__all__ = ["sdp_fwd", "sdp_fwd_ptr", "poll_status", "SdpError", "lib", "LIB_PATH", "SDP_FP16", "SDP_BF16",
           "set_wait_timeout_ms", "set_debug_flags", "last_status_detail", "strerror"]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libsdp.so")

SDP_FP16 = 0
SDP_BF16 = 1
SDP_OK = 0
SDP_ERR_INVALID_ARG = -1
SDP_ERR_UNSUPPORTED = -2
SDP_ERR_ALIGNMENT = -3
SDP_ERR_OVERFLOW = -4
SDP_ERR_CUDA = -5
SDP_ERR_DEVICE_TIMEOUT = -6
SDP_ERR_BAD_SEQLENS = -7

_DTYPE_CODE = {torch.float16: SDP_FP16, torch.bfloat16: SDP_BF16}

_lib = None


class SdpError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"sdp error {code}: {msg}")
        self.code = code


def lib() -> ctypes.CDLL:
    """The loaded libsdp.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run `python -m gqa_flash_attention_gb300.build` "
                               "(the CUDA library is required; there is no fallback path)")
        L = ctypes.CDLL(LIB_PATH)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        L.sdp_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
        L.sdp_fwd.restype = i
        L.sdp_fwd_causal.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
        L.sdp_fwd_causal.restype = i
        L.sdp_merge.argtypes = [vp, vp, i, ctypes.c_longlong, i, i, vp, vp, vp]
        L.sdp_merge.restype = i
        L.sdp_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, i, vp]
        L.sdp_fwd_varlen.restype = i
        L.sdp_fwd_splitkv_count.argtypes = [i, i, i, i, i, i, i, i]
        L.sdp_fwd_splitkv_count.restype = i
        L.sdp_fwd_splitkv_workspace_bytes.argtypes = [i, i, i, i, i, i, i, i]
        L.sdp_fwd_splitkv_workspace_bytes.restype = ctypes.c_longlong
        L.sdp_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, vp, ctypes.c_ulonglong, vp]
        L.sdp_fwd_splitkv.restype = i
        L.sdp_poll_status.argtypes = [vp]
        L.sdp_poll_status.restype = i
        L.sdp_last_status_detail.argtypes = []
        L.sdp_last_status_detail.restype = ctypes.c_uint
        L.sdp_set_wait_timeout_ms.argtypes = [ctypes.c_uint]
        L.sdp_set_wait_timeout_ms.restype = ctypes.c_uint
        L.sdp_set_debug_flags.argtypes = [i]
        L.sdp_set_debug_flags.restype = i
        L.sdp_last_cuda_error.argtypes = []
        L.sdp_last_cuda_error.restype = i
        L.sdp_strerror.argtypes = [i]
        L.sdp_strerror.restype = ctypes.c_char_p
        L.sdp_version.argtypes = []
        L.sdp_version.restype = i
        L.sdp_shutdown.argtypes = []
        L.sdp_shutdown.restype = None
        _lib = L
    return _lib


def strerror(code: int) -> str:
    return lib().sdp_strerror(int(code)).decode()


def _check(rc: int) -> None:
    if rc != SDP_OK:
        msg = strerror(rc)
        if rc == SDP_ERR_CUDA:
            msg += f" (cudaError {lib().sdp_last_cuda_error()})"
        raise SdpError(rc, msg)


def _index(device) -> int:
    """A CUDA device's index (a torch.device, or an int already)."""
    if isinstance(device, int):
        return device
    return torch.cuda.current_device() if device.index is None else device.index


def _on(device):
    """The device context of a call: none when `device` is already current (entering
    torch.cuda.device costs microseconds per call)."""
    idx = _index(device)
    if idx == torch.cuda.current_device():
        return contextlib.nullcontext()
    return torch.cuda.device(idx)


# The current stream's handle without building a torch.cuda.Stream object (which costs
# microseconds per call); the public route where this build of torch lacks the query.
_raw_current_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(stream, device) -> int:
    if stream is None:
        idx = _index(device)
        if _raw_current_stream is not None:
            return int(_raw_current_stream(idx))
        return torch.cuda.current_stream(idx).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def sdp_fwd_ptr(q: int, k: int, v: int, o: int, lse: int, B: int, Hq: int, Hkv: int, Sq: int, Skv: int, D: int,
                scale: float, dtype: int, stream: int = 0, causal: bool = False) -> int:
    """The raw C call (sdp_fwd, or sdp_fwd_causal) with integer addresses; returns the status code.
    (The argument types are declared on the function, so ctypes converts plain ints and floats.)"""
    L = _lib if _lib is not None else lib()
    fn = L.sdp_fwd_causal if causal else L.sdp_fwd
    return fn(q, k, v, o, lse, B, Hq, Hkv, Sq, Skv, D, scale, dtype, stream)


def sdp_fwd_splitkv_ptr(q: int, k: int, v: int, o: int, lse: int, B: int, Hq: int, Hkv: int, Sq: int, Skv: int,
                        D: int, scale: float, dtype: int, n_splits: int, workspace: int, workspace_bytes: int,
                        stream: int = 0) -> int:
    """The raw C call sdp_fwd_splitkv with integer addresses; returns the status code."""
    return int(lib().sdp_fwd_splitkv(ctypes.c_void_p(q), ctypes.c_void_p(k), ctypes.c_void_p(v),
                                     ctypes.c_void_p(o), ctypes.c_void_p(lse), int(B), int(Hq), int(Hkv), int(Sq),
                                     int(Skv), int(D), ctypes.c_float(scale), int(dtype), int(n_splits),
                                     ctypes.c_void_p(workspace), ctypes.c_ulonglong(workspace_bytes),
                                     ctypes.c_void_p(stream)))


def splitkv_count(B: int, Hq: int, Hkv: int, Sq: int, Skv: int, D: int, dtype: int, n_splits: int = 0) -> int:
    """Split count sdp_fwd_splitkv uses for these sizes on the current device (0 = automatic)."""
    rc = int(lib().sdp_fwd_splitkv_count(B, Hq, Hkv, Sq, Skv, D, dtype, n_splits))
    _check(min(rc, 0))
    return rc


def splitkv_workspace_bytes(B: int, Hq: int, Hkv: int, Sq: int, Skv: int, D: int, dtype: int,
                            n_splits: int = 0) -> int:
    """Workspace bytes sdp_fwd_splitkv needs for these sizes on the current device."""
    rc = int(lib().sdp_fwd_splitkv_workspace_bytes(B, Hq, Hkv, Sq, Skv, D, dtype, n_splits))
    _check(min(rc, 0))
    return rc


def sdp_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float | None = None,
            out: torch.Tensor | None = None, lse: torch.Tensor | None = None, return_lse: bool = True,
            stream=None, causal: bool = False, kv_splits: int = 1, workspace: torch.Tensor | None = None):
    """Grouped-query attention forward on sm_103a (causal: row i sees keys 0..i).

    q: [B, Hq, Sq, D]; k, v: [B, Hkv, Skv, D]; fp16 or bf16, contiguous, on one
    CUDA device; D in {128, 256}; Hq a multiple of Hkv. Returns (o, lse) with o
    like q and lse fp32 [B, Hq, Sq] (None when return_lse is False and no lse
    buffer is given). The work is enqueued on `stream` (default: the current
    stream) and not synchronised.

    kv_splits != 1 (0 = automatic) runs the split-KV forward for problems with
    few query tiles (decode): the keys are cut into runs whose partial results
    are merged. Its scratch is `workspace` (a contiguous CUDA byte tensor) or,
    when None, a tensor from torch's allocator. Not combinable with causal.
    """
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D [B, H, S, D]")
    # integer device indices (get_device() is -1 off the GPU): cheaper than torch.device objects
    dev = q.get_device()
    if dev < 0 or k.get_device() != dev or v.get_device() != dev:
        raise ValueError("q, k, v must be CUDA tensors on one device")
    dt = _DTYPE_CODE.get(q.dtype)
    if dt is None or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share one dtype, float16 or bfloat16")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous")
    B, Hq, Sq, D = q.shape
    kshape = k.shape
    if kshape[0] != B or kshape[3] != D or v.shape != kshape:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)}, k {tuple(k.shape)}, v {tuple(v.shape)}")
    Hkv, Skv = kshape[1], kshape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous() or out.get_device() != dev:
        raise ValueError("out must be a contiguous tensor shaped and typed like q")
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    if lse is not None and (lse.shape != (B, Hq, Sq) or lse.dtype != torch.float32 or not lse.is_contiguous()
                            or lse.get_device() != dev):
        raise ValueError("lse must be a contiguous float32 tensor [B, Hq, Sq] on q's device")
    if kv_splits != 1:
        if causal:
            raise ValueError("the split-KV forward has no causal mask")
        with _on(q.device):
            dt = _DTYPE_CODE[q.dtype]
            need = splitkv_workspace_bytes(B, Hq, Hkv, Sq, Skv, D, dt, kv_splits)
            if workspace is None:
                workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
                if isinstance(stream, torch.cuda.Stream):
                    workspace.record_stream(stream)
            elif not (workspace.is_cuda and workspace.device == q.device and workspace.is_contiguous()):
                raise ValueError("workspace must be a contiguous tensor on q's device")
            rc = sdp_fwd_splitkv_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                     0 if lse is None else lse.data_ptr(), B, Hq, Hkv, Sq, Skv, D, float(scale),
                                     dt, kv_splits, workspace.data_ptr(),
                                     workspace.numel() * workspace.element_size(),
                                     _stream_handle(stream, q.device))
        _check(rc)
        return out, lse
    with _on(dev):
        rc = sdp_fwd_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                         0 if lse is None else lse.data_ptr(), B, Hq, Hkv, Sq, Skv, D, float(scale), dt,
                         _stream_handle(stream, dev), causal=causal)
    if rc != SDP_OK:
        _check(rc)
    return out, lse


def sdp_fwd_varlen_ptr(q: int, k: int, v: int, o: int, lse: int, cu_q: int, cu_k: int, nseq: int, Hq: int,
                       Hkv: int, total_q: int, total_k: int, max_seqlen_q: int, D: int, scale: float, dtype: int,
                       causal: bool = False, stream: int = 0) -> int:
    """The raw C call sdp_fwd_varlen with integer addresses; returns the status code."""
    return int(lib().sdp_fwd_varlen(ctypes.c_void_p(q), ctypes.c_void_p(k), ctypes.c_void_p(v), ctypes.c_void_p(o),
                                    ctypes.c_void_p(lse), ctypes.c_void_p(cu_q), ctypes.c_void_p(cu_k), int(nseq),
                                    int(Hq), int(Hkv), int(total_q), int(total_k), int(max_seqlen_q), int(D),
                                    ctypes.c_float(scale), int(dtype), int(bool(causal)), ctypes.c_void_p(stream)))


def sdp_fwd_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens_q: torch.Tensor,
                   cu_seqlens_k: torch.Tensor, max_seqlen_q: int, scale: float | None = None,
                   causal: bool = False, out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                   return_lse: bool = True, stream=None):
    """Attention over a variable-length batch packed back to back.

    q: [total_q, Hq, D]; k, v: [total_k, Hkv, D] (token, head, dim), fp16 or
    bf16, contiguous, on one CUDA device; cu_seqlens_q / cu_seqlens_k: int32
    [nseq + 1] offsets on that device; max_seqlen_q: a host int >= every query
    length. Returns (o like q, lse fp32 [Hq, total_q] or None). Sequence
    offsets are checked on the device: bad ones show up in poll_status() as
    SDP_ERR_BAD_SEQLENS.
    """
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3:
        raise ValueError("q, k, v must be 3-D [tokens, heads, D]")
    tensors = (q, k, v, cu_seqlens_q, cu_seqlens_k)
    if not all(t.is_cuda for t in tensors) or len({t.device for t in tensors}) != 1:
        raise ValueError("q, k, v and the offsets must be CUDA tensors on one device")
    if q.dtype not in _DTYPE_CODE or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("q, k, v must share one dtype, float16 or bfloat16")
    if cu_seqlens_q.dtype != torch.int32 or cu_seqlens_k.dtype != torch.int32:
        raise ValueError("sequence offsets must be int32")
    if cu_seqlens_q.dim() != 1 or cu_seqlens_q.shape != cu_seqlens_k.shape or cu_seqlens_q.numel() < 2:
        raise ValueError("sequence offsets must be 1-D [nseq + 1] of equal length")
    if not all(t.is_contiguous() for t in tensors):
        raise ValueError("q, k, v and the offsets must be contiguous")
    total_q, Hq, D = q.shape
    total_k, Hkv = k.shape[0], k.shape[1]
    if k.shape[2] != D or v.shape != k.shape:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)}, k {tuple(k.shape)}, v {tuple(v.shape)}")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous() or out.device != q.device:
        raise ValueError("out must be a contiguous tensor shaped and typed like q")
    if lse is None and return_lse:
        lse = torch.empty((Hq, total_q), dtype=torch.float32, device=q.device)
    if lse is not None and (lse.shape != (Hq, total_q) or lse.dtype != torch.float32 or not lse.is_contiguous()
                            or lse.device != q.device):
        raise ValueError("lse must be a contiguous float32 tensor [Hq, total_q] on q's device")
    with _on(q.device):
        rc = sdp_fwd_varlen_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                0 if lse is None else lse.data_ptr(), cu_seqlens_q.data_ptr(),
                                cu_seqlens_k.data_ptr(), cu_seqlens_q.numel() - 1, Hq, Hkv, total_q, total_k,
                                int(max_seqlen_q), D, float(scale), _DTYPE_CODE[q.dtype], causal,
                                _stream_handle(stream, q.device))
    _check(rc)
    return out, lse


def sdp_merge(o_parts: torch.Tensor, lse_parts: torch.Tensor, out: torch.Tensor | None = None,
              lse: torch.Tensor | None = None, return_lse: bool = True, stream=None):
    """Merge partial attention results over disjoint key sets.

    o_parts: [P, ...rows..., D] fp16/bf16 (each part's normalised output, e.g.
    sdp_fwd over one key shard), lse_parts: [P, ...rows...] fp32. Returns
    (o [...rows..., D], lse [...rows...]) over the union of the keys.
    """
    if not (o_parts.is_cuda and lse_parts.is_cuda) or o_parts.device != lse_parts.device:
        raise ValueError("o_parts and lse_parts must be CUDA tensors on one device")
    if o_parts.dtype not in _DTYPE_CODE or lse_parts.dtype != torch.float32:
        raise ValueError("o_parts must be float16/bfloat16 and lse_parts float32")
    if not (o_parts.is_contiguous() and lse_parts.is_contiguous()):
        raise ValueError("o_parts and lse_parts must be contiguous")
    P, D = o_parts.shape[0], o_parts.shape[-1]
    if tuple(lse_parts.shape) != tuple(o_parts.shape[:-1]):
        raise ValueError("lse_parts must be o_parts' shape without the last dimension")
    rows = lse_parts.numel() // P
    if out is None:
        out = torch.empty(o_parts.shape[1:], dtype=o_parts.dtype, device=o_parts.device)
    if lse is None and return_lse:
        lse = torch.empty(lse_parts.shape[1:], dtype=torch.float32, device=o_parts.device)
    with _on(o_parts.device):
        rc = int(lib().sdp_merge(ctypes.c_void_p(o_parts.data_ptr()), ctypes.c_void_p(lse_parts.data_ptr()), int(P),
                                 int(rows), int(D), _DTYPE_CODE[o_parts.dtype], ctypes.c_void_p(out.data_ptr()),
                                 ctypes.c_void_p(0 if lse is None else lse.data_ptr()),
                                 ctypes.c_void_p(_stream_handle(stream, o_parts.device))))
    _check(rc)
    return out, lse


def poll_status(stream=None, device=None) -> int:
    """Synchronise the stream and return (and clear) the device status code."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        return int(lib().sdp_poll_status(ctypes.c_void_p(_stream_handle(stream, dev))))


def last_status_detail() -> int:
    return int(lib().sdp_last_status_detail())


def set_wait_timeout_ms(ms: int) -> int:
    return int(lib().sdp_set_wait_timeout_ms(int(ms)))


def set_debug_flags(flags: int) -> int:
    """Test hooks of the C library (0 by default; returns the previous flags).

    1: the load warp issues no copies (every wait runs out: the timeout path);
    2: never the CTA-pair kernel; 4: never pack a group's query heads; 8: the
    CTA-pair kernel at head dim 128 too; 16: one CTA (pair) per unit where a
    persistent kernel would run; 32: variable-length launches on the full grid
    instead of the compact tile list; 64: never the two-tile CTA-pair kernel at
    head dim 128; 128: the two-tile CTA-pair kernel (two query tiles per CTA,
    64-key steps) for dense non-causal head-dim-128 launches whose units pair.
    4, 16 and 32 give bit-identical results; 2, 8 and 128 switch kernels that
    compute the same function.
    """
    return int(lib().sdp_set_debug_flags(int(flags)))


def sdp_fwd_noalloc_ptr(q: int, k: int, v: int, o: int, lse: int, B: int, Hq: int, Hkv: int, Sq: int, Skv: int,
                        D: int, scale: float, dtype: int, stream: int = 0) -> int:
    """The C call sdp_fwd_noalloc with integer addresses; returns the status code.

    Same operation, arguments and launch as sdp_fwd_ptr (bit-identical
    outputs), but the library allocates no device memory for it: for callers
    whose device memory is owned entirely by their own pool or host
    application and that therefore cannot let a library call cudaMalloc. Its
    status word (and the persistent kernel's claim counters) live in a static
    array inside the library shared by all such calls, so overlapping calls on
    different unordered streams race on the status word; read it with
    noalloc_status(), not poll_status().
    """
    L = lib()
    fn = L.sdp_fwd_noalloc
    if fn.restype is not ctypes.c_int or fn.argtypes is None:
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        fn.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
        fn.restype = i
    return int(fn(ctypes.c_void_p(q), ctypes.c_void_p(k), ctypes.c_void_p(v), ctypes.c_void_p(o),
                  ctypes.c_void_p(lse), int(B), int(Hq), int(Hkv), int(Sq), int(Skv), int(D), ctypes.c_float(scale),
                  int(dtype), ctypes.c_void_p(stream)))


def noalloc_status(stream=None, device=None) -> int:
    """Synchronise the stream, then read and clear sdp_fwd_noalloc's status word (allocates nothing)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    fn = lib().sdp_fwd_noalloc_status
    if fn.restype is not ctypes.c_int or fn.argtypes is None:
        fn.argtypes = [ctypes.c_void_p]
        fn.restype = ctypes.c_int
    with torch.cuda.device(dev):
        return int(fn(ctypes.c_void_p(_stream_handle(stream, dev))))


# Short names of the main entry points.
fwd = sdp_fwd
fwd_varlen = sdp_fwd_varlen
merge = sdp_merge
