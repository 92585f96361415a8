"""The C ABI used from plain C: a client built with gcc against include/sdp.h
and libsdp.so (no Python or framework types across the boundary) computes the
same attention as the oracle."""
import os
import subprocess
import tempfile

import numpy as np
import pytest
import torch

import oracle
from gqa_flash_attention_gb300 import workloads
from gqa_flash_attention_gb300.workloads import Workload
from parity import ORACLE_DTYPE, assert_within, compare

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
PKG = os.path.join(ROOT, "gqa_flash_attention_gb300")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def build_client(out_dir):
    from gqa_flash_attention_gb300 import build
    build.build()
    exe = os.path.join(out_dir, "c_client")
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-o", exe, os.path.join(HERE, "c_client.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           "-L", PKG, "-lsdp", f"-Wl,-rpath,{PKG}", "-L", os.path.join(CUDA, "lib64"), "-lcudart"]
    subprocess.run(cmd, check=True)
    return exe


def test_c_client_builds_and_links():
    with tempfile.TemporaryDirectory() as d:
        exe = build_client(d)
        r = subprocess.run(["nm", "-D", "--undefined-only", exe], capture_output=True, text=True)
        assert "sdp_fwd" in r.stdout


@pytest.mark.gpu
@pytest.mark.parametrize("w,mode", [
    (Workload("c_gqa", 1, 8, 2, 300, 500, 128, "fp16", seed=95), ["fwd"]),
    (Workload("c_bf16", 2, 4, 4, 129, 130, 256, "bf16", seed=96), ["fwd"]),
    (Workload("c_causal", 1, 8, 2, 300, 300, 256, "fp16", seed=97, causal=True), ["causal"]),
    (Workload("c_splitkv", 2, 16, 2, 1, 3000, 256, "fp16", seed=98), ["splitkv", "0"]),
    (Workload("c_splitkv3", 1, 8, 4, 7, 2000, 128, "bf16", seed=99), ["splitkv", "3"]),
    (Workload("c_noalloc", 1, 16, 1, 1, 1000, 256, "fp16", seed=100), ["noalloc"]),
    # 160 units at head dim 128: the persistent single-CTA kernel on the legacy default stream
    (Workload("c_persist", 1, 8, 2, 2560, 500, 128, "fp16", seed=101), ["fwd"]),
    (Workload("c_persist_noalloc", 1, 8, 2, 2560, 500, 128, "bf16", seed=102), ["noalloc"]),
], ids=lambda x: x.name if isinstance(x, Workload) else "-".join(x))
def test_c_client_matches_the_oracle(w, mode):
    q, k, v = workloads.make_inputs(w)
    with tempfile.TemporaryDirectory() as d:
        exe = build_client(d)
        fin, fout = os.path.join(d, "in.bin"), os.path.join(d, "out.bin")
        with open(fin, "wb") as f:
            for t in (q, k, v):
                f.write(t.contiguous().view(torch.int16).numpy().tobytes())
        dt = 1 if w.dtype == "bf16" else 0
        r = subprocess.run([exe, fin, fout, *map(str, (w.B, w.Hq, w.Hkv, w.Sq, w.Skv, w.D, dt)),
                            repr(w.softmax_scale), *mode], capture_output=True, text=True, timeout=300)
        assert r.returncode == 0, r.stderr
        raw = open(fout, "rb").read()
    nq = q.numel()
    o = torch.from_numpy(np.frombuffer(raw[:2 * nq], dtype=np.int16).copy()).view(w.torch_dtype).view(q.shape)
    lse = torch.from_numpy(np.frombuffer(raw[2 * nq:], dtype=np.float32).copy()).view(w.B, w.Hq, w.Sq)
    ref_o, ref_l = oracle.sdp_fwd(q, k, v, ORACLE_DTYPE[w.dtype], w.shape, w.softmax_scale, causal=w.causal)
    assert_within(compare(o, lse, ref_o, ref_l, w.dtype), w.dtype)
