"""Sizes past 32-bit element offsets, and a long key sequence.

Q and O of the first case hold more than 2^31 elements each (4.3 GB apiece),
so every byte offset the TMA maps, the LSE index and the host validation
compute must be 64-bit. The second case streams 2048 KV tiles through one
CTA's online softmax. Inputs are drawn on the GPU (seeded torch generator,
standard normal rounded to fp16 / bf16) to keep the host out of the way; the
oracle checks sampled rows on copies of just the heads it needs.
"""
import numpy as np
import pytest
import torch

import gqa_flash_attention_gb300 as sdp
import oracle
from parity import assert_within, compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gqa_flash_attention_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    sdp.lib()


def randn(shape, dtype, gen):
    t = torch.empty(shape, dtype=dtype, device="cuda")
    flat = t.view(-1)
    step = 1 << 28
    for s in range(0, flat.numel(), step):
        n = min(step, flat.numel() - s)
        flat[s:s + n] = torch.randn(n, generator=gen, device="cuda", dtype=torch.float32).to(dtype)
    return t


def check_sampled(q, k, v, o, lse, heads, rows, scale, odt):
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k.shape[1], k.shape[2]
    G = Hq // Hkv
    groups = sorted({h // G for h in heads})
    # a reduced problem: the sampled query heads (as one head each of their own group)
    qs = torch.stack([q[0, h, rows] for h in heads]).unsqueeze(0).cpu()          # [1, nh, nr, D]
    ks = torch.stack([k[0, h // G] for h in heads]).unsqueeze(0).cpu()           # [1, nh, Skv, D]
    vs = torch.stack([v[0, h // G] for h in heads]).unsqueeze(0).cpu()
    nh, nr = len(heads), len(rows)
    ref_o, ref_l = oracle.sdp_fwd(qs, ks, vs, odt, (1, nh, nh, nr, Skv, D), scale)
    got_o = torch.stack([o[0, h, rows] for h in heads]).unsqueeze(0)
    got_l = torch.stack([lse[0, h, rows] for h in heads]).unsqueeze(0)
    return compare(got_o, got_l, ref_o, ref_l, "fp16" if odt == oracle.FP16 else "bf16"), groups


def test_more_than_2_31_elements_per_tensor():
    gen = torch.Generator(device="cuda").manual_seed(2024)
    B, Hq, Hkv, S, D = 1, 64, 8, 131201, 256   # 64 * 131201 * 256 > 2^31 elements in Q and O
    assert B * Hq * S * D > 2 ** 31
    q = randn((B, Hq, S, D), torch.float16, gen)
    k = randn((B, Hkv, S, D), torch.float16, gen)
    v = randn((B, Hkv, S, D), torch.float16, gen)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, Hq, S), float("nan"), device="cuda")
    scale = 1.0 / 16
    sdp.sdp_fwd(q, k, v, scale=scale, out=o, lse=lse)
    assert sdp.poll_status() == sdp.SDP_OK
    heads = [0, 31, 63]
    rows = [0, 1, 65535, 131071, 131199, 131200]
    st, _ = check_sampled(q, k, v, o, lse, heads, rows, scale, oracle.FP16)
    assert_within(st, "fp16")
    # the last rows of the last head sit past element 2^31: they were written
    assert not torch.isnan(o[0, 63, -1]).any() and not torch.isnan(lse[0, 63, -1])
    del q, k, v, o, lse
    torch.cuda.empty_cache()


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_long_key_sequence(dtype):
    gen = torch.Generator(device="cuda").manual_seed(7)
    B, Hq, Hkv, Sq, Skv, D = 1, 4, 1, 256, 262144 - 77, 128   # 2048 KV tiles, ragged tail
    q = randn((B, Hq, Sq, D), dtype, gen)
    k = randn((B, Hkv, Skv, D), dtype, gen)
    v = randn((B, Hkv, Skv, D), dtype, gen)
    o, lse = sdp.sdp_fwd(q, k, v)
    assert sdp.poll_status() == sdp.SDP_OK
    rows = list(np.random.default_rng(3).choice(Sq, 12, replace=False)) + [0, Sq - 1]
    odt = oracle.FP16 if dtype == torch.float16 else oracle.BF16
    st, _ = check_sampled(q, k, v, o, lse, [0, 3], sorted(int(r) for r in rows), 1.0 / np.sqrt(D), odt)
    assert_within(st, "fp16" if dtype == torch.float16 else "bf16")
