"""Seeded synthetic workloads for the grouped-query attention forward.

This module only draws random inputs and names shapes; it holds none of the
attention arithmetic. Both the CUDA path (tests, benchmark) and the oracle
consume what it produces.

Input recipe: standard-normal fp32 values from numpy's PCG64 generator
(bit-reproducible across machines), rounded to nearest-even into fp16 or
bf16. The peaky-softmax workload multiplies exactly ceil(1% * Skv) K rows per
(batch, KV head), chosen by a seeded permutation, by 8 before rounding (8 is
a power of two, so the order of scaling and rounding does not matter).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np
import torch

DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Skv: int
    D: int
    dtype: str = "fp16"
    seed: int = 0
    peaky_k: bool = False
    scale: float | None = None  # None means 1/sqrt(D)
    causal: bool = False        # row i sees keys 0..i
    kv_splits: int = 1          # launch: split-KV run count (0 = automatic, 1 = none)
    note: str = field(default="", compare=False)

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.D) if self.scale is None else float(self.scale)

    @property
    def torch_dtype(self) -> torch.dtype:
        return DTYPES[self.dtype]

    @property
    def shape(self):
        return (self.B, self.Hq, self.Hkv, self.Sq, self.Skv, self.D)

    def flops(self) -> int:
        """Matmul FLOPs: 4 * D per (query row, key it sees) per query head (two
        contractions): 4 * Sq * Skv * D, or, causal, 4 * D * sum_i min(i + 1, Skv)."""
        if not self.causal:
            return 4 * self.B * self.Hq * self.Sq * self.Skv * self.D
        full = min(self.Sq, self.Skv)  # rows 0..full-1 see i + 1 keys, the rest see all Skv
        seen = full * (full + 1) // 2 + (self.Sq - full) * self.Skv
        return 4 * self.B * self.Hq * seen * self.D

    def hbm_bytes(self) -> int:
        """Algorithmic HBM bytes: Q, K, V read once, O written once (16-bit), LSE fp32."""
        e = 2
        q = self.B * self.Hq * self.Sq * self.D * e
        kv = 2 * self.B * self.Hkv * self.Skv * self.D * e
        o = q
        lse = self.B * self.Hq * self.Sq * 4
        return q + kv + o + lse

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads of the attention-forward study (head dims 128 and 256,
# fp16 and bf16 I/O, GQA ratios 4:1 and 16:1, and plain multi-head).
WORKLOADS = {
    "gqa4_s256_d128_fp16": Workload("gqa4_s256_d128_fp16", 1, 4, 1, 256, 256, 128, "fp16", seed=1),
    "gqa16_s4k_d256_fp16": Workload("gqa16_s4k_d256_fp16", 1, 32, 2, 4096, 4096, 256, "fp16", seed=2),
    "gqa16_s16k_d256_fp16": Workload("gqa16_s16k_d256_fp16", 1, 32, 2, 16384, 16384, 256, "fp16", seed=3),
    "gqa4_b2_s8k_d128_bf16_peaky": Workload("gqa4_b2_s8k_d128_bf16_peaky", 2, 32, 8, 8192, 8192, 128, "bf16",
                                            seed=4, peaky_k=True),
    "mha_b4_s16k_d128_fp16": Workload("mha_b4_s16k_d128_fp16", 4, 32, 32, 16384, 16384, 128, "fp16", seed=5),
}

# The pages' headline shape: 32 query heads over 2 KV heads, head dim 256, 16K x 16K.
HEADLINE = "gqa16_s16k_d256_fp16"

# Causal counterparts (row i sees keys 0..i), the next step of the study; they
# are benchmark and parity cases beside the five workloads above.
CAUSAL_WORKLOADS = {
    "gqa16_s16k_d256_fp16_causal": WORKLOADS["gqa16_s16k_d256_fp16"].with_(name="gqa16_s16k_d256_fp16_causal",
                                                                           causal=True),
    "mha_b4_s16k_d128_fp16_causal": WORKLOADS["mha_b4_s16k_d128_fp16"].with_(name="mha_b4_s16k_d128_fp16_causal",
                                                                             causal=True),
}
# Small-Sq shapes (the study's dispatch picks kernels by query length, with a
# crossover at 16 rows): one-token decode over a long context, and 16 rows.
# They run the split-KV forward with an automatic split count.
DECODE_WORKLOADS = {
    "gqa16_decode_b8_s16k_d256_fp16": Workload("gqa16_decode_b8_s16k_d256_fp16", 8, 32, 2, 1, 16384, 256, "fp16",
                                               seed=8, kv_splits=0),
    "gqa4_decode_b4_s32k_d128_bf16": Workload("gqa4_decode_b4_s32k_d128_bf16", 4, 32, 8, 1, 32768, 128, "bf16",
                                              seed=9, kv_splits=0),
    "gqa16_sq16_s16k_d256_fp16": Workload("gqa16_sq16_s16k_d256_fp16", 1, 32, 2, 16, 16384, 256, "fp16",
                                          seed=10, kv_splits=0),
}
ALL_WORKLOADS = {**WORKLOADS, **CAUSAL_WORKLOADS, **DECODE_WORKLOADS}


@dataclass(frozen=True)
class VarlenWorkload:
    """A batch of sequences of different lengths packed back to back.

    Sequence b has lens_q[b] query rows and lens_k[b] key rows; Q is
    [total_q, Hq, D] and K, V are [total_k, Hkv, D] (token, head, dim).
    """
    name: str
    lens_q: tuple
    lens_k: tuple
    Hq: int
    Hkv: int
    D: int
    dtype: str = "fp16"
    seed: int = 0
    scale: float | None = None
    causal: bool = False
    note: str = field(default="", compare=False)

    @property
    def nseq(self) -> int:
        return len(self.lens_q)

    @property
    def total_q(self) -> int:
        return int(sum(self.lens_q))

    @property
    def total_k(self) -> int:
        return int(sum(self.lens_k))

    @property
    def max_q(self) -> int:
        return int(max(self.lens_q))

    @property
    def cu_q(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.lens_q)]).astype(np.int32)

    @property
    def cu_k(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.lens_k)]).astype(np.int32)

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.D) if self.scale is None else float(self.scale)

    @property
    def torch_dtype(self) -> torch.dtype:
        return DTYPES[self.dtype]

    def flops(self) -> int:
        """4 * D FLOPs per (query head, query row, key the row sees)."""
        seen = 0
        for lq, lk in zip(self.lens_q, self.lens_k):
            if not self.causal:
                seen += lq * lk
            else:
                full = min(lq, lk)
                seen += full * (full + 1) // 2 + (lq - full) * lk
        return 4 * self.Hq * self.D * seen

    def hbm_bytes(self) -> int:
        q = self.total_q * self.Hq * self.D * 2
        kv = 2 * self.total_k * self.Hkv * self.D * 2
        return 2 * q + kv + self.total_q * self.Hq * 4


def varlen_lengths(n: int, lo: int, hi: int, seed: int) -> tuple:
    """n lengths, log-uniform in [lo, hi] (PCG64, seeded), as a tuple of ints."""
    rng = np.random.default_rng(seed)
    x = np.exp(rng.uniform(math.log(lo), math.log(hi), size=n))
    return tuple(int(round(t)) for t in x)


_VL_A = varlen_lengths(12, 256, 16384, seed=11)
_VL_B = varlen_lengths(24, 64, 8192, seed=12)
# Packed prefill batches: a long-tailed mix of sequence lengths (log-uniform),
# so most sequences end inside a 128-row tile. Self-attention (keys =
# queries) on the headline head layout, and a bf16 batch whose key lengths
# (history + chunk) exceed the query lengths.
VARLEN_WORKLOADS = {
    "varlen12_gqa16_d256_fp16": VarlenWorkload("varlen12_gqa16_d256_fp16", _VL_A, _VL_A, 32, 2, 256, "fp16",
                                               seed=11),
    "varlen12_gqa16_d256_fp16_causal": VarlenWorkload("varlen12_gqa16_d256_fp16_causal", _VL_A, _VL_A, 32, 2, 256,
                                                      "fp16", seed=11, causal=True),
    "varlen24_gqa4_d128_bf16": VarlenWorkload("varlen24_gqa4_d128_bf16", _VL_B,
                                              tuple(x + y for x, y in zip(_VL_B, varlen_lengths(24, 1, 4096, 13))),
                                              32, 8, 128, "bf16", seed=12),
}


def _normal(rng: np.random.Generator, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    step = 1 << 26
    for s in range(0, n, step):
        out[s:s + step] = rng.standard_normal(min(step, n - s), dtype=np.float32)
    return out


def _round(x: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(x)
    return t.to(DTYPES[dtype])  # round to nearest even


def make_inputs(w: Workload):
    """(q, k, v) as contiguous CPU tensors of the workload's dtype.

    q: [B, Hq, Sq, D]; k, v: [B, Hkv, Skv, D].
    """
    rng = np.random.default_rng(w.seed)
    nq = w.B * w.Hq * w.Sq * w.D
    nkv = w.B * w.Hkv * w.Skv * w.D
    q = _normal(rng, nq)
    k = _normal(rng, nkv)
    v = _normal(rng, nkv)
    if w.peaky_k:
        k = k.reshape(w.B * w.Hkv, w.Skv, w.D)
        n_peak = math.ceil(0.01 * w.Skv)
        for bh in range(w.B * w.Hkv):
            idx = rng.permutation(w.Skv)[:n_peak]
            k[bh, idx, :] *= 8.0
        k = k.reshape(-1)
    q = _round(q, w.dtype).reshape(w.B, w.Hq, w.Sq, w.D)
    k = _round(k, w.dtype).reshape(w.B, w.Hkv, w.Skv, w.D)
    v = _round(v, w.dtype).reshape(w.B, w.Hkv, w.Skv, w.D)
    return q, k, v


def sample_rows(w: Workload, n: int = 256, seed: int | None = None) -> np.ndarray:
    """Seeded sample of query rows per (b, h): int32 [B, Hq, m], m = min(n, Sq).

    Every head's sample holds rows 0 and Sq-1; rows are sorted and distinct.
    """
    m = min(n, w.Sq)
    rng = np.random.default_rng(w.seed * 7919 + 17 if seed is None else seed)
    out = np.empty((w.B, w.Hq, m), dtype=np.int32)
    for b in range(w.B):
        for h in range(w.Hq):
            if m == w.Sq:
                out[b, h] = np.arange(w.Sq, dtype=np.int32)
                continue
            mid = rng.choice(np.arange(1, w.Sq - 1), size=m - 2, replace=False) if m > 2 else []
            rows = np.concatenate([[0], np.sort(mid), [w.Sq - 1]])[:m]
            out[b, h] = np.sort(rows).astype(np.int32)
    return out


def make_varlen_inputs(w: VarlenWorkload):
    """(q, k, v) as contiguous CPU tensors of the workload's dtype, packed
    (token, head, dim): q [total_q, Hq, D], k and v [total_k, Hkv, D]; same
    recipe as make_inputs. The sequence offsets are w.cu_q and w.cu_k."""
    rng = np.random.default_rng(w.seed)
    q = _normal(rng, w.total_q * w.Hq * w.D)
    k = _normal(rng, w.total_k * w.Hkv * w.D)
    v = _normal(rng, w.total_k * w.Hkv * w.D)
    q = _round(q, w.dtype).reshape(w.total_q, w.Hq, w.D)
    k = _round(k, w.dtype).reshape(w.total_k, w.Hkv, w.D)
    v = _round(v, w.dtype).reshape(w.total_k, w.Hkv, w.D)
    return q, k, v
