"""Helpers for comparing the CUDA path with the oracle.

Tolerances (relative rms = sqrt(sum (o - r)^2 / sum r^2) over all checked O
elements; max abs = max |o - r|), fixed by the attention-forward study's
accuracy targets for 16-bit inputs with fp32 softmax statistics:
fp16 I/O: rel rms <= 3e-3, max abs <= 2e-2; bf16 I/O: rel rms <= 6e-3, max abs
<= 4e-2. The log-sum-exp is fp32 in both kernels: max abs <= 1e-3.
NaNs are counted before anything else.
"""
import numpy as np
import torch

import oracle

TOL = {
    "fp16": dict(rel_rms=3e-3, max_abs=2e-2),
    "bf16": dict(rel_rms=6e-3, max_abs=4e-2),
}
LSE_MAX_ABS = 1e-3
ORACLE_DTYPE = {"fp16": oracle.FP16, "bf16": oracle.BF16}


def compare(o_gpu, lse_gpu, o_ref, lse_ref, dtype):
    o = o_gpu.double().cpu().numpy() if isinstance(o_gpu, torch.Tensor) else np.asarray(o_gpu, dtype=np.float64)
    stats = {"nan_o": int(np.isnan(o).sum()) + int(np.isinf(o).sum())}
    diff = o - o_ref
    stats["rel_rms"] = float(np.sqrt((diff ** 2).sum() / max((o_ref ** 2).sum(), 1e-300)))
    stats["max_abs"] = float(np.abs(diff).max()) if diff.size else 0.0
    if lse_gpu is not None:
        l = lse_gpu.double().cpu().numpy() if isinstance(lse_gpu, torch.Tensor) else np.asarray(lse_gpu)
        stats["nan_lse"] = int((~np.isfinite(l)).sum())
        stats["lse_max_abs"] = float(np.abs(l - lse_ref).max()) if l.size else 0.0
    return stats


def assert_within(stats, dtype):
    tol = TOL[dtype]
    assert stats["nan_o"] == 0, stats
    assert stats.get("nan_lse", 0) == 0, stats
    assert stats["rel_rms"] <= tol["rel_rms"], stats
    assert stats["max_abs"] <= tol["max_abs"], stats
    if "lse_max_abs" in stats:
        assert stats["lse_max_abs"] <= LSE_MAX_ABS, stats
