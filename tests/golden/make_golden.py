"""Writes tests/golden/oracle_gqa_small.txt from the oracle alone.

The fixture freezes the oracle's fp64 output on one tiny seeded grouped-query
case (4 query heads over 2 KV heads, 5 x 7, head dim 16, fp16 inputs), so that
a later change to the oracle, or a platform whose libm differs, shows up as a
diff. The values are not from the pages (they print no worked attention
example); the pins in tests/test_oracle.py tie the oracle to closed forms,
invariants, brute force and PyTorch's float64 attention.

Run: python tests/golden/make_golden.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from gqa_flash_attention_gb300.workloads import Workload, make_inputs  # noqa: E402

CASE = Workload("golden_gqa_small", B=1, Hq=4, Hkv=2, Sq=5, Skv=7, D=16, dtype="fp16", seed=99)


def compute():
    q, k, v = make_inputs(CASE)
    return oracle.sdp_fwd(q, k, v, oracle.FP16, CASE.shape, CASE.softmax_scale)


def main():
    o, lse = compute()
    path = os.path.join(HERE, "oracle_gqa_small.txt")
    with open(path, "w") as f:
        f.write("# oracle output, B=1 Hq=4 Hkv=2 Sq=5 Skv=7 D=16 fp16 seed=99 scale=1/sqrt(16)\n")
        f.write("# written by tests/golden/make_golden.py (oracle only)\n")
        f.write("# lines: 'lse b h i value' then 'o b h i d0..d15'\n")
        for h in range(CASE.Hq):
            for i in range(CASE.Sq):
                f.write(f"lse 0 {h} {i} {float(lse[0, h, i])!r}\n")
                f.write(f"o 0 {h} {i} " + " ".join(repr(float(x)) for x in o[0, h, i]) + "\n")


if __name__ == "__main__":
    main()
