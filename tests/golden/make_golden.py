"""Writes tests/golden/oracle_regression_small.json from the fp64 oracle only.

The pages print no numeric worked example for attention, so this fixture is a
regression record of the oracle itself (its independent pins live in
tests/test_oracle.py).  Run: python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import torch  # noqa: E402

from oracle import attn_fwd_oracle  # noqa: E402


def case():
    g = torch.Generator("cpu").manual_seed(4242)
    B, N, Hq, Hkv, d = 1, 12, 4, 2, 8
    q = torch.randn((B, N, Hq, d), generator=g).to(torch.bfloat16)
    k = torch.randn((B, N, Hkv, d), generator=g).to(torch.bfloat16)
    v = torch.randn((B, N, Hkv, d), generator=g).to(torch.bfloat16)
    return dict(B=B, N=N, Hq=Hq, Hkv=Hkv, d=d, scale=d ** -0.5, causal=True), q, k, v


def main():
    meta, q, k, v = case()
    o, lse = attn_fwd_oracle(q, k, v, meta["B"], meta["Hq"], meta["Hkv"], meta["N"],
                             meta["d"], meta["scale"], meta["causal"])
    out = dict(meta, source="oracle/ (fp64 two-pass attention), seed 4242",
               o=o.reshape(-1).tolist(), lse=lse.reshape(-1).tolist())
    with open(os.path.join(HERE, "oracle_regression_small.json"), "w") as f:
        json.dump(out, f, indent=0)


if __name__ == "__main__":
    main()
