"""Writes oracle_small_int.json: the oracle's outputs on small, platform-
independent inputs (SplitMix64 small integers, exact in bf16).

Calls only ``oracle/`` and the input generators.  The fixture guards the
oracle against unintended changes and checks that x86 and Arm hosts agree
bit for bit.  Method: DeepSpeed PR #8602 "Plan B: Dual-Weight GEMV" (fused
mode) and PR #9057 "Changes" (HF-boundary mode, residual + zero-centred
RMSNorm).  Run:  python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import glu_inputs as gi  # noqa: E402

CASES = [  # (M, N, K, seed)
    (1, 7, 16, 1), (3, 5, 40, 2), (4, 9, 24, 3),
]


def inputs(M, N, K, seed):
    h = gi.small_int_bf16((M, K), seed * 10 + 1, -4, 4)
    g = gi.small_int_bf16((N, K), seed * 10 + 2, -2, 2)
    u = gi.small_int_bf16((N, K), seed * 10 + 3, -2, 2)
    x = gi.small_int_bf16((M, K), seed * 10 + 4, -6, 6)
    r = gi.small_int_bf16((M, K), seed * 10 + 5, -6, 6)
    w = gi.small_int_bf16((K,), seed * 10 + 6, -1, 1)
    return h, g, u, x, r, w


def compute():
    out = []
    for (M, N, K, seed) in CASES:
        h, g, u, x, r, w = inputs(M, N, K, seed)
        rec = {"M": M, "N": N, "K": K, "seed": seed}
        for mode in ("fused", "hf"):
            rec[f"glu_{mode}"] = oracle.glu_gemv(h, g, u, mode, nthreads=1).tolist()
        o, res, hn = oracle.add_rmsnorm_glu(x, r, w, 1e-6, g, u, "hf", nthreads=1)
        rec["norm_glu_hf"] = o.tolist()
        rec["norm_residual"] = res.tolist()
        rec["norm_h"] = hn.tolist()
        out.append(rec)
    return out


if __name__ == "__main__":
    with open(os.path.join(HERE, "oracle_small_int.json"), "w") as f:
        json.dump({"source": "tests/golden/make_golden.py (oracle only)", "cases": compute()}, f)
        f.write("\n")
