"""Writes oracle_tiny.txt: the oracle's forward (O, LSE) and backward (dQ, dK, dV) on one fixed,
seeded tiny input, as a regression fixture for later changes to the oracle.

Calls only the oracle (and the shared seeded input generator). Rerun it only when a change to
the oracle's arithmetic is justified by a passage of the pages; name that passage in the commit.
    python tests/golden/make_oracle_tiny.py
"""
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from io_aware_attention_fa2_gb300.inputs import make_qkv, normal, round_to_bits  # noqa: E402

CASE = dict(B=1, H=2, N=5, d=4, dtype="bf16", seed=4242, scale=0.5)


def compute():
    c = CASE
    qb, kb, vb = make_qkv(c["B"], c["H"], c["N"], c["d"], c["dtype"], c["seed"])
    dob = round_to_bits(normal((c["B"], c["N"], c["H"], c["d"]), c["seed"] + 9), c["dtype"])
    out = {}
    for causal in (False, True):
        o, lse = oracle.attention(qb, kb, vb, causal, c["scale"], dtype=c["dtype"])
        dq, dk, dv = oracle.attention_bwd(qb, kb, vb, dob, causal, c["scale"], dtype=c["dtype"])
        tag = "causal" if causal else "full"
        for name, arr in (("o", o), ("lse", lse), ("dq", dq), ("dk", dk), ("dv", dv)):
            out["%s_%s" % (name, tag)] = np.asarray(arr, dtype=np.float64).ravel()
    return out


def main():
    lines = [
        "# The oracle's outputs on one seeded tiny input (written by make_oracle_tiny.py, which",
        "# calls only the oracle). Forward: \"FlashAttention 优化原理与实现要点解析\" §1-§2 (the",
        "# definition), §7 (causal mask), LSE = m + ln l as kept per \"FlashAttention V2 核心原理与",
        "# 架构设计\" §2.3; backward: the chain-rule gradients of the same definition.",
        "# case: " + ", ".join("%s=%s" % kv for kv in CASE.items()),
        "# one array per line: name, then its values (row-major, the oracle's layouts) in %.17g",
    ]
    for name, arr in compute().items():
        lines.append(name + " " + " ".join("%.17g" % x for x in arr))
    with open(os.path.join(HERE, "oracle_tiny.txt"), "w") as f:
        f.write("\n".join(lines) + "\n")


if __name__ == "__main__":
    main()
