"""Writes tests/golden/worked_example.json from the CPU oracle only.

A 3-token, one-head example with d_k = 2, d_v = 3 and small rational inputs
(alpha = 1/2 via g = ln(1/2)).  The pages print no worked example, so the
stored values are the oracle's; tests/test_oracle_golden.py pins them to
exact rational arithmetic of the gated delta rule (page "IsoExec: 切换 SkyRL
中的训练器-推理不匹配", section "Chunkwise-Parallel Recurrent (CPR) Gated
DeltaNet") and guards the oracle against regressions.

Run:  python tests/golden/make_golden.py
"""
import json
import math
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402

EXAMPLE = dict(
    q=[[[1, 2]], [[-1, 1]], [[0.5, -2]]],
    k=[[[1, 0]], [[0.5, 0.5]], [[-1, 1]]],
    v=[[[1, -1, 2]], [[0, 3, -1]], [[2, 2, 0.5]]],
    g_over_ln_half=[[0], [1], [2]],          # alpha = (1/2)^n
    beta=[[0.5], [0.25], [0.75]],
    h0=[[[[1, 0, -1], [0.5, 2, 0]]]],
    dO=[[[1, 0, -1]], [[2, 1, 0]], [[-1, 0.5, 1]]],
    dHT=[[[[0, 1, 0], [1, 0, -1]]]],
    scale=0.5,
)


def main():
    ex = EXAMPLE
    q, k, v = (np.array(ex[n], dtype=np.float64) for n in ("q", "k", "v"))
    g = np.array(ex["g_over_ln_half"], dtype=np.float64) * math.log(0.5)
    beta = np.array(ex["beta"], dtype=np.float64)
    h0 = np.array(ex["h0"], dtype=np.float64)
    dO = np.array(ex["dO"], dtype=np.float64)
    dHT = np.array(ex["dHT"], dtype=np.float64)
    cu = [0, 3]
    o, hT = oracle.gdn_fwd(q, k, v, g, beta, cu, h0=h0, scale=ex["scale"])
    gr = oracle.gdn_bwd(q, k, v, g, beta, cu, dO, h0=h0, dHT=dHT, scale=ex["scale"])
    out = dict(source="oracle.gdn_fwd / oracle.gdn_bwd (fp64)", inputs=ex,
               o=o.tolist(), hT=hT.tolist(), **{n: a.tolist() for n, a in gr.items()})
    with open(os.path.join(HERE, "worked_example.json"), "w") as f:
        json.dump(out, f, separators=(",", ":"))
        f.write("\n")


if __name__ == "__main__":
    main()
