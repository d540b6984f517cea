"""Pin: a worked example in exact rational arithmetic.

tests/golden/worked_example.json holds the oracle's fp64 output for a tiny
example with rational inputs (written by tests/golden/make_golden.py).  Here
the gated delta rule
    S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T,  o_t = S_t (scale q_t)
(page "IsoExec: 切换 SkyRL 中的训练器-推理不匹配", section
"Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet") is evaluated with
Python Fractions -- explicit matrices, no rounding -- and the gradients with
forward-mode dual numbers over Fractions, one input direction at a time.
The stored values must match the exact ones to fp64 rounding, and the oracle
must still reproduce the stored values.
"""
import json
import math
import os
from fractions import Fraction as F

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example.json")


class Dual:
    """a + b eps, eps^2 = 0, over Fractions."""
    __slots__ = ("a", "b")

    def __init__(self, a, b=F(0)):
        self.a, self.b = F(a), F(b)

    def __add__(self, o):
        o = o if isinstance(o, Dual) else Dual(o)
        return Dual(self.a + o.a, self.b + o.b)

    __radd__ = __add__

    def __sub__(self, o):
        o = o if isinstance(o, Dual) else Dual(o)
        return Dual(self.a - o.a, self.b - o.b)

    def __rsub__(self, o):
        return Dual(o) - self

    def __mul__(self, o):
        o = o if isinstance(o, Dual) else Dual(o)
        return Dual(self.a * o.a, self.a * o.b + self.b * o.a)

    __rmul__ = __mul__


def _alpha(n, dg):
    # alpha = exp(g), g = n ln(1/2) + eps dg  =>  alpha = 2^-n (1 + eps dg)
    a = F(1, 2 ** n)
    return Dual(a, a * dg)


def _exact(ex, seed_dir=None):
    """Exact forward; seed_dir = (name, index) puts eps on that input."""
    T, dk, dv = 3, 2, 3

    def val(name, *idx):
        x = ex[name]
        for i in idx:
            x = x[i]
        d = F(1) if seed_dir == (name, idx) else F(0)
        return Dual(F(x), d)

    S = [[val("h0", 0, 0, j, i) for j in range(dk)] for i in range(dv)]  # S = h0^T
    loss = Dual(0)
    os_ = []
    for t in range(T):
        n = ex["g_over_ln_half"][t][0]
        dg = F(1) if seed_dir == ("g", (t, 0)) else F(0)
        a = _alpha(n, dg)
        b = val("beta", t, 0)
        kk = [val("k", t, 0, j) for j in range(dk)]
        vv = [val("v", t, 0, i) for i in range(dv)]
        qq = [val("q", t, 0, j) for j in range(dk)]
        # M = I - b k k^T ; S <- a S M + b v k^T
        M = [[(Dual(1) if r == c else Dual(0)) - b * kk[r] * kk[c] for c in range(dk)]
             for r in range(dk)]
        S = [[a * sum((S[i][r] * M[r][c] for r in range(dk)), Dual(0)) + b * vv[i] * kk[c]
              for c in range(dk)] for i in range(dv)]
        o = [F(ex["scale"]) * sum((S[i][j] * qq[j] for j in range(dk)), Dual(0))
             for i in range(dv)]
        os_.append(o)
        loss = loss + sum((o[i] * F(ex["dO"][t][0][i]) for i in range(dv)), Dual(0))
    hT = [[S[i][j] for i in range(dv)] for j in range(dk)]
    loss = loss + sum((hT[j][i] * F(ex["dHT"][0][0][j][i]) for j in range(dk) for i in range(dv)),
                      Dual(0))
    return os_, hT, loss


def _rel(a, b):
    a, b = np.asarray(a, float), np.asarray(b, float)
    return float(np.max(np.abs(a - b)) / max(1.0, np.max(np.abs(b))))


def test_golden_matches_exact_arithmetic():
    gold = json.load(open(GOLDEN))
    ex = gold["inputs"]
    o, hT, _ = _exact(ex)
    assert _rel(gold["o"], [[[float(x.a) for x in row]] for row in o]) < 1e-14
    assert _rel(gold["hT"], [[[[float(x.a) for x in r] for r in hT]]]) < 1e-14
    grads = {"q": "dq", "k": "dk", "v": "dv", "beta": "dbeta", "g": "dg", "h0": "dh0"}
    for name, gname in grads.items():
        ref = np.array(gold[gname], dtype=float)
        got = np.zeros_like(ref)
        for idx in np.ndindex(*ref.shape):
            _, _, loss = _exact(ex, (name, tuple(idx)))
            got[idx] = float(loss.b)
        assert _rel(ref, got) < 1e-13, name


def test_oracle_reproduces_golden():
    gold = json.load(open(GOLDEN))
    ex = gold["inputs"]
    arr = lambda n: np.array(ex[n], dtype=np.float64)
    g = arr("g_over_ln_half") * math.log(0.5)
    o, hT = oracle.gdn_fwd(arr("q"), arr("k"), arr("v"), g, arr("beta"), [0, 3], h0=arr("h0"),
                           scale=ex["scale"])
    assert _rel(o, gold["o"]) < 1e-15 and _rel(hT, gold["hT"]) < 1e-15
    gr = oracle.gdn_bwd(arr("q"), arr("k"), arr("v"), g, arr("beta"), [0, 3], arr("dO"),
                        h0=arr("h0"), dHT=arr("dHT"), scale=ex["scale"])
    for n in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        assert _rel(gr[n], gold[n]) < 1e-15, n
