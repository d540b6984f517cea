"""Pins for the projection oracle (oracle.gemm): a brute-force triple loop on small
shapes and two special cases with exact answers."""
import numpy as np

import oracle


def _brute(x, w):
    m, k = x.shape
    n = w.shape[1]
    y = np.zeros((m, n))
    for i in range(m):
        for j in range(n):
            acc = 0.0
            for t in range(k):
                acc += float(x[i, t]) * float(w[t, j])
            y[i, j] = acc
    return y


def test_gemm_oracle_brute_force():
    rng = np.random.default_rng(11)
    for m, k, n in [(1, 1, 1), (3, 5, 2), (7, 16, 9)]:
        x = rng.standard_normal((m, k)).astype(np.float32)
        w = rng.standard_normal((k, n)).astype(np.float32)
        np.testing.assert_allclose(oracle.gemm(x, w), _brute(x, w), rtol=1e-12, atol=1e-12)


def test_gemm_oracle_identity_and_permutation():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((6, 8)).astype(np.float32)
    assert np.array_equal(oracle.gemm(x, np.eye(8, dtype=np.float32)), x.astype(np.float64))
    perm = rng.permutation(8)
    p = np.eye(8, dtype=np.float32)[:, perm]          # column j of x P is column perm[j] of x
    assert np.array_equal(oracle.gemm(x, p), x[:, perm].astype(np.float64))
