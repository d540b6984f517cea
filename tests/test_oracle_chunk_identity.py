"""Pin: the oracle's token recurrence equals an independently derived fp64
chunkwise-parallel form for every chunk size, including C = 1 and C = T.

The chunk form (derived from the gated delta rule; the page "IsoExec: 切换
SkyRL 中的训练器-推理不匹配", section "Chunkwise-Parallel Recurrent (CPR)
Gated DeltaNet", names the chunkwise-parallel form without writing it out).
Within a chunk with start state H (d_k x d_v), gam = cumsum(g), G = exp(gam),
E[r, s] = exp(gam_r - gam_s):
    A     = strict_lower(diag(b) (K K^T * E))
    T     = (I + A)^-1
    U     = T diag(b) V,   W = T diag(b G) K
    Delta = U - W H
    O     = scale (diag(G) Q H + (Q K^T * E * lower) Delta)
    H'    = G_last H + (diag(E[last, :]) K)^T Delta
This is a different algorithm from the recurrence (a triangular solve per
chunk instead of T rank-1 updates), so agreement pins both.
"""
import numpy as np
import pytest


def chunk_form(q, k, v, g, beta, cu, h0, C, scale=1.0):
    n_tok, H, dk = q.shape
    dv = v.shape[2]
    o = np.zeros((n_tok, H, dv))
    hT = np.zeros((len(cu) - 1, H, dk, dv))
    for b in range(len(cu) - 1):
        for h in range(H):
            S = np.zeros((dk, dv)) if h0 is None else h0[b, h].copy()
            for c0 in range(cu[b], cu[b + 1], C):
                c1 = min(c0 + C, cu[b + 1])
                Q, K, V = q[c0:c1, h], k[c0:c1, h], v[c0:c1, h]
                gm = np.cumsum(g[c0:c1, h])
                G = np.exp(gm)
                E = np.exp(gm[:, None] - gm[None, :])
                bt = beta[c0:c1, h]
                n = c1 - c0
                A = np.tril(bt[:, None] * (K @ K.T) * E, -1)
                Tm = np.linalg.inv(np.eye(n) + A)
                U = Tm @ (bt[:, None] * V)
                W = Tm @ ((bt * G)[:, None] * K)
                D = U - W @ S
                P = np.tril((Q @ K.T) * E)
                o[c0:c1, h] = scale * (G[:, None] * (Q @ S) + P @ D)
                S = G[-1] * S + (E[-1][:, None] * K).T @ D
            hT[b, h] = S
    return o, hT


@pytest.mark.parametrize("C", [1, 4, 16, 64, 10_000])
def test_recurrence_equals_chunk_form(oracle_mod, C):
    rng = np.random.default_rng(11)
    lens = [70, 3, 129]
    H, dk, dv = 2, 8, 6
    N = sum(lens)
    q = rng.standard_normal((N, H, dk))
    k = rng.standard_normal((N, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    v = rng.standard_normal((N, H, dv))
    g = -rng.uniform(0.001, 0.1, (N, H))
    beta = 1 / (1 + np.exp(-rng.standard_normal((N, H))))
    h0 = 0.3 * rng.standard_normal((len(lens), H, dk, dv))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    o_r, h_r = oracle_mod.gdn_fwd(q, k, v, g, beta, cu, h0=h0, scale=0.9)
    o_c, h_c = chunk_form(q, k, v, g, beta, cu, h0, C, scale=0.9)
    err_o = np.max(np.abs(o_r - o_c)) / np.max(np.abs(o_r))
    err_h = np.max(np.abs(h_r - h_c)) / np.max(np.abs(h_r))
    assert err_o < 1e-11 and err_h < 1e-11, (err_o, err_h)
