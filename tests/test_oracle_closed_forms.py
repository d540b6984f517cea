"""Pins of the fp64 oracle against closed forms the gated delta rule fixes.

The rule (page "IsoExec: 切换 SkyRL 中的训练器-推理不匹配", section
"Chunkwise-Parallel Recurrent (CPR) Gated DeltaNet"; Gated DeltaNet):
    S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T,  o_t = S_t q_t.
H = S^T is the stored state.  Shapes use d_k != d_v so that a transposed
operand cannot pass.
"""
import numpy as np
import pytest

RTOL = 1e-12


def _rand(rng, T, H, dk, dv, unit_k=True):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    if unit_k:
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    g = -rng.uniform(0.001, 0.1, (T, H))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    return q, k, v, g, beta


def _close(a, b, tol=RTOL):
    scale = max(1.0, float(np.max(np.abs(b))))
    np.testing.assert_allclose(a, b, rtol=0, atol=tol * scale)


def test_beta0_alpha1_keeps_state(oracle_mod):
    rng = np.random.default_rng(1)
    T, H, dk, dv = 9, 2, 5, 3
    q, k, v, g, beta = _rand(rng, T, H, dk, dv)
    g[:] = 0.0
    beta[:] = 0.0
    h0 = rng.standard_normal((1, H, dk, dv))
    o, hT = oracle_mod.gdn_fwd(q, k, v, g, beta, [0, T], h0=h0, scale=0.7)
    # o_t = S_0 (0.7 q_t) = 0.7 * h0^T q_t
    want = 0.7 * np.einsum("thk,hkv->thv", q, h0[0])
    _close(o, want)
    _close(hT, h0)


def test_alpha0_resets_state(oracle_mod):
    rng = np.random.default_rng(2)
    T, H, dk, dv = 6, 2, 4, 7
    q, k, v, g, beta = _rand(rng, T, H, dk, dv, unit_k=False)
    g[:] = -1e4          # exp(-1e4) == 0.0 in fp64
    h0 = rng.standard_normal((1, H, dk, dv))
    o, hT = oracle_mod.gdn_fwd(q, k, v, g, beta, [0, T], h0=h0)
    # S_t = b_t v_t k_t^T  =>  o_t = b_t v_t (k_t . q_t)
    want = beta[..., None] * v * np.einsum("thk,thk->th", k, q)[..., None]
    _close(o, want)
    want_h = beta[-1][:, None, None] * np.einsum("hk,hv->hkv", k[-1], v[-1])
    _close(hT[0], want_h)


def test_single_token_from_zero_state(oracle_mod):
    rng = np.random.default_rng(3)
    H, dk, dv = 3, 6, 4
    q, k, v, g, beta = _rand(rng, 1, H, dk, dv, unit_k=False)
    o, hT = oracle_mod.gdn_fwd(q, k, v, g, beta, [0, 1])
    # S_1 = a S_0(...) + b v k^T with S_0 = 0  =>  o = b v (k . q)
    want = beta[0][:, None] * v[0] * np.einsum("hk,hk->h", k[0], q[0])[:, None]
    _close(o[0], want)
    _close(hT[0], beta[0][:, None, None] * np.einsum("hk,hv->hkv", k[0], v[0]))


def test_delta_rule_invariant_unit_keys(oracle_mod):
    """With |k_t| = 1:  S_t k_t = a_t (1 - b_t) S_{t-1} k_t + b_t v_t,
    and with a = b = 1 the new state maps k_t exactly to v_t."""
    rng = np.random.default_rng(4)
    T, H, dk, dv = 12, 2, 5, 3
    q, k, v, g, beta = _rand(rng, T, H, dk, dv, unit_k=True)
    h0 = rng.standard_normal((1, H, dk, dv))
    for t in range(1, T + 1):
        _, Hp = oracle_mod.gdn_fwd(q[:t - 1], k[:t - 1], v[:t - 1], g[:t - 1], beta[:t - 1],
                                   [0, t - 1], h0=h0)
        _, Hc = oracle_mod.gdn_fwd(q[:t], k[:t], v[:t], g[:t], beta[:t], [0, t], h0=h0)
        kt, vt, a, b = k[t - 1], v[t - 1], np.exp(g[t - 1]), beta[t - 1]
        lhs = np.einsum("hkv,hk->hv", Hc[0], kt)          # S_t k_t
        prev = np.einsum("hkv,hk->hv", Hp[0], kt)         # S_{t-1} k_t
        _close(lhs, (a * (1 - b))[:, None] * prev + b[:, None] * vt)
    g1 = np.zeros_like(g)
    b1 = np.ones_like(beta)
    _, Hc = oracle_mod.gdn_fwd(q, k, v, g1, b1, [0, T], h0=h0)
    _close(np.einsum("hkv,hk->hv", Hc[0], k[-1]), v[-1])


def test_linearity_in_v_and_h0(oracle_mod):
    rng = np.random.default_rng(5)
    T, H, dk, dv = 10, 2, 4, 6
    q, k, v, g, beta = _rand(rng, T, H, dk, dv)
    h0 = rng.standard_normal((1, H, dk, dv))
    o1, h1 = oracle_mod.gdn_fwd(q, k, v, g, beta, [0, T], h0=h0)
    o2, h2 = oracle_mod.gdn_fwd(q, k, -2.5 * v, g, beta, [0, T], h0=-2.5 * h0)
    _close(o2, -2.5 * o1)
    _close(h2, -2.5 * h1)
    # superposition: (v, h0) = (v, 0) + (0, h0)
    oa, _ = oracle_mod.gdn_fwd(q, k, v, g, beta, [0, T])
    ob, _ = oracle_mod.gdn_fwd(q, k, 0 * v, g, beta, [0, T], h0=h0)
    _close(o1, oa + ob)


def test_orthogonal_keys_reduce_to_gated_linear_attention(oracle_mod):
    """Mutually orthogonal keys switch off the delta correction between
    tokens, leaving causal gated linear attention, which is brute-forced here:
        o_t = G_t S_0 q_t + sum_{s<=t} exp(gam_t - gam_s) b_s (k_s . q_t) v_s
    (S_0 k_s = 0 is arranged by choosing h0 orthogonal to every key)."""
    rng = np.random.default_rng(6)
    T, H, dk, dv = 6, 2, 8, 5
    q = rng.standard_normal((T, H, dk))
    v = rng.standard_normal((T, H, dv))
    g = -rng.uniform(0.001, 0.5, (T, H))
    beta = rng.uniform(0.1, 0.9, (T, H))
    k = np.zeros((T, H, dk))
    h0 = np.zeros((1, H, dk, dv))
    for h in range(H):
        Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
        k[:, h, :] = Qm[:T].copy() * rng.uniform(0.5, 2.0, (T, 1))
        # h0 rows lie in the span of the unused directions
        rest = Qm[T:]
        h0[0, h] = rest.T @ rng.standard_normal((dk - T, dv))
    o, _ = oracle_mod.gdn_fwd(q, k, v, g, beta, [0, T], h0=h0)
    gam = np.cumsum(g, axis=0)
    want = np.zeros_like(o)
    for h in range(H):
        for t in range(T):
            acc = np.exp(gam[t, h]) * (h0[0, h].T @ q[t, h])
            for s in range(t + 1):
                acc = acc + np.exp(gam[t, h] - gam[s, h]) * beta[s, h] * (k[s, h] @ q[t, h]) * v[s, h]
            want[t, h] = acc
    _close(o, want, 1e-11)


def test_packed_sequences_are_independent(oracle_mod):
    rng = np.random.default_rng(7)
    lens = [5, 1, 0, 9]
    H, dk, dv = 2, 4, 3
    N = sum(lens)
    q, k, v, g, beta = _rand(rng, N, H, dk, dv)
    h0 = rng.standard_normal((len(lens), H, dk, dv))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    o, hT = oracle_mod.gdn_fwd(q, k, v, g, beta, cu, h0=h0)
    for b, (a, e) in enumerate(zip(cu[:-1], cu[1:])):
        ob, hb = oracle_mod.gdn_fwd(q[a:e], k[a:e], v[a:e], g[a:e], beta[a:e], [0, e - a],
                                    h0=h0[b:b + 1])
        np.testing.assert_array_equal(o[a:e], ob)
        np.testing.assert_array_equal(hT[b], hb[0])


def test_bad_cu_seqlens_rejected(oracle_mod):
    rng = np.random.default_rng(8)
    q, k, v, g, beta = _rand(rng, 4, 1, 2, 2)
    with pytest.raises((ValueError, AssertionError)):
        oracle_mod.gdn_fwd(q, k, v, g, beta, [0, 3, 2, 4])
