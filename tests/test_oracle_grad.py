"""Pins of the oracle's hand-derived reverse recurrence (gradients).

Loss L = sum(dO * o) + sum(dHT * hT) with o, hT from the fp64 forward.
  * central finite differences of the oracle's own forward, every input
    element including h0 (h = 1e-6, fp64);
  * single-token closed forms from S_0 = 0:
        dq = b (v.dO) k,  dk = b (v.dO) q,  dv = b (k.q) dO,
        db = (k.q)(v.dO), dg = 0;
  * with b = 0 (state only decays):  dh0 = sum_t G_t q_t dO_t^T;
  * the VJP/JVP dot-product identity on a random direction.
The forward itself is pinned in test_oracle_closed_forms.py and
test_oracle_chunk_identity.py, so agreement with its finite differences pins
the backward.
"""
import numpy as np
import pytest


def _inputs(rng, lens, H, dk, dv):
    N = sum(lens)
    q = rng.standard_normal((N, H, dk))
    k = rng.standard_normal((N, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((N, H, dv))
    g = -rng.uniform(0.001, 0.3, (N, H))
    beta = 1 / (1 + np.exp(-rng.standard_normal((N, H))))
    h0 = 0.5 * rng.standard_normal((len(lens), H, dk, dv))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0), cu


def _loss(oracle_mod, x, cu, dO, dHT, scale):
    o, hT = oracle_mod.gdn_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], cu, h0=x["h0"],
                               scale=scale)
    return float(np.sum(o * dO) + np.sum(hT * dHT))


@pytest.mark.parametrize("seg", [1, 3, 64])
def test_finite_differences_all_inputs(oracle_mod, seg):
    rng = np.random.default_rng(21)
    lens = [7, 4]
    H, dk, dv = 2, 3, 4
    x, cu = _inputs(rng, lens, H, dk, dv)
    dO = rng.standard_normal((sum(lens), H, dv))
    dHT = rng.standard_normal((len(lens), H, dk, dv))
    scale = 0.8
    grads = oracle_mod.gdn_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], cu, dO, h0=x["h0"],
                               dHT=dHT, scale=scale, seg=seg)
    names = dict(q="dq", k="dk", v="dv", g="dg", beta="dbeta", h0="dh0")
    h = 1e-6
    for name, gname in names.items():
        arr = x[name]
        fd = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = arr[idx]
            arr[idx] = old + h
            lp = _loss(oracle_mod, x, cu, dO, dHT, scale)
            arr[idx] = old - h
            lm = _loss(oracle_mod, x, cu, dO, dHT, scale)
            arr[idx] = old
            fd[idx] = (lp - lm) / (2 * h)
        got = grads[gname]
        err = np.max(np.abs(got - fd)) / max(1e-3, np.max(np.abs(fd)))
        assert err < 1e-6, (name, err)


def test_single_token_closed_form(oracle_mod):
    rng = np.random.default_rng(22)
    H, dk, dv = 3, 5, 4
    q = rng.standard_normal((1, H, dk))
    k = rng.standard_normal((1, H, dk))
    v = rng.standard_normal((1, H, dv))
    g = -rng.uniform(0.01, 0.5, (1, H))
    beta = rng.uniform(0.1, 0.9, (1, H))
    dO = rng.standard_normal((1, H, dv))
    r = oracle_mod.gdn_bwd(q, k, v, g, beta, [0, 1], dO)
    kq = np.einsum("hk,hk->h", k[0], q[0])
    vd = np.einsum("hv,hv->h", v[0], dO[0])
    b = beta[0]
    np.testing.assert_allclose(r["dq"][0], (b * vd)[:, None] * k[0], atol=1e-13)
    np.testing.assert_allclose(r["dk"][0], (b * vd)[:, None] * q[0], atol=1e-13)
    np.testing.assert_allclose(r["dv"][0], (b * kq)[:, None] * dO[0], atol=1e-13)
    np.testing.assert_allclose(r["dbeta"][0], kq * vd, atol=1e-13)
    np.testing.assert_allclose(r["dg"][0], 0.0, atol=1e-13)


def test_beta_zero_dh0_closed_form(oracle_mod):
    rng = np.random.default_rng(23)
    T, H, dk, dv = 9, 2, 4, 3
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    v = rng.standard_normal((T, H, dv))
    g = -rng.uniform(0.01, 0.2, (T, H))
    beta = np.zeros((T, H))
    dO = rng.standard_normal((T, H, dv))
    h0 = rng.standard_normal((1, H, dk, dv))
    r = oracle_mod.gdn_bwd(q, k, v, g, beta, [0, T], dO, h0=h0)
    G = np.exp(np.cumsum(g, axis=0))
    want = np.einsum("th,thk,thv->hkv", G, q, dO)
    np.testing.assert_allclose(r["dh0"][0], want, atol=1e-12)
    # and o_t = G_t h0^T q_t, so dg_t = sum_{r>=t} G_r q_r^T h0 dO_r
    per_tok = G * np.einsum("thk,hkv,thv->th", q, h0[0], dO)
    want_dg = np.cumsum(per_tok[::-1], axis=0)[::-1]
    np.testing.assert_allclose(r["dg"], want_dg, atol=1e-12)


def test_vjp_jvp_dot_product(oracle_mod):
    """<dL/dx, u> equals the directional derivative of L along u."""
    rng = np.random.default_rng(24)
    lens = [13]
    H, dk, dv = 1, 6, 5
    x, cu = _inputs(rng, lens, H, dk, dv)
    dO = rng.standard_normal((13, H, dv))
    dHT = rng.standard_normal((1, H, dk, dv))
    r = oracle_mod.gdn_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], cu, dO, h0=x["h0"],
                           dHT=dHT)
    u = {n: rng.standard_normal(a.shape) for n, a in x.items()}
    gmap = dict(q="dq", k="dk", v="dv", g="dg", beta="dbeta", h0="dh0")
    lhs = sum(float(np.sum(r[gmap[n]] * u[n])) for n in x)
    h = 1e-6
    xp = {n: x[n] + h * u[n] for n in x}
    xm = {n: x[n] - h * u[n] for n in x}
    rhs = (_loss(oracle_mod, xp, cu, dO, dHT, 1.0) - _loss(oracle_mod, xm, cu, dO, dHT, 1.0)) / (2 * h)
    assert abs(lhs - rhs) <= 1e-7 * max(1.0, abs(rhs))
