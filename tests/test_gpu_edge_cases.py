"""GPU parity on the gated delta rule's own edge cases, where the chunk form is
fragile and random inputs do not reach:

* beta = 0, g = 0: the state is left unchanged (alpha = 1) and o_t = S_0 q_t;
* g = -1e4 on tokens in the middle of chunks: alpha ~ 0 resets the state there,
  and every later decay inside the chunk is an exponential of a difference of two
  large in-chunk prefixes;
* beta = 1, g = 0 on unit keys: the delta rule writes v_t exactly (S_t k_t = v_t);
* strong gates g ~ -U(0.5, 5): exp(gam_r) underflows inside one chunk while
  exp(gam_r - gam_s) for nearby rows does not;
* beta alternating 0 and 1 row by row.

(Page "IsoExec: 切换 SkyRL 中的训练器-推理不匹配", section "Chunkwise-Parallel
Recurrent (CPR) Gated DeltaNet": the gated delta rule; the closed forms follow from
its definition.)  Each case runs under the tensor-core contract (bf16, d = 128) and
the SIMT fp32 contract (d = 64): the forward and the backward against the fp64
oracle element by element, and decode steps that continue a prefill bit for bit."""
import pytest
import torch

import infer_consistent_linear_gb300 as cpr
import oracle
from infer_consistent_linear_gb300.synth import make_inputs
from gpu_helpers import TOL_BF16, TOL_F32, assert_bitwise, assert_close, require_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"

CASES = ("beta0_g0", "reset", "beta1_g0", "strong", "beta01")
CONTRACTS = {
    "tc": dict(io=torch.bfloat16, d=128, tol=TOL_BF16,
               kw=dict(operand_policy=cpr.CPR_POLICY_TC_BF16X3, dv_splits=2)),
    "simt_f32": dict(io=torch.float32, d=64, tol=TOL_F32,
                     kw=dict(operand_policy=cpr.CPR_POLICY_SIMT_F32, dv_splits=2)),
}
GRADS = ("dq", "dk", "dv", "dg", "dbeta", "dh0")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _positions(cu):
    """Sequence-relative position of every token."""
    pos = torch.empty(int(cu[-1]), dtype=torch.int64)
    for b in range(len(cu) - 1):
        pos[cu[b]:cu[b + 1]] = torch.arange(cu[b + 1] - cu[b])
    return pos


def edge_inputs(case, lens, H, d, io, with_grad=False, seed=21):
    """Seeded inputs of the usual recipe with the gate / beta pattern of `case`."""
    x = make_inputs(lens, H, d, d, io_dtype=io, seed=seed, h0_std=0.1, with_grad=with_grad,
                    g_range=(0.5, 5.0) if case == "strong" else (0.001, 0.1))
    pos = _positions(x.cu_seqlens.tolist())
    if case == "beta0_g0":
        x.g.zero_()
        x.beta.zero_()
    elif case == "reset":
        # positions 30, 67, 104, ... : mid-chunk, first rows and a chunk's last row
        hit = (pos % 37 == 30)[:, None].expand_as(x.g)
        x.g[hit] = -1e4
    elif case == "beta1_g0":
        x.g.zero_()
        x.beta.fill_(1.0)
    elif case == "beta01":
        x.beta.copy_((pos % 2).to(torch.float32)[:, None].expand_as(x.beta))
    return x


def _contract(name):
    p = CONTRACTS[name]
    return p, cpr.default_contract(p["io"], p["d"], **p["kw"])


@pytest.mark.parametrize("cname", list(CONTRACTS))
@pytest.mark.parametrize("case", CASES)
def test_edge_forward_parity(case, cname):
    p, c = _contract(cname)
    lens, H = [200, 130, 64, 1], 2
    x = edge_inputs(case, lens, H, p["d"], p["io"])
    xd = x.to(DEV)
    o, fin = cpr.cpr_gdn_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, h0=xd.h0, contract=c)
    torch.cuda.synchronize()
    assert cpr.get_device_error() == 0
    o_ref, h_ref = oracle.gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, h0=x.h0)
    assert_close("o", o, o_ref, p["tol"])
    assert_close("final_state", fin, h_ref, p["tol"])
    if case == "beta0_g0":
        # alpha = 1, beta = 0: every update is the identity, exactly
        assert_bitwise("final state = h0", fin, xd.h0)
    if case == "beta1_g0":
        # beta = alpha = 1, unit keys: S_T k_T = v_T for each sequence's last token
        cu = x.cu_seqlens.tolist()
        for b in range(len(lens)):
            t = cu[b + 1] - 1
            Sk = torch.einsum("hdj,hd->hj", fin[b].double().cpu(), x.k[t].double())
            assert_close(f"S k = v (seq {b})", Sk, x.v[t].double(), p["tol"])


@pytest.mark.parametrize("cname", list(CONTRACTS))
@pytest.mark.parametrize("case", CASES)
def test_edge_decode_continues_prefill(case, cname):
    """Prefill of ragged lengths, then 70 decode steps (past a chunk boundary); every
    step's output equals the one-shot forward's bit for bit, and that forward is
    within tolerance of the oracle."""
    p, c = _contract(cname)
    pre, steps, H = [100, 64, 1, 30], 70, 2
    full = [L + steps for L in pre]
    x = edge_inputs(case, full, H, p["d"], p["io"], seed=22)
    xd = x.to(DEV)
    o_full, fin_full = cpr.cpr_gdn_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, h0=xd.h0,
                                       contract=c)
    cu = x.cu_seqlens.tolist()
    sel = torch.cat([torch.arange(cu[b], cu[b] + pre[b]) for b in range(len(pre))]).to(DEV)
    cu_pre = torch.tensor([0] + torch.cumsum(torch.tensor(pre), 0).tolist(), dtype=torch.int32,
                          device=DEV)
    o_pre, _, cache = cpr.cpr_gdn_prefill(xd.q[sel], xd.k[sel], xd.v[sel], xd.g[sel], xd.beta[sel],
                                          cu_pre, h0=xd.h0, contract=c)
    assert_bitwise("prefill part", o_pre, o_full[sel])
    for t in range(steps):
        idx = torch.tensor([cu[b] + pre[b] + t for b in range(len(pre))], device=DEV)
        ot = cpr.cpr_gdn_decode_step(xd.q[idx], xd.k[idx], xd.v[idx], xd.g[idx], xd.beta[idx],
                                     cache, contract=c)
        assert_bitwise(f"decode step {t}", ot, o_full[idx])
    torch.cuda.synchronize()
    assert cpr.get_device_error() == 0
    o_ref, _ = oracle.gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, h0=x.h0)
    assert_close("o vs oracle", o_full, o_ref, p["tol"])


@pytest.mark.parametrize("cname", list(CONTRACTS))
@pytest.mark.parametrize("case", CASES)
def test_edge_backward_parity(case, cname):
    p, c = _contract(cname)
    lens, H = [150, 64, 1, 100], 2
    x = edge_inputs(case, lens, H, p["d"], p["io"], with_grad=True, seed=23)
    gen = torch.Generator().manual_seed(24)
    dHT = torch.randn(len(lens), H, p["d"], p["d"], generator=gen)
    xd = x.to(DEV)
    got = cpr.cpr_gdn_bwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, xd.dO, h0=xd.h0,
                          dHT=dHT.to(DEV), contract=c)
    torch.cuda.synchronize()
    assert cpr.get_device_error() == 0
    ref = oracle.gdn_bwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, x.dO, h0=x.h0, dHT=dHT)
    for n in GRADS:
        assert_close(n, got[n], ref[n], p["tol"])
