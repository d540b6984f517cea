"""GPU parity at the benchmark workloads' full sizes, in the launch configuration
bench.py times (tensor-core contract, two d_v splits; the trainer as a training
forward plus the backward from its saved tiles).  The oracle computes sampled
(sequence, head) pairs one at a time; bit identity (decode vs prefill, each
varlen sequence alone vs packed) is checked on everything."""
import pytest
import torch

import infer_consistent_linear_gb300 as cpr
import oracle
from infer_consistent_linear_gb300.synth import make_inputs, varlen_lengths
from gpu_helpers import TOL_BF16, assert_bitwise, assert_close, require_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"
D = 128
GRADS = ("dq", "dk", "dv", "dg", "dbeta")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _contract():
    return cpr.default_contract(torch.bfloat16, D, dv_splits=2, operand_policy=cpr.CPR_POLICY_TC_BF16X3)


def _one(x, cu, b, h, with_grad=False):
    """Inputs of sequence b, head h alone (CPU tensors) for the oracle."""
    sl = slice(cu[b], cu[b + 1])
    pick = lambda t: None if t is None else t[sl, h:h + 1].contiguous()
    one = dict(q=pick(x.q), k=pick(x.k), v=pick(x.v), g=pick(x.g), beta=pick(x.beta),
               cu=torch.tensor([0, cu[b + 1] - cu[b]], dtype=torch.int32))
    if with_grad:
        one["dO"] = pick(x.dO)
    return one


def test_prefill_workload_sampled_heads():
    lens, H = [4096] * 4, 16
    x = make_inputs(lens, H, D, D, io_dtype=torch.bfloat16, seed=0)
    xd = x.to(DEV)
    o, fin = cpr.cpr_gdn_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, contract=_contract())
    torch.cuda.synchronize()
    assert cpr.get_device_error() == 0
    o, fin, cu = o.cpu(), fin.cpu(), x.cu_seqlens.tolist()
    for b, h in [(0, 0), (2, 7), (3, 15)]:
        one = _one(x, cu, b, h)
        o_ref, h_ref = oracle.gdn_fwd(one["q"], one["k"], one["v"], one["g"], one["beta"], one["cu"])
        assert_close(f"o[{b},{h}]", o[cu[b]:cu[b + 1], h:h + 1], o_ref, TOL_BF16)
        assert_close(f"final[{b},{h}]", fin[b:b + 1, h:h + 1], h_ref, TOL_BF16)


@pytest.mark.parametrize("with_states", [False, True])
def test_trainer_workload_sampled_heads(with_states):
    """The Trainer configuration as timed (h0 = 0, no dHT) and with an initial state and an
    upstream gradient of the final state, which the timed runs leave out."""
    lens, H = [4096] * 8, 16
    x = make_inputs(lens, H, D, D, io_dtype=torch.bfloat16, seed=0, with_grad=True,
                    h0_std=0.1 if with_states else 0.0)
    dHT = None
    if with_states:
        gen = torch.Generator().manual_seed(5)
        dHT = torch.randn(len(lens), H, D, D, generator=gen)
    xd = x.to(DEV)
    c = _contract()
    ws = torch.empty(cpr.workspace_bytes(c, cpr.CPR_OP_BWD, len(lens), sum(lens), H),
                     dtype=torch.uint8, device=DEV)
    o, fin = cpr.cpr_gdn_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, h0=xd.h0, contract=c,
                             workspace=ws, train=True)
    got = cpr.cpr_gdn_bwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, xd.dO, h0=xd.h0,
                          dHT=None if dHT is None else dHT.to(DEV), contract=c, workspace=ws, saved=True)
    torch.cuda.synchronize()
    assert cpr.get_device_error() == 0
    got = {k: v.cpu() for k, v in got.items()}
    o, fin, cu = o.cpu(), fin.cpu(), x.cu_seqlens.tolist()
    for b, h in [(1, 3), (6, 12)]:
        one = _one(x, cu, b, h, with_grad=True)
        h0 = None if x.h0 is None else x.h0[b:b + 1, h:h + 1].contiguous()
        dht = None if dHT is None else dHT[b:b + 1, h:h + 1].contiguous()
        o_ref, h_ref = oracle.gdn_fwd(one["q"], one["k"], one["v"], one["g"], one["beta"], one["cu"], h0=h0)
        ref = oracle.gdn_bwd(one["q"], one["k"], one["v"], one["g"], one["beta"], one["cu"], one["dO"],
                             h0=h0, dHT=dht)
        sl = slice(cu[b], cu[b + 1])
        assert_close(f"o[{b},{h}]", o[sl, h:h + 1], o_ref, TOL_BF16)
        assert_close(f"final[{b},{h}]", fin[b:b + 1, h:h + 1], h_ref, TOL_BF16)
        for n in GRADS:
            assert_close(f"{n}[{b},{h}]", got[n][sl, h:h + 1], ref[n], TOL_BF16)
        assert_close(f"dh0[{b},{h}]", got["dh0"][b:b + 1, h:h + 1], ref["dh0"], TOL_BF16)


def test_decode_workload_bitwise_and_sampled_heads():
    n_seq, H, L, steps = 64, 32, 2048, 512
    x = make_inputs([L + steps] * n_seq, H, D, D, io_dtype=torch.bfloat16, seed=0)
    xd = x.to(DEV)
    c = _contract()
    o_full, _ = cpr.cpr_gdn_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, contract=c)
    cu = x.cu_seqlens.tolist()
    sel = torch.cat([torch.arange(cu[b], cu[b] + L) for b in range(n_seq)]).to(DEV)
    cu_pre = torch.arange(0, (n_seq + 1) * L, L, dtype=torch.int32, device=DEV)
    o_pre, _, cache = cpr.cpr_gdn_prefill(xd.q[sel], xd.k[sel], xd.v[sel], xd.g[sel], xd.beta[sel],
                                          cu_pre, contract=c, want_final=False)
    assert_bitwise("prefill part", o_pre, o_full[sel])
    base = torch.tensor(cu[:-1], device=DEV) + L
    for t in range(steps):
        idx = base + t
        ot = cpr.cpr_gdn_decode_step(xd.q[idx], xd.k[idx], xd.v[idx], xd.g[idx], xd.beta[idx],
                                     cache, contract=c)
        assert_bitwise(f"decode step {t}", ot, o_full[idx])
        if (t + 1) % 64 == 0:  # the committed chunk-boundary states
            n_done = L + t + 1
            keep = torch.cat([torch.arange(cu[b], cu[b] + n_done) for b in range(n_seq)]).to(DEV)
            cub = torch.arange(0, (n_seq + 1) * n_done, n_done, dtype=torch.int32, device=DEV)
            _, fin = cpr.cpr_gdn_fwd(xd.q[keep], xd.k[keep], xd.v[keep], xd.g[keep], xd.beta[keep],
                                     cub, contract=c)
            assert_bitwise(f"states after {n_done} tokens", cache.state(), fin)
    torch.cuda.synchronize()
    assert cpr.get_device_error() == 0
    o_full = o_full.cpu()
    for b, h in [(0, 0), (41, 29)]:
        one = _one(x, cu, b, h)
        o_ref, _ = oracle.gdn_fwd(one["q"], one["k"], one["v"], one["g"], one["beta"], one["cu"])
        assert_close(f"o[{b},{h}] (decode = prefill bits)", o_full[cu[b]:cu[b + 1], h:h + 1], o_ref, TOL_BF16)


def test_varlen_workload_batch_invariance_and_sampled_heads():
    lens, H = varlen_lengths(48, 128, 8192, seed=0), 16
    x = make_inputs(lens, H, D, D, io_dtype=torch.bfloat16, seed=0, with_grad=True)
    xd = x.to(DEV)
    c = _contract()
    n_tok = sum(lens)
    ws = torch.empty(cpr.workspace_bytes(c, cpr.CPR_OP_BWD, len(lens), n_tok, H), dtype=torch.uint8,
                     device=DEV)
    o, fin = cpr.cpr_gdn_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, contract=c,
                             workspace=ws, train=True)
    got = cpr.cpr_gdn_bwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, xd.dO, contract=c,
                          workspace=ws, saved=True)
    torch.cuda.synchronize()
    assert cpr.get_device_error() == 0
    cu = x.cu_seqlens.tolist()
    order = sorted(range(len(lens)), key=lambda i: lens[i])
    for b in (order[0], order[len(order) // 2], order[-1]):   # alone at B = 1: same bits
        sl = slice(cu[b], cu[b + 1])
        cub = torch.tensor([0, lens[b]], dtype=torch.int32, device=DEV)
        o1, f1 = cpr.cpr_gdn_fwd(xd.q[sl], xd.k[sl], xd.v[sl], xd.g[sl], xd.beta[sl], cub, contract=c)
        g1 = cpr.cpr_gdn_bwd(xd.q[sl], xd.k[sl], xd.v[sl], xd.g[sl], xd.beta[sl], cub, xd.dO[sl],
                             contract=c)
        assert_bitwise(f"o[seq {b}]", o1, o[sl])
        assert_bitwise(f"final[seq {b}]", f1, fin[b:b + 1])
        for n in GRADS:
            assert_bitwise(f"{n}[seq {b}]", g1[n], got[n][sl])
        assert_bitwise(f"dh0[seq {b}]", g1["dh0"], got["dh0"][b:b + 1])
    got = {k: v.cpu() for k, v in got.items()}
    o = o.cpu()
    for b, h in [(order[0], 5), (order[-1], 11)]:
        one = _one(x, cu, b, h, with_grad=True)
        o_ref, _ = oracle.gdn_fwd(one["q"], one["k"], one["v"], one["g"], one["beta"], one["cu"])
        ref = oracle.gdn_bwd(one["q"], one["k"], one["v"], one["g"], one["beta"], one["cu"], one["dO"])
        sl = slice(cu[b], cu[b + 1])
        assert_close(f"o[{b},{h}]", o[sl, h:h + 1], o_ref, TOL_BF16)
        for n in GRADS:
            assert_close(f"{n}[{b},{h}]", got[n][sl, h:h + 1], ref[n], TOL_BF16)
