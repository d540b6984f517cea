"""GPU bit-identity across execution cases under one contract: prefill vs
decode (with the state resynchronised every C tokens), chunk-aligned splits
of a sequence, batch composition, d_v split count, and run-to-run.  Also the
device-side error paths (bad cu_seqlens, a cache made under another
contract).  Source of the requirement: page "IsoExec: 切换 SkyRL 中的训练器-
推理不匹配", CPR table row "Bitwise Exact"."""
import pytest
import torch

import infer_consistent_linear_gb300 as cpr
import oracle
from infer_consistent_linear_gb300.synth import make_inputs
from gpu_helpers import TOL_BF16, TOL_F32, assert_bitwise, assert_close, require_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _decode_vs_prefill(io, d, pre_lens, n_steps, H, check_oracle_tol=None, **contract_overrides):
    n_seq = len(pre_lens)
    full_lens = [L + n_steps for L in pre_lens]
    x = make_inputs(full_lens, H, d, d, io_dtype=io, seed=7, h0_std=0.1).to(DEV)
    c = cpr.simt_contract(io, d, **contract_overrides)
    o_full, _ = cpr.cpr_gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, h0=x.h0, contract=c)
    cu = x.cu_seqlens.tolist()
    sel = torch.cat([torch.arange(cu[b], cu[b] + pre_lens[b]) for b in range(n_seq)]).to(DEV)
    cu_pre = torch.tensor([0] + torch.cumsum(torch.tensor(pre_lens), 0).tolist(), dtype=torch.int32,
                          device=DEV)
    o_pre, _, cache = cpr.cpr_gdn_prefill(x.q[sel], x.k[sel], x.v[sel], x.g[sel], x.beta[sel],
                                          cu_pre, h0=x.h0, contract=c)
    assert_bitwise("prefill part", o_pre, o_full[sel])
    for t in range(n_steps):
        idx = torch.tensor([cu[b] + pre_lens[b] + t for b in range(n_seq)], device=DEV)
        ot = cpr.cpr_gdn_decode_step(x.q[idx], x.k[idx], x.v[idx], x.g[idx], x.beta[idx], cache,
                                     contract=c)
        assert_bitwise(f"decode step {t}", ot, o_full[idx])
        for b in range(n_seq):  # committed states equal a prefill's final state
            n_done = pre_lens[b] + t + 1
            if n_done % 64 == 0:
                cub = torch.tensor([0, n_done], dtype=torch.int32, device=DEV)
                sl = slice(cu[b], cu[b] + n_done)
                _, fin = cpr.cpr_gdn_fwd(x.q[sl], x.k[sl], x.v[sl], x.g[sl], x.beta[sl], cub,
                                         h0=x.h0[b:b + 1], contract=c)
                assert_bitwise(f"state seq {b} at {n_done}", cache.state()[b:b + 1], fin)
    torch.cuda.synchronize()
    assert cpr.get_device_error() == 0
    if check_oracle_tol:
        xc = make_inputs(full_lens, H, d, d, io_dtype=io, seed=7, h0_std=0.1)
        o_ref, _ = oracle.gdn_fwd(xc.q, xc.k, xc.v, xc.g, xc.beta, xc.cu_seqlens, h0=xc.h0)
        assert_close("o (decode path) vs oracle", o_full, o_ref, check_oracle_tol)


def test_tiny_config_prefill_equals_256_decode_steps():
    # fp32, B=1, H=2, T=256, d=64: decode from an empty prefill
    _decode_vs_prefill(torch.float32, 64, [0], 256, 2, check_oracle_tol=TOL_F32)


def test_decode_bf16_ragged_prefills():
    _decode_vs_prefill(torch.bfloat16, 128, [100, 64, 0, 1, 63], 70, 2, check_oracle_tol=TOL_BF16)


def test_decode_bf16_d64():
    _decode_vs_prefill(torch.bfloat16, 64, [30, 128], 40, 3)


def test_chunk_aligned_split():
    c = cpr.simt_contract(torch.bfloat16, 128)
    x = make_inputs([300], 2, 128, 128, io_dtype=torch.bfloat16, seed=2, h0_std=0.1).to(DEV)
    o_all, fin_all = cpr.cpr_gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, h0=x.h0, contract=c)
    for T1 in (64, 128, 256):
        cu1 = torch.tensor([0, T1], dtype=torch.int32, device=DEV)
        cu2 = torch.tensor([0, 300 - T1], dtype=torch.int32, device=DEV)
        o1, f1, cache = cpr.cpr_gdn_prefill(x.q[:T1], x.k[:T1], x.v[:T1], x.g[:T1], x.beta[:T1],
                                            cu1, h0=x.h0, contract=c)
        assert torch.equal(cache.pos().cpu(), torch.tensor([0], dtype=torch.int32))
        assert_bitwise("cache state == final", cache.state(), f1)
        o2, f2 = cpr.cpr_gdn_fwd(x.q[T1:], x.k[T1:], x.v[T1:], x.g[T1:], x.beta[T1:], cu2, h0=f1,
                                 contract=c)
        assert_bitwise(f"o first part T1={T1}", o1, o_all[:T1])
        assert_bitwise(f"o second part T1={T1}", o2, o_all[T1:])
        assert_bitwise(f"final T1={T1}", f2, fin_all)


def test_batch_invariance_fwd_bwd():
    lens = [77, 200, 1, 0, 128, 64]
    H, d = 2, 128
    c = cpr.simt_contract(torch.bfloat16, d)
    x = make_inputs(lens, H, d, d, io_dtype=torch.bfloat16, seed=11, h0_std=0.1,
                    with_grad=True).to(DEV)
    o, fin = cpr.cpr_gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, h0=x.h0, contract=c)
    gr = cpr.cpr_gdn_bwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, x.dO, h0=x.h0, contract=c)
    cu = x.cu_seqlens.tolist()
    for b, L in enumerate(lens):
        sl = slice(cu[b], cu[b + 1])
        cub = torch.tensor([0, L], dtype=torch.int32, device=DEV)
        h0b = x.h0[b:b + 1].contiguous()
        ob, fb = cpr.cpr_gdn_fwd(x.q[sl], x.k[sl], x.v[sl], x.g[sl], x.beta[sl], cub, h0=h0b,
                                 contract=c)
        gb = cpr.cpr_gdn_bwd(x.q[sl], x.k[sl], x.v[sl], x.g[sl], x.beta[sl], cub,
                             x.dO[sl].contiguous(), h0=h0b, contract=c)
        assert_bitwise(f"o seq {b}", ob, o[sl])
        assert_bitwise(f"final seq {b}", fb, fin[b:b + 1])
        for n in ("dq", "dk", "dv", "dg", "dbeta"):
            assert_bitwise(f"{n} seq {b}", gb[n], gr[n][sl])
        assert_bitwise(f"dh0 seq {b}", gb["dh0"], gr["dh0"][b:b + 1])


def test_dv_split_count_does_not_change_bits():
    x = make_inputs([150, 33], 2, 128, 128, io_dtype=torch.bfloat16, seed=12, h0_std=0.1).to(DEV)
    outs = []
    for s in (1, 2, 4):
        c = cpr.simt_contract(torch.bfloat16, 128, dv_splits=s)
        outs.append(cpr.cpr_gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, h0=x.h0, contract=c))
    for o, f in outs[1:]:
        assert_bitwise("o", o, outs[0][0])
        assert_bitwise("final", f, outs[0][1])


def test_run_to_run_determinism():
    c = cpr.simt_contract(torch.bfloat16, 128)
    x = make_inputs([333, 64], 2, 128, 128, io_dtype=torch.bfloat16, seed=13, h0_std=0.1,
                    with_grad=True).to(DEV)
    r1 = cpr.cpr_gdn_bwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, x.dO, h0=x.h0, contract=c)
    r2 = cpr.cpr_gdn_bwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, x.dO, h0=x.h0, contract=c)
    for n in r1:
        assert_bitwise(n, r1[n], r2[n])


def test_device_error_bad_seqlens():
    c = cpr.simt_contract(torch.bfloat16, 64)
    x = make_inputs([10, 10], 1, 64, 64, io_dtype=torch.bfloat16, seed=1).to(DEV)
    cpr.get_device_error(clear=True)
    o = torch.full((20, 1, 64), 7.0, device=DEV)
    bad = torch.tensor([0, 15, 12], dtype=torch.int32, device=DEV)  # not monotone, wrong total
    cpr.cpr_gdn_fwd(x.q, x.k, x.v, x.g, x.beta, bad, contract=c, out=o)
    assert cpr.get_device_error(clear=True) == 8
    assert bool((o == 7.0).all())   # nothing written
    bad2 = torch.tensor([0, 10, 19], dtype=torch.int32, device=DEV)  # last != n_tok
    cpr.cpr_gdn_fwd(x.q, x.k, x.v, x.g, x.beta, bad2, contract=c, out=o)
    assert cpr.get_device_error(clear=True) == 8


def test_decode_rejects_cache_of_another_contract():
    x = make_inputs([70], 1, 64, 64, io_dtype=torch.bfloat16, seed=1).to(DEV)
    ca = cpr.simt_contract(torch.bfloat16, 64, dv_splits=1)
    cb = cpr.simt_contract(torch.bfloat16, 64, dv_splits=2)
    cu = torch.tensor([0, 69], dtype=torch.int32, device=DEV)
    _, _, cache = cpr.cpr_gdn_prefill(x.q[:69], x.k[:69], x.v[:69], x.g[:69], x.beta[:69], cu,
                                      contract=ca)
    torch.cuda.synchronize()
    before = cache.blob.clone()
    cpr.get_device_error(clear=True)
    o = torch.full((1, 1, 64), 3.0, device=DEV)
    cpr.cpr_gdn_decode_step(x.q[69:], x.k[69:], x.v[69:], x.g[69:], x.beta[69:], cache,
                            contract=cb, out=o)
    assert cpr.get_device_error(clear=True) == 4
    assert torch.equal(cache.blob, before)
    assert bool((o == 3.0).all())
    cpr.cpr_gdn_decode_step(x.q[69:], x.k[69:], x.v[69:], x.g[69:], x.beta[69:], cache,
                            contract=ca, out=o)
    assert cpr.get_device_error(clear=True) == 0


def test_bounded_wait_expires_with_device_timeout_and_context_stays_usable():
    cpr.get_device_error(clear=True)
    assert cpr.selftest_wait_timeout(4096)                 # the wait ran out
    assert cpr.get_device_error(clear=True) == 9           # CPR_ERR_DEVICE_TIMEOUT recorded
    c = cpr.simt_contract(torch.bfloat16, 128, dv_splits=2, operand_policy=cpr.CPR_POLICY_TC_BF16X3)
    x = make_inputs([100], 2, 128, 128, io_dtype=torch.bfloat16, seed=3)
    o, _ = cpr.cpr_gdn_fwd(*(t.to(DEV) for t in (x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens)), contract=c)
    torch.cuda.synchronize()
    assert cpr.get_device_error() == 0
    o_ref, _ = oracle.gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens)
    assert_close("o after the timeout", o, o_ref, TOL_BF16)
