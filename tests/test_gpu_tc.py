"""GPU tests of the tensor-core operand policy (TC_BF16X3: tcgen05 MMAs with
bf16 hi/lo operand splitting): parity with the fp64 oracle and bit identity
across prefill, decode, chunk-aligned splits and batch composition under one
TC contract."""
import pytest
import torch

import infer_consistent_linear_gb300 as cpr
import oracle
from infer_consistent_linear_gb300.synth import make_inputs
from gpu_helpers import TOL_BF16, assert_bitwise, assert_close, require_gpu
from test_gpu_bitwise import _decode_vs_prefill

pytestmark = pytest.mark.gpu
DEV = "cuda"
TC = dict(operand_policy=cpr.CPR_POLICY_TC_BF16X3)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _tc(splits=2):
    return cpr.default_contract(torch.bfloat16, 128, dv_splits=splits, **TC)


@pytest.mark.parametrize("splits", [2, 4])
def test_tc_fwd_parity_ragged(splits):
    lens = [200, 64, 1, 130, 0, 257]
    x = make_inputs(lens, 3, 128, 128, io_dtype=torch.bfloat16, seed=3, h0_std=0.1)
    xd = x.to(DEV)
    o, fin = cpr.cpr_gdn_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, h0=xd.h0,
                             contract=_tc(splits))
    torch.cuda.synchronize()
    assert cpr.get_device_error() == 0
    o_ref, h_ref = oracle.gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, h0=x.h0)
    assert_close("o", o, o_ref, TOL_BF16)
    assert_close("final_state", fin, h_ref, TOL_BF16)


def test_tc_fwd_parity_long_sequence_scale():
    x = make_inputs([1000], 2, 128, 128, io_dtype=torch.bfloat16, seed=8, h0_std=0.2)
    xd = x.to(DEV)
    c = cpr.default_contract(torch.bfloat16, 128, dv_splits=2, scale=0.5, **TC)
    o, fin = cpr.cpr_gdn_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, h0=xd.h0, contract=c)
    o_ref, h_ref = oracle.gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, h0=x.h0, scale=0.5)
    assert_close("o", o, o_ref, TOL_BF16)
    assert_close("final_state", fin, h_ref, TOL_BF16)


@pytest.mark.parametrize("splits", [2, 4])
def test_tc_decode_equals_prefill(splits):
    _decode_vs_prefill(torch.bfloat16, 128, [100, 64, 0, 1, 63], 70, 2, check_oracle_tol=TOL_BF16,
                       operand_policy=cpr.CPR_POLICY_TC_BF16X3, dv_splits=splits)


def test_tc_decode_persistent_mixed_positions():
    """More (sequence, head) units than SMs and positions all over the chunk in one launch:
    each persistent CTA walks several units with different positions, some of them
    committing a chunk while the next unit's tiles are prefetched."""
    lens = [(17 * i) % 131 for i in range(38)] + [64, 128]
    _decode_vs_prefill(torch.bfloat16, 128, lens, 66, 8, operand_policy=cpr.CPR_POLICY_TC_BF16X3,
                       dv_splits=2)


def test_tc_chunk_aligned_split_and_batch_invariance():
    c = _tc()
    lens = [300, 77, 1, 128]
    x = make_inputs(lens, 2, 128, 128, io_dtype=torch.bfloat16, seed=2, h0_std=0.1).to(DEV)
    o, fin = cpr.cpr_gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, h0=x.h0, contract=c)
    cu = x.cu_seqlens.tolist()
    for b, L in enumerate(lens):
        sl = slice(cu[b], cu[b + 1])
        cub = torch.tensor([0, L], dtype=torch.int32, device=DEV)
        ob, fb = cpr.cpr_gdn_fwd(x.q[sl], x.k[sl], x.v[sl], x.g[sl], x.beta[sl], cub,
                                 h0=x.h0[b:b + 1].contiguous(), contract=c)
        assert_bitwise(f"o seq {b}", ob, o[sl])
        assert_bitwise(f"final seq {b}", fb, fin[b:b + 1])
    # chunk-aligned split of sequence 0
    T1 = 128
    s0 = slice(0, T1)
    s1 = slice(T1, 300)
    o1, f1 = cpr.cpr_gdn_fwd(x.q[s0], x.k[s0], x.v[s0], x.g[s0], x.beta[s0],
                             torch.tensor([0, T1], dtype=torch.int32, device=DEV),
                             h0=x.h0[0:1].contiguous(), contract=c)
    o2, f2 = cpr.cpr_gdn_fwd(x.q[s1], x.k[s1], x.v[s1], x.g[s1], x.beta[s1],
                             torch.tensor([0, 300 - T1], dtype=torch.int32, device=DEV), h0=f1,
                             contract=c)
    assert_bitwise("split o1", o1, o[s0])
    assert_bitwise("split o2", o2, o[s1])
    assert_bitwise("split final", f2, fin[0:1])


def test_tc_context_parallel_segments_bitwise():
    """Context-parallel prefill emulated on one GPU: every sequence cut into chunk-aligned
    segments (one per emulated rank), run one after another with the fp32 state handed
    on as the next segment's h0; outputs and final states equal the unsplit run bit for
    bit, whatever the cut points, and that run is within tolerance of the oracle."""
    c = _tc()
    lens, H = [1024, 700, 192, 65], 2
    xc = make_inputs(lens, H, 128, 128, io_dtype=torch.bfloat16, seed=6, h0_std=0.1)
    x = xc.to(DEV)
    o, fin = cpr.cpr_gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, h0=x.h0, contract=c)
    # the unsplit run, and so every segmented one, against the fp64 oracle on these inputs
    o_ref, h_ref = oracle.gdn_fwd(xc.q, xc.k, xc.v, xc.g, xc.beta, xc.cu_seqlens, h0=xc.h0)
    assert_close("o", o, o_ref, TOL_BF16)
    assert_close("final_state", fin, h_ref, TOL_BF16)
    cu = x.cu_seqlens.tolist()
    for R in (2, 4):
        for b, L in enumerate(lens):
            nch = (L + 63) // 64
            cuts = sorted({min(L, 64 * ((nch * r) // R)) for r in range(R + 1)})
            h = x.h0[b:b + 1].contiguous()
            for lo, hi in zip(cuts[:-1], cuts[1:]):
                sl = slice(cu[b] + lo, cu[b] + hi)
                cub = torch.tensor([0, hi - lo], dtype=torch.int32, device=DEV)
                os, h = cpr.cpr_gdn_fwd(x.q[sl], x.k[sl], x.v[sl], x.g[sl], x.beta[sl], cub, h0=h, contract=c)
                assert_bitwise(f"o seq {b} segment [{lo}, {hi}) of {R}", os, o[sl])
            assert_bitwise(f"final seq {b}, {R} segments", h, fin[b:b + 1])
    torch.cuda.synchronize()
    assert cpr.get_device_error() == 0


def test_tc_prefill_cache_refused_by_simt_decode():
    x = make_inputs([70], 1, 128, 128, io_dtype=torch.bfloat16, seed=1).to(DEV)
    cu = torch.tensor([0, 69], dtype=torch.int32, device=DEV)
    _, _, cache = cpr.cpr_gdn_prefill(x.q[:69], x.k[:69], x.v[:69], x.g[:69], x.beta[:69], cu,
                                      contract=_tc())
    cpr.get_device_error(clear=True)
    simt = cpr.simt_contract(torch.bfloat16, 128, dv_splits=2)
    cpr.cpr_gdn_decode_step(x.q[69:], x.k[69:], x.v[69:], x.g[69:], x.beta[69:], cache, contract=simt)
    assert cpr.get_device_error(clear=True) == 4


GRADS = ("dq", "dk", "dv", "dg", "dbeta", "dh0")


def _tc_bwd(x, c, dHT=None):
    xd = x.to(DEV)
    got = cpr.cpr_gdn_bwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, xd.dO, h0=xd.h0,
                          dHT=None if dHT is None else dHT.to(DEV), contract=c)
    torch.cuda.synchronize()
    assert cpr.get_device_error() == 0
    return got


@pytest.mark.parametrize("splits", [2, 4])
def test_tc_backward_parity_ragged_with_dHT(splits):
    lens = [150, 64, 1, 0, 200]
    x = make_inputs(lens, 2, 128, 128, io_dtype=torch.bfloat16, seed=5, h0_std=0.1, with_grad=True)
    gen = torch.Generator().manual_seed(11)
    dHT = torch.randn(len(lens), 2, 128, 128, generator=gen)
    got = _tc_bwd(x, _tc(splits), dHT)
    ref = oracle.gdn_bwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, x.dO, h0=x.h0, dHT=dHT)
    for n in GRADS:
        assert_close(n, got[n], ref[n], TOL_BF16)


def test_tc_backward_parity_no_dHT_scale():
    x = make_inputs([300, 65], 3, 128, 128, io_dtype=torch.bfloat16, seed=6, h0_std=0.2, with_grad=True)
    c = cpr.default_contract(torch.bfloat16, 128, dv_splits=2, scale=0.5, **TC)
    got = _tc_bwd(x, c)
    ref = oracle.gdn_bwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, x.dO, h0=x.h0, scale=0.5)
    for n in GRADS:
        assert_close(n, got[n], ref[n], TOL_BF16)


def test_tc_backward_deterministic_and_batch_invariant():
    lens = [130, 64, 257, 5]
    x = make_inputs(lens, 2, 128, 128, io_dtype=torch.bfloat16, seed=7, h0_std=0.1, with_grad=True)
    c = _tc()
    a = _tc_bwd(x, c)
    b = _tc_bwd(x, c)
    for n in GRADS:
        assert_bitwise(n, a[n], b[n])
    cu = x.cu_seqlens.tolist()
    for i in range(len(lens)):
        lo, hi = cu[i], cu[i + 1]
        xs = make_inputs([lens[i]], 2, 128, 128, io_dtype=torch.bfloat16, seed=0, with_grad=True)
        for f in ("q", "k", "v", "g", "beta", "dO"):
            setattr(xs, f, getattr(x, f)[lo:hi].clone())
        xs.h0 = x.h0[i:i + 1].clone()
        one = _tc_bwd(xs, c)
        for n in ("dq", "dk", "dv", "dg", "dbeta"):
            assert_bitwise(f"{n}[seq {i}]", one[n], a[n][lo:hi])
        assert_bitwise(f"dh0[seq {i}]", one["dh0"], a["dh0"][i:i + 1])


def test_tc_training_forward_and_saved_backward_are_bitwise_the_plain_calls():
    lens = [200, 64, 1, 130]
    x = make_inputs(lens, 2, 128, 128, io_dtype=torch.bfloat16, seed=9, h0_std=0.1, with_grad=True)
    xd = x.to(DEV)
    c = _tc()
    gen = torch.Generator().manual_seed(3)
    dHT = torch.randn(len(lens), 2, 128, 128, generator=gen).to(DEV)
    o, fin = cpr.cpr_gdn_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, h0=xd.h0, contract=c)
    ref = cpr.cpr_gdn_bwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, xd.dO, h0=xd.h0, dHT=dHT,
                          contract=c)
    ws = torch.empty(cpr.workspace_bytes(c, cpr.CPR_OP_BWD, len(lens), sum(lens), 2),
                     dtype=torch.uint8, device=DEV)
    o2, fin2 = cpr.cpr_gdn_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, h0=xd.h0, contract=c,
                               workspace=ws, train=True)
    got = cpr.cpr_gdn_bwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, xd.dO, h0=xd.h0, dHT=dHT,
                          contract=c, workspace=ws, saved=True)
    torch.cuda.synchronize()
    assert cpr.get_device_error() == 0
    assert_bitwise("o", o2, o)
    assert_bitwise("final", fin2, fin)
    for n in GRADS:
        assert_bitwise(n, got[n], ref[n])
