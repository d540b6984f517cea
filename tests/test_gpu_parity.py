"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle,
element by element, at sizes that span several chunks (C = 64) with ragged
tails, empty and one-token sequences, and nonzero initial states."""
import pytest
import torch

import infer_consistent_linear_gb300 as cpr
import oracle
from infer_consistent_linear_gb300.synth import make_inputs
from gpu_helpers import TOL_BF16, TOL_F32, assert_close, require_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _fwd_case(lens, H, d, io, tol, h0_std, splits=None):
    x = make_inputs(lens, H, d, d, io_dtype=io, seed=3, h0_std=h0_std)
    xd = x.to(DEV)
    c = cpr.simt_contract(io, d, **({"dv_splits": splits} if splits else {}))
    o, fin = cpr.cpr_gdn_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, h0=xd.h0, contract=c)
    torch.cuda.synchronize()
    assert cpr.get_device_error() == 0
    o_ref, h_ref = oracle.gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, h0=x.h0)
    assert_close("o", o, o_ref, tol)
    assert_close("final_state", fin, h_ref, tol)


@pytest.mark.parametrize("d", [64, 128])
def test_fwd_bf16_ragged(d):
    _fwd_case([200, 64, 1, 130, 0, 257], H=3, d=d, io=torch.bfloat16, tol=TOL_BF16, h0_std=0.1)


def test_fwd_fp32_tiny_config():
    # B=1, H=2, T=256, d=64, fp32 inputs: tolerance 1e-5 * RMS
    _fwd_case([256], H=2, d=64, io=torch.float32, tol=TOL_F32, h0_std=0.0)


def test_fwd_fp32_ragged_with_state():
    _fwd_case([99, 3, 128, 65], H=2, d=64, io=torch.float32, tol=TOL_F32, h0_std=0.3)


@pytest.mark.parametrize("splits", [1, 2, 4])
def test_fwd_dv_splits(splits):
    _fwd_case([140, 70], H=2, d=128, io=torch.bfloat16, tol=TOL_BF16, h0_std=0.1, splits=splits)


def _bwd_case(lens, H, d, io, tol, with_dHT=True):
    x = make_inputs(lens, H, d, d, io_dtype=io, seed=5, h0_std=0.1, with_grad=True)
    gen = torch.Generator().manual_seed(9)
    dHT = torch.randn(len(lens), H, d, d, generator=gen) if with_dHT else None
    xd = x.to(DEV)
    c = cpr.simt_contract(io, d)
    got = cpr.cpr_gdn_bwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, xd.dO, h0=xd.h0,
                          dHT=None if dHT is None else dHT.to(DEV), contract=c)
    torch.cuda.synchronize()
    assert cpr.get_device_error() == 0
    ref = oracle.gdn_bwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, x.dO, h0=x.h0, dHT=dHT)
    return {n: assert_close(n, got[n], ref[n], tol) for n in ("dq", "dk", "dv", "dg", "dbeta", "dh0")}


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_bf16_ragged(d):
    _bwd_case([150, 64, 1, 0, 200], H=2, d=d, io=torch.bfloat16, tol=TOL_BF16)


def test_bwd_fp32():
    _bwd_case([130, 7], H=2, d=64, io=torch.float32, tol=TOL_F32)


def test_bwd_without_dHT():
    _bwd_case([100], H=1, d=128, io=torch.bfloat16, tol=TOL_BF16, with_dHT=False)


def test_scale_parameter():
    x = make_inputs([90, 40], 2, 64, 64, io_dtype=torch.bfloat16, seed=4, with_grad=True)
    xd = x.to(DEV)
    c = cpr.simt_contract(torch.bfloat16, 64, scale=0.125)
    o, _ = cpr.cpr_gdn_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, contract=c)
    gr = cpr.cpr_gdn_bwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, xd.dO, contract=c)
    o_ref, _ = oracle.gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, scale=0.125)
    g_ref = oracle.gdn_bwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, x.dO, scale=0.125)
    assert_close("o", o, o_ref, TOL_BF16)
    for n in ("dq", "dk", "dv", "dg", "dbeta"):
        assert_close(n, gr[n], g_ref[n], TOL_BF16)


def test_zero_token_batch_passes_state_through():
    c = cpr.simt_contract(torch.bfloat16, 128)
    x = make_inputs([0, 0], 2, 128, 128, io_dtype=torch.bfloat16, seed=1, h0_std=0.5).to(DEV)
    o, fin = cpr.cpr_gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, h0=x.h0, contract=c)
    torch.cuda.synchronize()
    assert cpr.get_device_error() == 0
    assert o.numel() == 0
    assert torch.equal(fin, x.h0)
