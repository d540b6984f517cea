"""Batch-invariant projection GEMM: parity with the oracle, and a row's bits independent
of the batch it is in (other rows, its index, M) and of repeated runs."""
import pytest
import torch

import infer_consistent_linear_gb300 as cpr
import oracle
from gpu_helpers import TOL_F32, assert_bitwise, assert_close, require_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _inputs(m, k, n, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(m, k, generator=g).to(torch.bfloat16)
    w = (torch.randn(k, n, generator=g) / k ** 0.5).to(torch.bfloat16)
    return x, w


@pytest.mark.parametrize("leaf_k", [512, 256, 128])
def test_gemm_matches_oracle(leaf_k):
    x, w = _inputs(300, 512, 256, 1)
    y = cpr.cpr_gemm(x.to(DEV), w.to(DEV), leaf_k)
    torch.cuda.synchronize()
    assert cpr.get_device_error() == 0
    ref = oracle.gemm(x.float().numpy(), w.float().numpy())
    assert_close("Y", y.cpu(), ref, TOL_F32)


def test_gemm_batch_invariance():
    x, w = _inputs(517, 1024, 384, 2)
    xd, wd = x.to(DEV), w.to(DEV)
    y = cpr.cpr_gemm(xd, wd, 256)
    # the same rows at other indices, in batches of other sizes, with other neighbours
    y_sub = cpr.cpr_gemm(xd[57:190].contiguous(), wd, 256)
    assert_bitwise("rows 57..189 alone", y_sub, y[57:190])
    other, _ = _inputs(77, 1024, 384, 3)
    y_cat = cpr.cpr_gemm(torch.cat([other.to(DEV), xd]).contiguous(), wd, 256)
    assert_bitwise("rows after 77 others", y_cat[77:], y)
    y_one = cpr.cpr_gemm(xd[400:401].contiguous(), wd, 256)
    assert_bitwise("row 400 at M = 1", y_one, y[400:401])
    assert_bitwise("rerun", cpr.cpr_gemm(xd, wd, 256), y)
    torch.cuda.synchronize()
    assert cpr.get_device_error() == 0


def test_gemm_rejects_bad_shapes():
    x, w = _inputs(8, 192, 128, 4)
    with pytest.raises(cpr.CprError):
        cpr.cpr_gemm(x.to(DEV), w.to(DEV), 64)       # 3 leaves
    x2, w2 = _inputs(8, 128, 96, 5)
    with pytest.raises(cpr.CprError):
        cpr.cpr_gemm(x2.to(DEV), w2.to(DEV), 128)    # N not a multiple of 128


def test_gemm_many_tiles_per_cta_sampled_rows():
    """More 128 x 256 output tiles than SMs, so every persistent CTA walks several tiles
    (and the TMEM hand-off between a tile's epilogue and the next tile's MMAs repeats):
    sampled rows against the oracle, and a ragged last row tile."""
    m, k, n = 40000 + 37, 512, 2048
    x, w = _inputs(m, k, n, 6)
    y = cpr.cpr_gemm(x.to(DEV), w.to(DEV), 128).cpu()
    torch.cuda.synchronize()
    assert cpr.get_device_error() == 0
    rows = torch.cat([torch.arange(0, 8), torch.randint(8, m - 8, (56,), generator=torch.Generator().manual_seed(7)),
                      torch.arange(m - 8, m)])
    ref = oracle.gemm(x[rows].float().numpy(), w.float().numpy())
    assert_close("Y sampled rows", y[rows], ref, TOL_F32)
