"""The Python binding refuses, before anything reaches the C ABI or a kernel, tensors the
kernels would misread: host tensors (a host address handed to a kernel), another dtype,
inconsistent shapes (reads past the end of a shorter tensor) and non-contiguous views."""
import pytest
import torch

import infer_consistent_linear_gb300 as cpr
from infer_consistent_linear_gb300.synth import make_inputs


@pytest.fixture(scope="module")
def c():
    cpr.load_library()
    return cpr.default_contract(torch.bfloat16, 128, operand_policy=cpr.CPR_POLICY_TC_BF16X3, dv_splits=2)


def _x():
    return make_inputs([70, 30], 2, 128, 128, io_dtype=torch.bfloat16, seed=0, h0_std=0.1)


def _refused(fn, *args, match, **kw):
    with pytest.raises(cpr.CprError, match=match):
        fn(*args, **kw)


def test_host_tensors_refused(c):
    x = _x()   # correct dtypes and shapes, but on the host
    _refused(cpr.cpr_gdn_fwd, x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, contract=c, match="expected a CUDA")
    _refused(cpr.cpr_gdn_prefill, x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, contract=c, match="CUDA")
    _refused(cpr.cpr_gdn_recurrent_fwd, x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, contract=c, match="CUDA")
    _refused(cpr.cpr_gemm, torch.zeros(8, 64, dtype=torch.bfloat16), torch.zeros(64, 128, dtype=torch.bfloat16),
             64, match="CUDA")


def test_dtype_shape_and_layout_refused(c):
    x = _x()
    _refused(cpr.cpr_gdn_fwd, x.q.float(), x.k, x.v, x.g, x.beta, x.cu_seqlens, contract=c, match="q: dtype")
    _refused(cpr.cpr_gdn_fwd, x.q, x.k, x.v[:-1], x.g, x.beta, x.cu_seqlens, contract=c, match="v: shape")
    _refused(cpr.cpr_gdn_fwd, x.q, x.k, x.v, x.g.double(), x.beta, x.cu_seqlens, contract=c, match="g: dtype")
    _refused(cpr.cpr_gdn_fwd, x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens.long(), contract=c,
             match="cu_seqlens: dtype")
    _refused(cpr.cpr_gdn_fwd, x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, h0=x.h0[:1], contract=c,
             match="h0: shape")
    kt = x.k.transpose(1, 2).contiguous().transpose(1, 2)          # right shape, strided
    _refused(cpr.cpr_gdn_fwd, x.q, kt, x.v, x.g, x.beta, x.cu_seqlens, contract=c, match="k: not contiguous")
    _refused(cpr.cpr_gdn_bwd, x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, torch.zeros(100, 2, 128),
             contract=c, match="CUDA")
    _refused(cpr.cpr_gdn_bwd, x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, torch.zeros(99, 2, 128),
             contract=c, match="dO: shape")
    q1, k1, v1 = x.q[:2], x.k[:2], x.v[:2]
    _refused(cpr.cpr_gdn_recurrent_step, q1, k1, v1, x.g[:2], x.beta[:2], torch.zeros(2, 2, 128, 64),
             contract=c, match="state: shape")
    _refused(cpr.cpr_gemm, torch.zeros(8, 64, dtype=torch.bfloat16), torch.zeros(32, 128, dtype=torch.bfloat16),
             64, match="w: shape")
    _refused(cpr.cpr_gemm, torch.zeros(8, 64), torch.zeros(64, 128, dtype=torch.bfloat16), 64, match="x: dtype")


def test_decode_cache_must_match_contract_and_batch(c):
    """A caller's decode cache is checked against the layout of (contract, n_seq, H) before
    anything else: the C ABI takes no cache size, so a smaller cache would be written past
    its end.  The blobs live on the host here; the check runs before the device checks."""
    x = _x()   # 2 sequences, 2 heads
    good = cpr.new_decode_cache(c, 2, 2, "cpu")
    args = (x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens)
    _refused(cpr.cpr_gdn_prefill, *args, contract=c, cache=cpr.new_decode_cache(c, 1, 2, "cpu"),
             match="made for n_seq=1")
    _refused(cpr.cpr_gdn_prefill, *args, contract=c, cache=cpr.new_decode_cache(c, 2, 1, "cpu"),
             match="H=1")
    trunc = cpr.DecodeCache(good.blob[:-256], good.layout, 2, 2, 128, 128)
    _refused(cpr.cpr_gdn_prefill, *args, contract=c, cache=trunc, match="needs")
    rb = cpr.default_contract(torch.bfloat16, 128, operand_policy=cpr.CPR_POLICY_TC_BF16X3, dv_splits=2,
                              intra_order=cpr.CPR_ORDER_TOKENREC_V1)
    _refused(cpr.cpr_gdn_prefill, *args, contract=rb, cache=good, match="needs")   # reading-B layout is larger
    d64 = cpr.default_contract(torch.bfloat16, 64)
    _refused(cpr.cpr_gdn_prefill, x.q[..., :64].contiguous(), x.k[..., :64].contiguous(),
             x.v[..., :64].contiguous(), x.g, x.beta, x.cu_seqlens, contract=d64, cache=good, match="d_k=128")
    tok = (x.q[:2], x.k[:2], x.v[:2], x.g[:2], x.beta[:2])
    _refused(cpr.cpr_gdn_decode_step, *tok, cpr.new_decode_cache(c, 1, 2, "cpu"), contract=c, match="made for")
    _refused(cpr.cpr_gdn_decode_step, *tok, trunc, contract=c, match="needs")
    _refused(cpr.cpr_gdn_decode_step, *tok, "not a cache", contract=c, match="DecodeCache")
    # a matching cache passes this check; the host tensors are then refused
    _refused(cpr.cpr_gdn_prefill, *args, contract=c, cache=good, match="CUDA")
    _refused(cpr.cpr_gdn_decode_step, *tok, good, contract=c, match="CUDA")


def test_tensors_must_be_on_the_current_device():
    """Kernels launch on the current device's stream; tensors of another GPU are refused."""
    cpr._require_current(torch.device("cuda", 0), 0)
    cpr._require_current(torch.device("cuda", 3), 3)
    cpr._require_current(torch.device("cuda"), 1)    # no index: the current device
    with pytest.raises(cpr.CprError, match="current device is cuda:0"):
        cpr._require_current(torch.device("cuda", 1), 0)
