"""The allocation-free forward, cpr_gdn_fwd_noalloc, called through the C ABI.

It is meant for callers that cannot allocate device memory where they run the
forward (host callbacks, allocator hooks, fixed memory pools), so it takes no
workspace and uses a scratch array built into the library.  Two calls in a
row, with different inputs, under the tensor-core and the CUDA-core operand
policies, must give the same result as cpr_gdn_fwd with a caller workspace
(bit for bit, since the same kernels run) and stay within the parity tolerance
of the fp64 oracle.  A batch larger than the built-in scratch is refused
up front.  This file is collected last so a stop-at-first-failure run has
already run every other test; it also passes alone in a fresh process.
"""
import ctypes

import pytest
import torch

import infer_consistent_linear_gb300 as cpr
from infer_consistent_linear_gb300.synth import make_inputs
from gpu_helpers import TOL_BF16, assert_bitwise, rel_err, require_gpu

pytestmark = pytest.mark.gpu
DEV = "cuda"
SCRATCH_BYTES = 64 * 1024 * 1024


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(lib, c, x, o, fin):
    dig = (ctypes.c_uint8 * 32).from_buffer_copy(cpr.contract_digest(c))
    n_tok, H = x.q.shape[0], x.q.shape[1]
    n_seq = x.cu_seqlens.numel() - 1
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.cpr_gdn_fwd_noalloc(ctypes.byref(c), dig, _p(x.q), _p(x.k), _p(x.v), _p(x.g),
                                   _p(x.beta), _p(x.cu_seqlens), n_seq, n_tok, H, _p(x.h0), _p(o),
                                   _p(fin), stream)


@pytest.mark.parametrize("policy", ["tc", "simt"])
def test_noalloc_matches_workspace_forward_on_two_calls(policy):
    require_gpu()
    import oracle
    lib = cpr.load_library()
    pol = cpr.CPR_POLICY_TC_BF16X3 if policy == "tc" else cpr.CPR_POLICY_SIMT_F32
    c = cpr.default_contract(torch.bfloat16, 128, operand_policy=pol, dv_splits=2)
    for seed, lens in ((21, [200, 64, 1, 130]), (22, [333, 70])):
        xc = make_inputs(lens, 3, 128, 128, io_dtype=torch.bfloat16, seed=seed, h0_std=0.1)
        x = xc.to(DEV)
        o_ref, fin_ref = cpr.cpr_gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, h0=x.h0,
                                         contract=c)
        o = torch.full_like(o_ref, float("nan"))
        fin = torch.full_like(fin_ref, float("nan"))
        assert _noalloc(lib, c, x, o, fin) == 0, lib.cpr_last_error().decode()
        torch.cuda.synchronize()
        assert cpr.get_device_error() == 0
        o_or, fin_or = oracle.gdn_fwd(xc.q, xc.k, xc.v, xc.g, xc.beta, xc.cu_seqlens, h0=xc.h0)
        assert rel_err(o, o_or) <= TOL_BF16
        assert rel_err(fin, fin_or) <= TOL_BF16
        assert_bitwise("o", o, o_ref)
        assert_bitwise("final", fin, fin_ref)


def test_noalloc_refuses_batch_larger_than_its_scratch():
    require_gpu()
    lib = cpr.load_library()
    c = cpr.default_contract(torch.bfloat16, 128)
    n_tok, H = 8 * 4096, 16
    assert cpr.workspace_bytes(c, cpr.CPR_OP_FWD, 8, n_tok, H) > SCRATCH_BYTES
    dig = (ctypes.c_uint8 * 32).from_buffer_copy(cpr.contract_digest(c))
    dummy = torch.empty(16, device=DEV)
    p = ctypes.c_void_p(dummy.data_ptr())
    rc = lib.cpr_gdn_fwd_noalloc(ctypes.byref(c), dig, p, p, p, p, p, p, 8, n_tok, H, None, p,
                                 None, None)
    assert rc == 7
    assert "scratch" in lib.cpr_last_error().decode()
