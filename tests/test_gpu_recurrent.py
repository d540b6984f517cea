"""Stage-table ablation paths (the token recurrence): parity with the oracle, bit
agreement between the recurrent prefill and recurrent decode steps, and the property
the comparison is about: a chunked prefill followed by recurrent decode steps ("native
mixed") is close to the oracle but not bit-identical to a one-shot prefill."""
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


@pytest.mark.parametrize("io,d,tol", [(torch.bfloat16, 128, TOL_BF16), (torch.float32, 64, TOL_F32)])
def test_recurrent_fwd_matches_oracle(io, d, tol):
    lens, H = [200, 64, 1, 0, 130], 2
    x = make_inputs(lens, H, d, d, io_dtype=io, seed=3, h0_std=0.1)
    xd = x.to(DEV)
    c = cpr.default_contract(io, d)
    o, fin = cpr.cpr_gdn_recurrent_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, h0=xd.h0, contract=c)
    torch.cuda.synchronize()
    assert cpr.get_device_error() == 0
    o_ref, h_ref = oracle.gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, h0=x.h0)
    assert_close("o", o.cpu(), o_ref, tol)
    assert_close("final", fin.cpu(), h_ref, tol)
    o2, fin2 = cpr.cpr_gdn_recurrent_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, h0=xd.h0,
                                         contract=c)
    assert_bitwise("o rerun", o2, o)
    assert_bitwise("final rerun", fin2, fin)


def test_recurrent_steps_equal_recurrent_prefill():
    pre, steps, H, d = [70, 64, 0, 5], 40, 2, 128
    full = [L + steps for L in pre]
    x = make_inputs(full, H, d, d, io_dtype=torch.bfloat16, seed=4, h0_std=0.1).to(DEV)
    c = cpr.default_contract(torch.bfloat16, d)
    o_full, fin_full = cpr.cpr_gdn_recurrent_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, h0=x.h0,
                                                 contract=c)
    cu = x.cu_seqlens.tolist()
    sel = torch.cat([torch.arange(cu[b], cu[b] + pre[b]) for b in range(len(pre))]).to(DEV)
    cu_pre = torch.tensor([0] + torch.cumsum(torch.tensor(pre), 0).tolist(), dtype=torch.int32, device=DEV)
    _, state = cpr.cpr_gdn_recurrent_fwd(x.q[sel], x.k[sel], x.v[sel], x.g[sel], x.beta[sel], cu_pre,
                                         h0=x.h0, contract=c)
    for t in range(steps):
        idx = torch.tensor([cu[b] + pre[b] + t for b in range(len(pre))], device=DEV)
        ot = cpr.cpr_gdn_recurrent_step(x.q[idx], x.k[idx], x.v[idx], x.g[idx], x.beta[idx], state,
                                        contract=c)
        assert_bitwise(f"step {t}", ot, o_full[idx])
    assert_bitwise("final state", state, fin_full)
    torch.cuda.synchronize()
    assert cpr.get_device_error() == 0


def test_native_mixed_is_close_but_not_bitwise():
    """Chunked (tensor-core) prefill, then recurrent decode from its final state: the
    outputs stay within tolerance of the oracle, and differ in bits from the one-shot
    prefill that CPR's decode reproduces exactly."""
    pre, steps, H, d = [128, 100, 64, 37], 30, 2, 128
    full = [L + steps for L in pre]
    x = make_inputs(full, H, d, d, io_dtype=torch.bfloat16, seed=5, h0_std=0.1)
    xd = x.to(DEV)
    c = cpr.default_contract(torch.bfloat16, d, dv_splits=2, operand_policy=cpr.CPR_POLICY_TC_BF16X3)
    o_full, _ = cpr.cpr_gdn_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, h0=xd.h0, contract=c)
    cu = x.cu_seqlens.tolist()
    sel = torch.cat([torch.arange(cu[b], cu[b] + pre[b]) for b in range(len(pre))]).to(DEV)
    cu_pre = torch.tensor([0] + torch.cumsum(torch.tensor(pre), 0).tolist(), dtype=torch.int32, device=DEV)
    _, state = cpr.cpr_gdn_fwd(xd.q[sel], xd.k[sel], xd.v[sel], xd.g[sel], xd.beta[sel], cu_pre,
                               h0=xd.h0, contract=c)
    outs, idxs = [], []
    for t in range(steps):
        idx = torch.tensor([cu[b] + pre[b] + t for b in range(len(pre))], device=DEV)
        outs.append(cpr.cpr_gdn_recurrent_step(xd.q[idx], xd.k[idx], xd.v[idx], xd.g[idx], xd.beta[idx],
                                               state, contract=c))
        idxs.append(idx)
    torch.cuda.synchronize()
    assert cpr.get_device_error() == 0
    o_dec = torch.stack(outs)                       # [steps, n_seq, H, d]
    o_pre = torch.stack([o_full[i] for i in idxs])
    differ = int((o_dec.view(torch.int32) != o_pre.view(torch.int32)).sum())
    assert differ > 0, "native mixed decode unexpectedly reproduced the prefill's bits"
    o_ref, _ = oracle.gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, h0=x.h0)
    o_ref = torch.as_tensor(o_ref)
    o_ref_steps = torch.stack([o_ref[i.cpu()] for i in idxs])
    assert_close("native mixed decode vs oracle", o_dec.cpu(), o_ref_steps, TOL_BF16)


def _tc():
    return cpr.default_contract(torch.bfloat16, 128, dv_splits=2, operand_policy=cpr.CPR_POLICY_TC_BF16X3)


def _rb():
    """Reading B as its own contract: intra_order TOKENREC_V1 on the tensor-core policy."""
    return cpr.default_contract(torch.bfloat16, 128, dv_splits=2, operand_policy=cpr.CPR_POLICY_TC_BF16X3,
                                intra_order=cpr.CPR_ORDER_TOKENREC_V1)


def test_reading_b_matches_oracle_and_differs_from_reading_a():
    """Reading B: the chunk form's boundary states, the token recurrence inside each chunk.
    Within tolerance of the oracle like reading A, with the same final state (the same
    chunk-form forward), not the same bits as reading A's outputs, and another digest."""
    lens, H = [200, 64, 1, 0, 130], 2
    x = make_inputs(lens, H, 128, 128, io_dtype=torch.bfloat16, seed=8, h0_std=0.1)
    xd = x.to(DEV)
    ob, fb = cpr.cpr_gdn_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, h0=xd.h0, contract=_rb())
    oa, fa = cpr.cpr_gdn_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, h0=xd.h0, contract=_tc())
    torch.cuda.synchronize()
    assert cpr.get_device_error() == 0
    assert cpr.contract_digest(_rb()) != cpr.contract_digest(_tc())
    o_ref, h_ref = oracle.gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, h0=x.h0)
    assert_close("o reading B", ob.cpu(), o_ref, TOL_BF16)
    assert_close("o reading A", oa.cpu(), o_ref, TOL_BF16)
    assert_bitwise("final state", fb, fa)
    assert int((ob.view(torch.int32) != oa.view(torch.int32)).sum()) > 0
    ob2, _ = cpr.cpr_gdn_fwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, h0=xd.h0, contract=_rb())
    assert_bitwise("reading B rerun", ob2, ob)


def test_reading_b_first_chunk_is_the_token_recurrence():
    """With no initial state every sequence's first boundary state is zero, so reading B's
    first chunk is exactly the token recurrence from zero (cpr_gdn_recurrent_fwd)."""
    lens, H = [130, 64, 40], 2
    x = make_inputs(lens, H, 128, 128, io_dtype=torch.bfloat16, seed=9).to(DEV)
    ob, _ = cpr.cpr_gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, contract=_rb())
    cu = x.cu_seqlens.tolist()
    for b, L in enumerate(lens):
        n = min(L, 64)
        sl = slice(cu[b], cu[b] + n)
        cub = torch.tensor([0, n], dtype=torch.int32, device=DEV)
        orr, _ = cpr.cpr_gdn_recurrent_fwd(x.q[sl], x.k[sl], x.v[sl], x.g[sl], x.beta[sl], cub,
                                           contract=cpr.default_contract(torch.bfloat16, 128))
        assert_bitwise(f"first chunk of seq {b}", ob[sl], orr)
    torch.cuda.synchronize()
    assert cpr.get_device_error() == 0


def test_reading_b_decode_equals_reading_b_prefill():
    """Reading B end to end under its contract: a prefill (the decode cache also keeps the
    running in-chunk state and the partial chunk's token rows), then decode steps (one
    token of the recurrence each, restarting from hi + lo of the committed state at each
    chunk's first row; a completed chunk is committed by the chunk form's prep and state
    pass over its buffered rows) give the bits of a one-shot forward over the full
    sequences, and the committed states are the chunk form's."""
    pre, steps, H = [100, 64, 0, 37, 130], 70, 2
    full = [L + steps for L in pre]
    x = make_inputs(full, H, 128, 128, io_dtype=torch.bfloat16, seed=10, h0_std=0.1).to(DEV)
    cb = _rb()
    o_full, _ = cpr.cpr_gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, h0=x.h0, contract=cb)
    cu = x.cu_seqlens.tolist()
    sel = torch.cat([torch.arange(cu[b], cu[b] + pre[b]) for b in range(len(pre))]).to(DEV)
    cu_pre = torch.tensor([0] + torch.cumsum(torch.tensor(pre), 0).tolist(), dtype=torch.int32, device=DEV)
    o_pre, _, cache = cpr.cpr_gdn_prefill(x.q[sel], x.k[sel], x.v[sel], x.g[sel], x.beta[sel], cu_pre,
                                          h0=x.h0, contract=cb)
    assert_bitwise("prefill part", o_pre, o_full[sel])
    for t in range(steps):
        idx = torch.tensor([cu[b] + pre[b] + t for b in range(len(pre))], device=DEV)
        ot = cpr.cpr_gdn_decode_step(x.q[idx], x.k[idx], x.v[idx], x.g[idx], x.beta[idx], cache, contract=cb)
        assert_bitwise(f"reading-B decode step {t}", ot, o_full[idx])
        for b in range(len(pre)):
            n_done = pre[b] + t + 1
            if n_done % 64 == 0:
                sl = slice(cu[b], cu[b] + n_done)
                _, fin = cpr.cpr_gdn_fwd(x.q[sl], x.k[sl], x.v[sl], x.g[sl], x.beta[sl],
                                         torch.tensor([0, n_done], dtype=torch.int32, device=DEV),
                                         h0=x.h0[b:b + 1], contract=_tc())
                assert_bitwise(f"committed state seq {b} at {n_done}", cache.state()[b:b + 1], fin)
    torch.cuda.synchronize()
    assert cpr.get_device_error() == 0


def test_reading_b_nocommit_steps_same_bits():
    """cpr_gdn_decode_step_nocommit on every step in which no sequence completes its chunk
    (the caller tracks the positions from its own lengths) and cpr_gdn_decode_step on the
    others: the same bits as a one-shot forward, and the same committed states."""
    pre, steps, H = [100, 64, 0, 37, 130], 70, 2
    full = [L + steps for L in pre]
    x = make_inputs(full, H, 128, 128, io_dtype=torch.bfloat16, seed=10, h0_std=0.1).to(DEV)
    cb = _rb()
    o_full, _ = cpr.cpr_gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, h0=x.h0, contract=cb)
    cu = x.cu_seqlens.tolist()
    sel = torch.cat([torch.arange(cu[b], cu[b] + pre[b]) for b in range(len(pre))]).to(DEV)
    cu_pre = torch.tensor([0] + torch.cumsum(torch.tensor(pre), 0).tolist(), dtype=torch.int32, device=DEV)
    _, _, cache = cpr.cpr_gdn_prefill(x.q[sel], x.k[sel], x.v[sel], x.g[sel], x.beta[sel], cu_pre,
                                      h0=x.h0, contract=cb)
    n_free = 0
    for t in range(steps):
        idx = torch.tensor([cu[b] + pre[b] + t for b in range(len(pre))], device=DEV)
        free = all((pre[b] + t) % 64 != 63 for b in range(len(pre)))
        n_free += free
        ot = cpr.cpr_gdn_decode_step(x.q[idx], x.k[idx], x.v[idx], x.g[idx], x.beta[idx], cache, contract=cb,
                                     no_commit=free)
        assert_bitwise(f"reading-B decode step {t} (no_commit={free})", ot, o_full[idx])
        for b in range(len(pre)):
            n_done = pre[b] + t + 1
            if n_done % 64 == 0:
                sl = slice(cu[b], cu[b] + n_done)
                _, fin = cpr.cpr_gdn_fwd(x.q[sl], x.k[sl], x.v[sl], x.g[sl], x.beta[sl],
                                         torch.tensor([0, n_done], dtype=torch.int32, device=DEV),
                                         h0=x.h0[b:b + 1], contract=_tc())
                assert_bitwise(f"committed state seq {b} at {n_done}", cache.state()[b:b + 1], fin)
    torch.cuda.synchronize()
    assert cpr.get_device_error() == 0
    assert 0 < n_free < steps


def test_reading_b_nocommit_refused_when_a_chunk_completes():
    """A no-commit step while a sequence sits at its chunk's last row (its step would
    complete the chunk) is refused on the device: nothing is written, no position moves,
    CPR_ERR_COMMIT_DUE is recorded; the ordinary step then runs as usual.  Under reading A,
    whose step commits inside its own kernel, the claim changes nothing."""
    x = make_inputs([64 + 63 + 1, 10 + 1], 2, 128, 128, io_dtype=torch.bfloat16, seed=12).to(DEV)
    cu = x.cu_seqlens.tolist()
    pre = [127, 10]
    sel = torch.cat([torch.arange(cu[b], cu[b] + pre[b]) for b in range(2)]).to(DEV)
    cu_pre = torch.tensor([0, 127, 137], dtype=torch.int32, device=DEV)
    idx = torch.tensor([cu[0] + 127, cu[1] + 10], device=DEV)
    tok = (x.q[idx], x.k[idx], x.v[idx], x.g[idx], x.beta[idx])
    for c in (_rb(), _tc()):
        o_full, _ = cpr.cpr_gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, contract=c)
        _, _, cache = cpr.cpr_gdn_prefill(x.q[sel], x.k[sel], x.v[sel], x.g[sel], x.beta[sel], cu_pre,
                                          contract=c)
        assert cpr.get_device_error(clear=True) == 0
        if c.intra_order == cpr.CPR_ORDER_TOKENREC_V1:
            before = cache.blob.clone()
            o = torch.full((2, 2, 128), 7.0, device=DEV)
            cpr.cpr_gdn_decode_step(*tok, cache, contract=c, out=o, no_commit=True)
            torch.cuda.synchronize()
            assert cpr.get_device_error(clear=True) == cpr.CPR_ERR_COMMIT_DUE
            assert torch.equal(cache.blob, before)
            assert bool((o == 7.0).all())
            ot = cpr.cpr_gdn_decode_step(*tok, cache, contract=c)
        else:
            ot = cpr.cpr_gdn_decode_step(*tok, cache, contract=c, no_commit=True)
        torch.cuda.synchronize()
        assert cpr.get_device_error(clear=True) == 0
        assert_bitwise(f"step after the claim ({'B' if c.intra_order == cpr.CPR_ORDER_TOKENREC_V1 else 'A'})",
                       ot, o_full[idx])


def test_reading_a_cache_refused_by_reading_b_decode():
    """A decode cache made under reading A carries reading A's digest and layout.  The
    binding refuses it for a reading-B decode step on the host (its layout is not reading
    B's).  Through the C ABI, in a blob of reading B's size, the device-side header check
    refuses it: nothing is written and CPR_ERR_CONTRACT_MISMATCH is recorded."""
    import ctypes
    x = make_inputs([100], 2, 128, 128, io_dtype=torch.bfloat16, seed=11).to(DEV)
    _, _, cache = cpr.cpr_gdn_prefill(x.q[:99], x.k[:99], x.v[:99], x.g[:99], x.beta[:99],
                                      torch.tensor([0, 99], dtype=torch.int32, device=DEV), contract=_tc())
    assert cpr.get_device_error(clear=True) == 0
    tok = (x.q[99:], x.k[99:], x.v[99:], x.g[99:], x.beta[99:])
    with pytest.raises(cpr.CprError, match="needs|layout"):
        cpr.cpr_gdn_decode_step(*tok, cache, contract=_rb())
    rb = _rb()
    blob = torch.zeros(cpr.cache_layout(rb, 1, 2).total_bytes, dtype=torch.uint8, device=DEV)
    blob[:cache.blob.numel()] = cache.blob
    before = blob.clone()
    o = torch.empty(1, 2, 128, dtype=torch.float32, device=DEV)
    lib = cpr.load_library()
    dig = (ctypes.c_uint8 * 32).from_buffer_copy(cpr.contract_digest(rb))
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = lib.cpr_gdn_decode_step(ctypes.byref(rb), dig, *[p(t) for t in tok], 1, 2, p(blob), p(o),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, lib.cpr_last_error().decode()
    assert cpr.get_device_error(clear=True) == 4      # CPR_ERR_CONTRACT_MISMATCH
    assert torch.equal(blob, before)


@pytest.mark.parametrize("io,d,tol", [(torch.bfloat16, 128, TOL_BF16), (torch.float32, 64, TOL_F32)])
def test_recurrent_bwd_matches_oracle(io, d, tol):
    """"Recurrent everywhere" training: the reverse token recurrence on the GPU against the
    oracle's hand-derived adjoint, ragged sequences (segment boundaries at 16 tokens
    crossed, an empty and a one-token sequence), h0 and dHT given."""
    lens, H = [70, 16, 1, 0, 40], 2
    x = make_inputs(lens, H, d, d, io_dtype=io, seed=12, h0_std=0.1, with_grad=True)
    gen = torch.Generator().manual_seed(13)
    dHT = torch.randn(len(lens), H, d, d, generator=gen)
    xd = x.to(DEV)
    c = cpr.default_contract(io, d)
    got = cpr.cpr_gdn_recurrent_bwd(xd.q, xd.k, xd.v, xd.g, xd.beta, xd.cu_seqlens, xd.dO, h0=xd.h0,
                                    dHT=dHT.to(DEV), contract=c)
    torch.cuda.synchronize()
    assert cpr.get_device_error() == 0
    ref = oracle.gdn_bwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, x.dO, h0=x.h0, dHT=dHT)
    for n in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        assert_close(n, got[n], ref[n], tol)


def test_recurrent_bwd_deterministic_and_batch_invariant():
    lens, H, d = [50, 33, 17], 2, 128
    x = make_inputs(lens, H, d, d, io_dtype=torch.bfloat16, seed=14, h0_std=0.1, with_grad=True).to(DEV)
    c = cpr.default_contract(torch.bfloat16, d)
    a = cpr.cpr_gdn_recurrent_bwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, x.dO, h0=x.h0, contract=c)
    b = cpr.cpr_gdn_recurrent_bwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, x.dO, h0=x.h0, contract=c)
    for n in a:
        assert_bitwise(n, a[n], b[n])
    cu = x.cu_seqlens.tolist()
    for i, L in enumerate(lens):
        sl = slice(cu[i], cu[i + 1])
        one = cpr.cpr_gdn_recurrent_bwd(x.q[sl], x.k[sl], x.v[sl], x.g[sl], x.beta[sl],
                                        torch.tensor([0, L], dtype=torch.int32, device=DEV),
                                        x.dO[sl].contiguous(), h0=x.h0[i:i + 1].contiguous(), contract=c)
        for n in ("dq", "dk", "dv", "dg", "dbeta"):
            assert_bitwise(f"{n}[seq {i}]", one[n], a[n][sl])
        assert_bitwise(f"dh0[seq {i}]", one["dh0"], a["dh0"][i:i + 1])
    torch.cuda.synchronize()
    assert cpr.get_device_error() == 0
